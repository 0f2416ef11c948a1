/*
 * oracle.c -- plain, slow, fp64 CPU oracle for exact softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test suite, the package's smoke check and the benchmark's
 * CPU-baseline / reference leg do.  It shares no code, header, table or helper
 * with the CUDA library.
 *
 * What it computes (per head; tensors are [BH][N][d], row-major, fp64):
 *
 *   forward  (standard attention, "FlashAttention-1" page, 10.2.1: S = QK^T,
 *             P = softmax(S), O = PV, with the stable softmax that subtracts the
 *             row max m_i and divides by l_i; the 1/sqrt(d) factor of the
 *             Flash Attention V1/V2/V3 page's Python demo is the caller's `scale`):
 *        S_ij = scale * sum_k Q_ik K_jk          (causal: S_ij = -inf for j > i)
 *        m_i  = max_j S_ij,   l_i = sum_j exp(S_ij - m_i)
 *        P_ij = exp(S_ij - m_i) / l_i,   O_i = sum_j P_ij V_j
 *        lse_i = m_i + ln l_i
 *
 *   backward ("FlashAttention-1" page, 10.2.4, with the scale made explicit and
 *             the softmax backward in the form dS = P o (dP - delta)):
 *        dV = P^T dO,  dP = dO V^T,  delta_i = sum_k dO_ik O_ik,
 *        dS = P o (dP - delta),  dQ = scale dS K,  dK = scale dS^T Q
 *
 *   tiled forward (online softmax, "Flash Attention V1/V2/V3" page, Python demo
 *             and "5.4 FlashAttention" page, listing 3-1): Q in row blocks of Br,
 *             K/V in blocks of Bc; running max m, running sum l and unnormalised
 *             output o; each block rescales the old state by exp(m_old - m_new)
 *             and the output is divided by l once at the end.  Exists only to
 *             check that the result does not depend on the block sizes.
 *
 *   e4m3     OCP 8-bit floating point E4M3 (bias 7, no infinities, S.1111.111 is
 *            NaN, largest finite 448): decode, and round-to-nearest-even encode
 *            with saturation to +-448.
 *
 * Parallelism: OpenMP over rows (forward) or over rows within one head
 * (backward).  `nthreads` <= 0 means "OpenMP default".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

ORACLE_API int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One query row of one head: materialise the row S_i and P_i (length N), then
 * O_i = P_i V.  Returns lse_i.  `srow` is caller scratch of length N. */
static double fwd_one_row(const double* q_i, const double* k, const double* v, long N,
                          long d, double scale, int causal, long i, double* srow,
                          double* o_i) {
    /* S_i (masked entries are -inf) */
    double m = -INFINITY;
    for (long j = 0; j < N; ++j) {
        if (causal && j > i) {
            srow[j] = -INFINITY;
            continue;
        }
        const double* k_j = k + j * d;
        double acc = 0.0;
        for (long c = 0; c < d; ++c) acc += q_i[c] * k_j[c];
        srow[j] = scale * acc;
        if (srow[j] > m) m = srow[j];
    }
    /* l_i = sum_j exp(S_ij - m_i);  P_ij = exp(S_ij - m_i) / l_i */
    double l = 0.0;
    for (long j = 0; j < N; ++j) {
        double e = (srow[j] == -INFINITY) ? 0.0 : exp(srow[j] - m);
        srow[j] = e;
        l += e;
    }
    for (long j = 0; j < N; ++j) srow[j] /= l;
    /* O_i = sum_j P_ij V_j */
    for (long c = 0; c < d; ++c) o_i[c] = 0.0;
    for (long j = 0; j < N; ++j) {
        const double p = srow[j];
        if (p == 0.0) continue;
        const double* v_j = v + j * d;
        for (long c = 0; c < d; ++c) o_i[c] += p * v_j[c];
    }
    return m + log(l);
}

/* Selected rows of ONE head.  q, k, v: [N][d].  rows: nrows query indices.
 * o: [nrows][d], lse: [nrows]. */
ORACLE_API void oracle_fwd_rows(const double* q, const double* k, const double* v, long N,
                                long d, double scale, int causal, const long* rows,
                                long nrows, double* o, double* lse, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < nrows; ++r) {
            const long i = rows[r];
            lse[r] = fwd_one_row(q + i * d, k, v, N, d, scale, causal, i, srow, o + r * d);
        }
        free(srow);
    }
}

/* All rows of all BH heads.  q, k, v, o: [BH][N][d]; lse: [BH][N]. */
ORACLE_API void oracle_fwd(const double* q, const double* k, const double* v, long BH,
                           long N, long d, double scale, int causal, double* o,
                           double* lse, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 4) collapse(2)
        for (long h = 0; h < BH; ++h) {
            for (long i = 0; i < N; ++i) {
                const size_t base = (size_t)h * N * d;
                lse[h * N + i] = fwd_one_row(q + base + i * d, k + base, v + base, N, d, scale,
                                             causal, i, srow, o + base + i * d);
            }
        }
        free(srow);
    }
}

/* Online-softmax (tiled) forward, in the pages' order: for each block of Br
 * query rows, sweep the K/V blocks of Bc rows, keep m (init -inf), l (init 0)
 * and the unnormalised o (init 0); per block: m_new = max(m, rowmax(s)),
 * p = exp(s - m_new), l = l*exp(m - m_new) + rowsum(p),
 * o = o*exp(m - m_new) + p V_blk; finally O = o / l.
 * A row whose running max is still -inf (all keys so far masked) uses 0 as the
 * reference so that the rescale factor is 1 and p is 0 instead of NaN. */
ORACLE_API void oracle_fwd_tiled(const double* q, const double* k, const double* v, long BH,
                                 long N, long d, double scale, int causal, long Br, long Bc,
                                 double* o, double* lse) {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Br * Bc));
    double* m = (double*)malloc(sizeof(double) * (size_t)Br);
    double* l = (double*)malloc(sizeof(double) * (size_t)Br);
    double* acc = (double*)malloc(sizeof(double) * (size_t)(Br * d));
    for (long h = 0; h < BH; ++h) {
        const double* qh = q + (size_t)h * N * d;
        const double* kh = k + (size_t)h * N * d;
        const double* vh = v + (size_t)h * N * d;
        for (long i0 = 0; i0 < N; i0 += Br) {
            const long br = (i0 + Br <= N) ? Br : N - i0;
            for (long r = 0; r < br; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.0;
                for (long c = 0; c < d; ++c) acc[r * d + c] = 0.0;
            }
            for (long j0 = 0; j0 < N; j0 += Bc) {
                const long bc = (j0 + Bc <= N) ? Bc : N - j0;
                for (long r = 0; r < br; ++r) {
                    const long i = i0 + r;
                    /* score block s = scale * q_blk k_blk^T (masked -> -inf) */
                    double mblk = -INFINITY;
                    for (long t = 0; t < bc; ++t) {
                        const long j = j0 + t;
                        double x;
                        if (causal && j > i) {
                            x = -INFINITY;
                        } else {
                            double a = 0.0;
                            for (long c = 0; c < d; ++c) a += qh[i * d + c] * kh[j * d + c];
                            x = scale * a;
                        }
                        s[r * Bc + t] = x;
                        if (x > mblk) mblk = x;
                    }
                    const double m_new = (mblk > m[r]) ? mblk : m[r];
                    const double ref = (m_new == -INFINITY) ? 0.0 : m_new;
                    const double alpha = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - ref);
                    double rowsum = 0.0;
                    for (long t = 0; t < bc; ++t) {
                        const double x = s[r * Bc + t];
                        const double p = (x == -INFINITY) ? 0.0 : exp(x - ref);
                        s[r * Bc + t] = p;
                        rowsum += p;
                    }
                    l[r] = l[r] * alpha + rowsum;
                    for (long c = 0; c < d; ++c) {
                        double pv = 0.0;
                        for (long t = 0; t < bc; ++t) pv += s[r * Bc + t] * vh[(j0 + t) * d + c];
                        acc[r * d + c] = acc[r * d + c] * alpha + pv;
                    }
                    m[r] = m_new;
                }
            }
            for (long r = 0; r < br; ++r) {
                const long i = i0 + r;
                for (long c = 0; c < d; ++c)
                    o[(size_t)h * N * d + i * d + c] = acc[r * d + c] / l[r];
                lse[h * N + i] = m[r] + log(l[r]);
            }
        }
    }
    free(s);
    free(m);
    free(l);
    free(acc);
}

/* Analytic backward of O = softmax(scale QK^T [masked]) V for all BH heads.
 * Per head it materialises P (N x N) from scratch, then
 *   O = P V, delta_i = dO_i . O_i, dV = P^T dO, dP = dO V^T,
 *   dS = P o (dP - delta), dQ = scale dS K, dK = scale dS^T Q.
 * q, k, v, dout, dq, dk, dv: [BH][N][d]. */
ORACLE_API void oracle_bwd(const double* q, const double* k, const double* v,
                           const double* dout, long BH, long N, long d, double scale,
                           int causal, double* dq, double* dk, double* dv, int nthreads) {
    set_threads(nthreads);
    double* P = (double*)malloc(sizeof(double) * (size_t)N * (size_t)N);
    double* dS = (double*)malloc(sizeof(double) * (size_t)N * (size_t)N);
    double* O = (double*)malloc(sizeof(double) * (size_t)N * (size_t)d);
    double* delta = (double*)malloc(sizeof(double) * (size_t)N);
    for (long h = 0; h < BH; ++h) {
        const size_t base = (size_t)h * N * d;
        const double* qh = q + base;
        const double* kh = k + base;
        const double* vh = v + base;
        const double* doh = dout + base;
        double* dqh = dq + base;
        double* dkh = dk + base;
        double* dvh = dv + base;
        /* P (row softmax of the masked, scaled scores), O = P V, delta = rowsum(dO o O),
         * dP = dO V^T and dS = P o (dP - delta): all row-local */
#pragma omp parallel for schedule(dynamic, 8)
        for (long i = 0; i < N; ++i) {
            double* Pi = P + (size_t)i * N;
            double mx = -INFINITY;
            for (long j = 0; j < N; ++j) {
                if (causal && j > i) {
                    Pi[j] = -INFINITY;
                    continue;
                }
                double a = 0.0;
                for (long c = 0; c < d; ++c) a += qh[i * d + c] * kh[j * d + c];
                Pi[j] = scale * a;
                if (Pi[j] > mx) mx = Pi[j];
            }
            double l = 0.0;
            for (long j = 0; j < N; ++j) {
                Pi[j] = (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - mx);
                l += Pi[j];
            }
            for (long j = 0; j < N; ++j) Pi[j] /= l;
            double* Oi = O + (size_t)i * d;
            for (long c = 0; c < d; ++c) Oi[c] = 0.0;
            for (long j = 0; j < N; ++j)
                for (long c = 0; c < d; ++c) Oi[c] += Pi[j] * vh[j * d + c];
            double dl = 0.0;
            for (long c = 0; c < d; ++c) dl += doh[i * d + c] * Oi[c];
            delta[i] = dl;
            double* dSi = dS + (size_t)i * N;
            for (long j = 0; j < N; ++j) {
                double dp = 0.0;
                for (long c = 0; c < d; ++c) dp += doh[i * d + c] * vh[j * d + c];
                dSi[j] = Pi[j] * (dp - dl);
            }
        }
        /* dQ = scale dS K (row i of dQ needs row i of dS).  Each dQ_ic is the sum over
         * j = 0, 1, ..., N-1 from 0.0; the loops run j outside c so that K is read by rows. */
#pragma omp parallel for schedule(static)
        for (long i = 0; i < N; ++i) {
            const double* dSi = dS + (size_t)i * N;
            double* dqi = dqh + i * d;
            for (long c = 0; c < d; ++c) dqi[c] = 0.0;
            for (long j = 0; j < N; ++j)
                for (long c = 0; c < d; ++c) dqi[c] += dSi[j] * kh[j * d + c];
            for (long c = 0; c < d; ++c) dqi[c] *= scale;
        }
        /* dV = P^T dO and dK = scale dS^T Q (row j needs column j of P and dS).  Each
         * element is the sum over i = 0, 1, ..., N-1 from 0.0; a thread owns a range of
         * rows j and runs i outside j, so P, dS, dO and Q are all read by rows. */
#pragma omp parallel
        {
            const int nt = omp_get_num_threads(), t = omp_get_thread_num();
            const long j0 = N * t / nt, j1 = N * (t + 1) / nt;
            for (long j = j0; j < j1; ++j)
                for (long c = 0; c < d; ++c) dvh[j * d + c] = dkh[j * d + c] = 0.0;
            for (long i = 0; i < N; ++i) {
                const double* Pi = P + (size_t)i * N;
                const double* dSi = dS + (size_t)i * N;
                for (long j = j0; j < j1; ++j)
                    for (long c = 0; c < d; ++c) {
                        dvh[j * d + c] += Pi[j] * doh[i * d + c];
                        dkh[j * d + c] += dSi[j] * qh[i * d + c];
                    }
            }
            for (long j = j0; j < j1; ++j)
                for (long c = 0; c < d; ++c) dkh[j * d + c] *= scale;
        }
    }
    free(P);
    free(dS);
    free(O);
    free(delta);
}

/* ---- OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (value = m/8 * 2^-6); S.1111.111 is NaN; there
 * are no infinities, so S.1111.110 = +-448 is the largest finite value. */
ORACLE_API double oracle_e4m3_to_f64(uint8_t x) {
    const int sign = (x >> 7) & 1;
    const int e = (x >> 3) & 0xF;
    const int mant = x & 0x7;
    double val;
    if (e == 0xF && mant == 0x7) return NAN;
    if (e == 0)
        val = ldexp((double)mant / 8.0, -6);
    else
        val = ldexp(1.0 + (double)mant / 8.0, e - 7);
    return sign ? -val : val;
}

/* Round to the nearest E4M3 value, ties to an even mantissa, saturating to
 * +-448 (NaN in -> NaN code 0x7F). Found by exhaustive nearest search over the
 * 126 finite non-negative codes, so it follows the definition directly. */
ORACLE_API uint8_t oracle_f64_to_e4m3(double v) {
    if (isnan(v)) return 0x7F;
    const uint8_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x80 : 0x00;
    const double a = fabs(v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    uint8_t best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double cv = oracle_e4m3_to_f64((uint8_t)c);
        const double err = fabs(cv - a);
        /* strictly closer wins; on an exact tie the even mantissa (even code) wins */
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

ORACLE_API void oracle_e4m3_decode(const uint8_t* x, long n, double descale, double* out) {
    for (long i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f64(x[i]) * descale;
}

ORACLE_API void oracle_e4m3_encode(const double* v, long n, uint8_t* out) {
    for (long i = 0; i < n; ++i) out[i] = oracle_f64_to_e4m3(v[i]);
}
