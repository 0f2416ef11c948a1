// bwd_dq_sm103.cu -- dQ of the recomputation backward for d = 128, query-parallel.
//
// At d = 128 the key-parallel backward kernel fills TMEM with S^T, dP^T, dV and dK,
// so dQ is computed here instead, one CTA per (head, 128-query block i), sweeping
// the key blocks j ("FlashAttention-1" page, 10.2.4, with P rebuilt from the saved
// statistic):
//     S_ij = Q_i K_j^T,  P_ij = exp(S_ij - lse_i),  dP_ij = dO_i V_j^T,
//     dS_ij = P_ij o (dP_ij - delta_i),  dQ_i = scale * sum_j dS_ij K_j.
// dQ_i accumulates in TMEM over the whole sweep and is written once as bf16: no
// atomics and no fp32 accumulator in device memory.
//
// Layout: warp 0 TMA (Q_i and dO_i once; K_j / V_j in a 2-stage ring), warp 1 MMA,
// warps 4-7 and 8-11 one query row per thread, for keys 0-63 / 64-127 of block j.
// TMEM: S 0-127 (dS bf16 written back inside the columns each half read: keys
// 64h..64h+63 -> columns 64h..64h+31), dP 128-255, dQ 256-383.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

constexpr int kBlk = 128;
constexpr int kThreads = 384;
constexpr int kStages = 2;

template <int D>
struct DqCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = kBlk * D * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffDO = kTile;
    static constexpr int kOffK = 2 * kTile;                      // kStages
    static constexpr int kOffV = kOffK + kStages * kTile;        // kStages
    static constexpr int kSmemBytes = kOffV + kStages * kTile;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kIdescSS = idesc_bf16(128, 128, false, false);  // S, dP
    static constexpr uint32_t kIdescDQ = idesc_bf16(128, D, false, true);     // dQ += dS K
};
static_assert(DqCfg<128>::kSmemAlloc <= 232448, "smem");

struct DqArgs {
    const float* ws_nlse2;   // [BH][Np]: -lse * log2(e) (-inf on pad rows)
    const float* ws_ndelta;  // [BH][Np]: -delta
    void* dq;
    int N, Np, n_q, BH;      // BH: query heads (B * H)
    int H, H_kv;             // query heads and K/V heads per batch; H_kv divides H
    int causal;
    float c_log2;            // scale * log2(e)
    float scale;
    DevCtl ctl;
};

struct DqBars {
    uint64_t q_full;
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t sp_full, ds_full, all_done, drain;
};

__device__ __forceinline__ void record_timeout(const DevCtl& ctl, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(ctl.status, kDevOk, kDevTimeout);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const DqArgs args) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) DqBars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const uint32_t sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // causal: the query block with the most key blocks goes first for every head
    const int bh = args.causal ? static_cast<int>(blockIdx.x % args.BH) : static_cast<int>(blockIdx.x / args.n_q);
    const int qb = args.causal ? args.n_q - 1 - static_cast<int>(blockIdx.x / args.BH)
                               : static_cast<int>(blockIdx.x % args.n_q);
    // grouped-query attention: query head bh reads K/V head bh_kv of its group
    const int bh_kv = (bh / args.H) * args.H_kv + (bh % args.H) / (args.H / args.H_kv);
    const int N = args.N, Np = args.Np;
    const int n_kv = args.causal ? qb + 1 : Np / kBlk;  // key blocks this query block meets
    const uint64_t lim = args.ctl.wait_ns;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bars.q_full), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bars.kv_full[s]), 1);
            mbar_init(smem_u32(&bars.kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&bars.sp_full), 1);
        mbar_init(smem_u32(&bars.ds_full), 256);
        mbar_init(smem_u32(&bars.all_done), 1);
        mbar_init(smem_u32(&bars.drain), 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ================================================================ producer
        if (lane == 0) {
            const uint32_t qf = smem_u32(&bars.q_full);
            mbar_arrive_expect_tx(qf, 2 * C::kTile);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(sb + C::kOffQ + c * 16384, &tm_q, qf, 64 * c, qb * kBlk, bh);
                tma_load_3d(sb + C::kOffDO + c * 16384, &tm_do, qf, 64 * c, qb * kBlk, bh);
            }
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % kStages;
                if (j >= kStages &&
                    !mbar_wait(smem_u32(&bars.kv_empty[s]), ((j / kStages) & 1) ^ 1, lim, &abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t kf = smem_u32(&bars.kv_full[s]);
                mbar_arrive_expect_tx(kf, 2 * C::kTile);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(sb + C::kOffK + s * C::kTile + c * 16384, &tm_k, kf, 64 * c, j * kBlk, bh_kv);
                    tma_load_3d(sb + C::kOffV + s * C::kTile + c * 16384, &tm_v, kf, 64 * c, j * kBlk, bh_kv);
                }
                issued = j + 1;
            }
            if (!ok) record_timeout(args.ctl, &abort_flag);
            const volatile int never = 0;
            mbar_wait(qf, 0, kDrainWaitNs, &never);
            for (int j = max(0, issued - kStages); j < issued; ++j)
                mbar_wait(smem_u32(&bars.kv_full[j % kStages]), (j / kStages) & 1, kDrainWaitNs, &never);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            // Operand descriptors as low words built once (see sdesc_sw128_lo): K-major
            // (leading byte offset 16) for S and dP, MN-major (16384) for K in dQ; each MMA
            // adds its K step's offset / 16.
            constexpr uint32_t kDescHi = sdesc_sw128_hi(1024);
            constexpr uint32_t kStage16 = C::kTile >> 4;
            const uint32_t q_lo = sdesc_sw128_lo(sb + C::kOffQ, 16), do_lo = sdesc_sw128_lo(sb + C::kOffDO, 16);
            const uint32_t k_lo = sdesc_sw128_lo(sb + C::kOffK, 16), v_lo = sdesc_sw128_lo(sb + C::kOffV, 16);
            const uint32_t k_mn = sdesc_sw128_lo(sb + C::kOffK, 16384);
            // S = Q K_j^T and dP = dO V_j^T (both operands K-major along d)
            auto issue_sp = [&](int s) {
                const uint32_t kl = k_lo + s * kStage16, vl = v_lo + s * kStage16;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off16 = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    if (kk == 0)
                        mma_ss_w<false, -1>(tmem + C::kColS, q_lo, kl, kDescHi, C::kIdescSS, 0u);
                    else
                        mma_ss_w<false, 1>(tmem + C::kColS, q_lo + off16, kl + off16, kDescHi, C::kIdescSS);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off16 = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    if (kk == 0)
                        mma_ss_w<false, -1>(tmem + C::kColDP, do_lo, vl, kDescHi, C::kIdescSS, 0u);
                    else
                        mma_ss_w<false, 1>(tmem + C::kColDP, do_lo + off16, vl + off16, kDescHi, C::kIdescSS);
                }
                mma_commit(smem_u32(&bars.sp_full));
            };
            bool ok = mbar_wait(smem_u32(&bars.q_full), 0, lim, &abort_flag);
            if (ok) ok = mbar_wait(smem_u32(&bars.kv_full[0]), 0, lim, &abort_flag);
            if (ok) {
                tc_fence_after();
                issue_sp(0);
            }
            for (int j = 0; j < n_kv && ok; ++j) {
                const int s = j % kStages;
                ok = mbar_wait(smem_u32(&bars.ds_full), j & 1, lim, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                // dQ += dS_j K_j: A = dS from TMEM (queries x keys), B = K_j MN-major (d contiguous)
                const uint32_t km = k_mn + s * kStage16;
#pragma unroll
                for (int kk = 0; kk < kBlk / 16; ++kk) {
                    if (kk == 0)
                        mma_ts_w<false, -1>(tmem + C::kColDQ, tmem + C::kColS, km, kDescHi, C::kIdescDQ, j > 0 ? 1u : 0u);
                    else
                        mma_ts_w<false, 1>(tmem + C::kColDQ, tmem + C::kColS + 64 * (kk >> 2) + 8 * (kk & 3),
                                           km + 128 * kk, kDescHi, C::kIdescDQ);
                }
                mma_commit(smem_u32(&bars.kv_empty[s]));  // K_j and V_j consumed
                if (j + 1 < n_kv) {
                    const int s1 = (j + 1) % kStages;
                    ok = mbar_wait(smem_u32(&bars.kv_full[s1]), ((j + 1) / kStages) & 1, lim, &abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    issue_sp(s1);  // in issue order after dQ_j, which still reads dS_j
                }
            }
            if (ok) mma_commit(smem_u32(&bars.all_done));
            if (!ok) record_timeout(args.ctl, &abort_flag);
            mma_commit(smem_u32(&bars.drain));
            const volatile int never = 0;
            mbar_wait(smem_u32(&bars.drain), 0, kDrainWaitNs, &never);
        }
    } else if (warp >= 4) {
        // ================================================================ dS warpgroups
        const int half = (warp - 4) / 4;  // keys 64*half .. 64*half+63 of each block
        const int wq = warp % 4;
        const int row = wq * 32 + lane;
        const int qrow = qb * kBlk + row;
        const uint32_t lb = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const size_t srow = static_cast<size_t>(bh) * Np + qrow;  // padded rows exist up to Np
        const float nl = args.ws_nlse2[srow], nd = args.ws_ndelta[srow];
        const float2 c2 = make_float2(args.c_log2, args.c_log2);
        const float2 nl2 = make_float2(nl, nl), nd2 = make_float2(nd, nd);
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            ok = mbar_wait(smem_u32(&bars.sp_full), j & 1, lim, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t rs[2][32], rp[2][32];
            tmem_ld32_async(lb + C::kColS + 64 * half, rs[0]);
            tmem_ld32_async(lb + C::kColS + 64 * half + 32, rs[1]);
            tmem_ld32_async(lb + C::kColDP + 64 * half, rp[0]);
            tmem_ld32_async(lb + C::kColDP + 64 * half + 32, rp[1]);
            tmem_wait_ld();
            reg_fence(rs[0]);
            reg_fence(rs[1]);
            reg_fence(rp[0]);
            reg_fence(rp[1]);
            // causal diagonal block: query row r sees keys 0..r of the block
            const bool diag = args.causal && (j == qb);
            uint32_t pk[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const int e = 2 * (x % 16);
                const uint32_t* S = rs[x / 16];
                const uint32_t* P = rp[x / 16];
                float2 a = __ffma2_rn(make_float2(__uint_as_float(S[e]), __uint_as_float(S[e + 1])), c2, nl2);
                if (diag) {
                    const int key = 64 * half + 32 * (x / 16) + e;
                    if (key > row) a.x = -INFINITY;
                    if (key + 1 > row) a.y = -INFINITY;
                }
                const float2 p = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                const float2 g = __fadd2_rn(make_float2(__uint_as_float(P[e]), __uint_as_float(P[e + 1])), nd2);
                const float2 ds = __fmul2_rn(p, g);
                pk[x] = pack_bf16x2(ds.x, ds.y);
            }
            tmem_st32(lb + C::kColS + 64 * half, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.ds_full));
        }
        if (ok) {
            ok = mbar_wait(smem_u32(&bars.all_done), 0, lim, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (!ok) {
            if (lane == 0) record_timeout(args.ctl, &abort_flag);
        } else {
            tc_fence_after();
            // this half stores columns half*D/2 .. +D/2 of its row: dQ = scale * accumulator
            const float sc = args.scale;
            uint16_t* out = static_cast<uint16_t*>(args.dq) + (static_cast<size_t>(bh) * N + qrow) * D;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                const int col = half * (D / 2) + 32 * h;
                uint32_t r[32];
                tmem_ld32(lb + C::kColDQ + col, r);
                if (qrow < N) {
                    uint4* o4 = reinterpret_cast<uint4*>(out + col);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        o4[x] = make_uint4(
                            pack_bf16x2(__uint_as_float(r[8 * x]) * sc, __uint_as_float(r[8 * x + 1]) * sc),
                            pack_bf16x2(__uint_as_float(r[8 * x + 2]) * sc, __uint_as_float(r[8 * x + 3]) * sc),
                            pack_bf16x2(__uint_as_float(r[8 * x + 4]) * sc, __uint_as_float(r[8 * x + 5]) * sc),
                            pack_bf16x2(__uint_as_float(r[8 * x + 6]) * sc, __uint_as_float(r[8 * x + 7]) * sc));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace

int launch_bwd_dq(const void* q, const void* k, const void* v, const void* dO,
                  const float* ws_nlse2, const float* ws_ndelta, void* dq, int B, int H, int H_kv,
                  int N, int d, float scale, int causal, DevCtl ctl, cudaStream_t s) {
    if (d != 128) return -1;
    const int BH = B * H, BH_kv = B * H_kv;
    using C = DqCfg<128>;
    CUtensorMap tq, tk, tv, tdo;
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    int rc = make_map_3d(&tq, q, dt, 2, 128, N, BH, 64, kBlk);
    if (rc == 0) rc = make_map_3d(&tk, k, dt, 2, 128, N, BH_kv, 64, kBlk);
    if (rc == 0) rc = make_map_3d(&tv, v, dt, 2, 128, N, BH_kv, 64, kBlk);
    if (rc == 0) rc = make_map_3d(&tdo, dO, dt, 2, 128, N, BH, 64, kBlk);
    if (rc != 0) return rc;
    static uint64_t attr_set = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(attr_set & (1ull << dev))) {
        cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
        if (e != cudaSuccess) return static_cast<int>(e);
        if (dev < 64) attr_set |= 1ull << dev;
    }
    DqArgs a;
    a.ws_nlse2 = ws_nlse2;
    a.ws_ndelta = ws_ndelta;
    a.dq = dq;
    a.N = N;
    a.Np = round_up(N, kBlk);
    a.n_q = a.Np / kBlk;
    a.BH = BH;
    a.H = H;
    a.H_kv = H_kv;
    a.causal = causal ? 1 : 0;
    a.c_log2 = scale * 1.4426950408889634f;
    a.scale = scale;
    a.ctl = ctl;
    // an ordinary launch: with programmatic serialization its CTAs would only sit
    // waiting through the dK/dV kernel's tail (measured 0.3% slower)
    bwd_dq_kernel<128><<<a.n_q * BH, kThreads, C::kSmemAlloc, s>>>(tq, tk, tv, tdo, a);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace fa
