// fwd_sm103.cu -- attention forward on the sm_103a tensor core (tcgen05 + TMEM + TMA).
//
// What it computes is the online-softmax forward of the "FlashAttention-1"
// page (10.2.2-10.2.3) in the unnormalised form of the "5.4 FlashAttention"
// page's listing 3-1 and the Python demo of the "Flash Attention V1/V2/V3演进"
// page: per query row a running max m, a running sum l and an unnormalised
// output o; each K/V block rescales the old state by alpha = exp(m_old - m_new)
// and adds exp(S - m_new) V; o / l once at the end; lse = m + ln l is saved for
// the backward.  Work split as the V2 section describes (one CTA owns its query
// rows and sweeps all K/V blocks, so O is final after one pass); scale and log2(e)
// are folded into one multiply before exp2, and the causal mask is applied in
// the score step.
//
// GB300 design (not the A100/H100 designs the pages sketch):
//   * Work item = 2 query tiles of 128 rows (one head).  bf16: one persistent CTA per SM
//     works through items, its TMEM, barriers and K/V ring carrying over from item to
//     item (the next item's Q and K/V load while one finishes); E4M3: one CTA per item.
//     O is written by each softmax thread as its row; lse likewise.
//   * 12 warps:
//       warp 0      TMA producer: each item's Q, then V_j and K_{j+1} as one bundle on
//                   one barrier into 2-slot rings
//       warp 1      MMA issuer (one thread) + TMEM owner
//       warps 4-7   softmax for query tile 0, warps 8-11 for query tile 1
//   * TMEM (512 columns): S_t (128 fp32 columns per tile), O_t (d columns);
//     P_t is written back over S_t as bf16 (or E4M3) and fed to the P V MMA
//     straight from TMEM.
//   * MMA order per K/V block j: O_0 += P_0 V_j, S_0 = Q_0 K_{j+1}^T,
//     O_1 += P_1 V_j, S_1 = Q_1 K_{j+1}^T -- the two softmax warpgroups
//     alternate with the tensor core (ping-pong).  MMAs issued by one thread
//     run in order, so the commit that publishes S_t(j+1) also proves that
//     O_t += P_t(j) V_j is finished; the softmax warps may then rescale O_t.
//   * E4M3: P_t goes to a 16 KB shared-memory tile instead (S and O of both tiles
//     fill TMEM), and the P V MMA reads it from there.  S_t(j+1) is then issued as
//     soon as the softmax warps have read S_t(j) out of TMEM (s_free), ahead of
//     O_t += P_t(j) V_j; a pv_done commit after each P V MMA tells the softmax
//     warps when P_t's tile may be rewritten and O_t rescaled.
//   * Lazy rescale: the reference max used for exp2 moves only when a row's
//     block max exceeds it by more than kTau (log2 units).  O and l always share
//     the same reference, so the result is exact for any threshold; p stays
//     <= 2^kTau (fine for bf16 and below the E4M3 limit of 448).
//   * Solo items (bf16): when the last round of pairs would leave SMs idle, its pairs are
//     dealt as single 128-row tiles, and a pair whose second tile lies past N runs as its
//     first tile alone.  Both softmax warpgroups then hold the tile's rows and take
//     alternate key blocks (warpgroup t the blocks t, t+2, ...), each with its own running
//     max, sum and O_t; warpgroup 0 merges the two halves at the end with the two-state
//     combination of the "FlashAttention-1" page (10.2.2).
//   * Every wait is bounded; on a timeout the kernel records it, drains its own
//     TMA loads and MMAs, frees TMEM and exits.
#include <cmath>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

constexpr int kBM = 128;         // query rows per tile
constexpr int kBN = 128;         // keys per K/V block
constexpr int kStages = 2;       // K/V ring depth
constexpr int kThreads = 384;    // 12 warps
constexpr float kTau = 8.0f;     // lazy-rescale threshold, log2 units

struct FwdArgs {
    void* o;          // bf16 [BH][N][D], or float32 when o_f32
    float* lse;
    int N;            // query rows per head
    int N_kv;         // keys per head (= N except for a key shard)
    int delta;        // causal: key j reaches query i iff j <= i + delta (0 unless sharded)
    int n_pairs;      // query-tile pairs per head
    int BH;           // query heads (B * H)
    int n_items;      // work items: n_pair_items pairs, then single tiles (solo items)
    int n_pair_items; // items dealt as whole pairs; pair n_pair_items + s/2 gives solo s
    float c_log2;     // scale * log2(e) (times the FP8 descales)
    float o_scale;    // multiplies O at the end (FP8: v descale), 1 otherwise
    int causal;
    int H, H_kv;                 // query heads and K/V heads per batch (H % H_kv == 0)
    const float* qk_descale_q;   // optional per-(b, h) FP8 descales (device); null: none
    const float* qk_descale_k;   //   indexed by the tensor's own head (b*H + h / b*H_kv + g)
    const float* v_descale;      //   (per-block kernel: [head][ceil(rows / 128)])
    DevCtl ctl;
};

template <int D, bool FP8>
struct Cfg {
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr int kRowBytes = D * kElem;
    static constexpr int kChunks = kRowBytes / 128;        // 128-byte swizzle columns
    static constexpr int kBoxX = 128 / kElem;              // elements per chunk row
    static constexpr int kChunkBytes = 128 * 128;          // 128 rows x 128 B
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kKStep = FP8 ? 32 : 16;           // K per MMA
    static constexpr int kStepBytes = kKStep * kElem;      // = 32
    // shared memory: Q0, Q1, K[kStages], V[kStages]
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    // E4M3: P_t goes to shared memory (one 128 x 128-byte swizzled tile per query tile), so
    // that S_t(j+1) can be computed into S_t's TMEM columns while the softmax warps still turn
    // S_t(j) into P_t(j); S and O of both tiles already take all 512 TMEM columns.
    static constexpr bool kPsmem = FP8;
    static constexpr int kPBytes = kBM * kBN;              // E4M3 P tile
    static constexpr int kOffP = kOffV + kStages * kTileBytes;
    static constexpr int kSmemBytes = kOffP + (kPsmem ? 2 * kPBytes : 0);
    static constexpr int kSmemAlloc = kSmemBytes + 1024;   // slack for 1 KB alignment
    // TMEM columns
    static constexpr uint32_t kColS0 = 0, kColS1 = 128;
    static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kIdescS = FP8 ? idesc_e4m3(kBM, kBN, false, false)
                                            : idesc_bf16(kBM, kBN, false, false);
    static constexpr uint32_t kIdescO = FP8 ? idesc_e4m3(kBM, D, false, true)
                                            : idesc_bf16(kBM, D, false, true);
};

struct Bars {
    uint64_t q_full;
    uint64_t q_free;  // an item's last S MMAs have read the Q buffers
    uint64_t kv_full[kStages], kv_empty[kStages];  // ring slot u: bundles n, n % kStages == u
    uint64_t s_full[2], p_full[2], o_done[2];
    uint64_t s_free[2], pv_done[2];  // kPsmem: S_t read out of TMEM; O_t += P_t V done
    uint64_t merge_ml;    // solo item: warpgroup 1's running max and sum are in shared memory
    uint64_t merge_done;  // solo item: warpgroup 0 has read O_1 (which may then be overwritten)
    uint64_t drain;
};

__device__ __forceinline__ void record_timeout(const DevCtl& ctl, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(ctl.status, kDevOk, kDevTimeout);
}

// 32 consecutive TMEM columns of this thread's lane into r[OFF..OFF+31], no wait.
template <int OFF>
__device__ __forceinline__ void tmem_ld32_at(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]),
          "=r"(r[OFF + 4]), "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]),
          "=r"(r[OFF + 8]), "=r"(r[OFF + 9]), "=r"(r[OFF + 10]), "=r"(r[OFF + 11]),
          "=r"(r[OFF + 12]), "=r"(r[OFF + 13]), "=r"(r[OFF + 14]), "=r"(r[OFF + 15]),
          "=r"(r[OFF + 16]), "=r"(r[OFF + 17]), "=r"(r[OFF + 18]), "=r"(r[OFF + 19]),
          "=r"(r[OFF + 20]), "=r"(r[OFF + 21]), "=r"(r[OFF + 22]), "=r"(r[OFF + 23]),
          "=r"(r[OFF + 24]), "=r"(r[OFF + 25]), "=r"(r[OFF + 26]), "=r"(r[OFF + 27]),
          "=r"(r[OFF + 28]), "=r"(r[OFF + 29]), "=r"(r[OFF + 30]), "=r"(r[OFF + 31])
        : "r"(taddr)
        : "memory");
}

// Wait for this thread's outstanding TMEM loads, then route every loaded register
// through an empty asm so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld_fence(uint32_t (&r)[128]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 128; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Max (or, for a negative score scale, min) of the 128 raw scores: four
// independent 3-input chains over r[4..123], then r[124..127].
__device__ __forceinline__ float block_extreme(const uint32_t (&r)[128], bool want_max) {
    float a[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) a[k] = __uint_as_float(r[k]);
    if (want_max) {
#pragma unroll
        for (int i = 4; i < 124; i += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                a[k] = max3f(a[k], __uint_as_float(r[i + 2 * k]), __uint_as_float(r[i + 2 * k + 1]));
        a[0] = max3f(a[0], __uint_as_float(r[124]), __uint_as_float(r[125]));
        a[1] = max3f(a[1], __uint_as_float(r[126]), __uint_as_float(r[127]));
        return max3f(a[0], a[1], fmaxf(a[2], a[3]));
    }
#pragma unroll
    for (int i = 4; i < 124; i += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            a[k] = min3f(a[k], __uint_as_float(r[i + 2 * k]), __uint_as_float(r[i + 2 * k + 1]));
    a[0] = min3f(a[0], __uint_as_float(r[124]), __uint_as_float(r[125]));
    a[1] = min3f(a[1], __uint_as_float(r[126]), __uint_as_float(r[127]));
    return min3f(a[0], a[1], fminf(a[2], a[3]));
}

// SHARD: forward over a key shard (N_kv keys, causal offset delta, float32 O,
// rows that see no key); compiled separately so the plain forward carries none of it.
// PB (FP8 only): the descales are per 128-row block of each head instead of per head.
//
// Persistent: a CTA works through (head, query-tile pair) items, its k-th item being
// x = k * gridDim.x + (blockIdx.x, or gridDim.x - 1 - blockIdx.x in odd rounds).  Every
// barrier counts its phases across items: per item with at least one key block (q_full,
// q_free, o_done), per K/V block (s_full, p_full, s_free, pv_done) or per bundle
// (kv_full, kv_empty), so TMEM, the barriers and the K/V ring carry over from one item to
// the next, and the next item's Q and first bundle load while this item finishes.  An
// item whose queries see no key (in a causal key shard; or a solo tile past N) involves
// neither the producer nor the MMA thread: the softmax warps write its O = 0 and lse = -inf
// (the solo tile has no rows to write).  Per-tile barriers count each tile's own blocks,
// since a solo item gives the two tiles different numbers of blocks.
template <int D, bool FP8, bool SHARD, bool PB = false>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
    using C = Cfg<D, FP8>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    __shared__ float merge_m[kBM], merge_l[kBM];  // solo item: warpgroup 1's max and sum per row

    const uint32_t smem_base =
        (smem_u32(smem_raw) + 1023u) & ~1023u;  // 1 KB aligned for the 128 B swizzle
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int N = args.N;
    const int N_kv = SHARD ? args.N_kv : N;
    const int delta = SHARD ? args.delta : 0;
    const int n_items = args.n_items;
    const int G = static_cast<int>(gridDim.x);
    // E4M3 runs one CTA per item (see the launch); with a compile-time single pass every
    // running counter below is a constant there
    constexpr bool kPersist = !FP8;
    constexpr int kItemsMax = kPersist ? 0x7fffffff : 1;
    constexpr bool kSolo = !FP8 && !SHARD;  // single-tile items (E4M3 and shards: pairs only)

    // this CTA's k-th item, dealt in alternating (snake) order so that no CTA always
    // takes the heaviest item of a round (causal items are ordered heaviest first)
    auto item_x = [&](int k) {
        return k * G + ((k & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
    };
    struct Item {
        int bh, bh_kv, r0, n_kv;
        bool solo;  // one query tile (rows r0 .. r0 + 127), not two
    };
    // Item x's tiles.  Items below n_pair_items are pairs in the order below; the rest
    // are single tiles, solo item s being tile s % 2 of pair n_pair_items + s / 2.
    // Pair order, non-causal: head-major, every pair of a head together (the head's K/V
    // stays in L2).  Causal: a pair's work grows with its index, so items run heaviest pair
    // first across all heads, which with the alternating deal keeps the CTAs' loads within
    // a few blocks of each other.  (Head-major order leaves the last heads' heaviest pairs
    // for the end; heaviest first within groups of heads whose K/V fits in L2 kept K/V in L2
    // but left the loads 4-14% apart, and measured 0.4-11% slower.)
    auto item_at = [&](int x) {
        int p = x, tile = 0;
        bool solo = false;
        if (kSolo && x >= args.n_pair_items) {
            p = args.n_pair_items + (x - args.n_pair_items) / 2;
            tile = (x - args.n_pair_items) & 1;
            solo = true;
        }
        int bh, pair;
        if (args.causal) {
            pair = args.n_pairs - 1 - p / args.BH;
            bh = p % args.BH;
        } else {
            bh = p / args.n_pairs;
            pair = args.n_pairs - 1 - (p % args.n_pairs);
        }
        Item I;
        I.bh = bh;
        // grouped-query attention: H / H_kv query heads share one K/V head
        I.bh_kv = (bh / args.H) * args.H_kv + (bh % args.H) / (args.H / args.H_kv);
        I.r0 = pair * 2 * kBM + tile * kBM;
        // a pair whose second tile lies wholly past N is its first tile alone
        if (kSolo && !solo && I.r0 + kBM >= N) solo = true;
        I.solo = solo;
        // keys these query rows can see; none at all when a causal key shard lies wholly
        // after them, or for a solo tile past N
        const int kv_end = args.causal ? min(N_kv, I.r0 + (solo ? kBM : 2 * kBM) + delta) : N_kv;
        I.n_kv = (I.r0 < N && (!SHARD || kv_end > 0)) ? (kv_end + kBN - 1) / kBN : 0;
        return I;
    };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bars.q_full), 1);
        mbar_init(smem_u32(&bars.q_free), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bars.kv_full[s]), 1);
            mbar_init(smem_u32(&bars.kv_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bars.s_full[t]), 1);
            mbar_init(smem_u32(&bars.p_full[t]), 128);
            mbar_init(smem_u32(&bars.o_done[t]), 1);
            mbar_init(smem_u32(&bars.s_free[t]), 128);
            mbar_init(smem_u32(&bars.pv_done[t]), 1);
        }
        mbar_init(smem_u32(&bars.merge_ml), 128);
        mbar_init(smem_u32(&bars.merge_done), 128);
        mbar_init(smem_u32(&bars.drain), 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint64_t lim = args.ctl.wait_ns;
    // launched while the previous kernel in the stream may still run (its outputs may be
    // these inputs): set up above, read nothing global before it has completed
    griddep_wait();
    griddep_launch_dependents();

    // 384 threads x 168 registers at launch: warpgroup 0 (load, MMA) gives up to
    // 120 per thread, the two softmax warpgroups take 184 (128*120 + 256*184 <= 384*168).
    if (warp < 4) {
    regs_dec<120>();
    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            const uint32_t qf = smem_u32(&bars.q_full);
            int gb = 0;  // bundles issued, over all items
            int kq = 0;  // items whose Q was issued (items with at least one key block)
            bool ok = true;
            const volatile int never = 0;
            for (int k = 0; ok && k < kItemsMax; ++k) {
                const int x = item_x(k);
                if (x >= n_items) break;
                const Item I = item_at(x);
                if (I.n_kv == 0) continue;
                // Q of this item once the last S MMAs of the previous one have read the Q buffers
                if (kq > 0 && !mbar_wait(smem_u32(&bars.q_free), (kq - 1) & 1, lim, &abort_flag)) {
                    ok = false;
                    break;
                }
                const int n_q = I.solo ? 1 : 2;
                mbar_arrive_expect_tx(qf, n_q * C::kTileBytes);
                for (int t = 0; t < n_q; ++t)
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(smem_base + C::kOffQ + t * C::kTileBytes + c * C::kChunkBytes, &tm_q,
                                    qf, c * C::kBoxX, I.r0 + t * kBM, I.bh);
                ++kq;
                // Bundle n = {K_n (n < n_kv), V_{n-1} (n >= 1)} in slot gb % kStages of both
                // rings, on one barrier: the MMA thread waits once per block for V_j and
                // K_{j+1}, and releases the slot once after their last reader.
                for (int n = 0; I.n_kv > 0 && n <= I.n_kv; ++n, ++gb) {
                    const int u = gb % kStages;
                    if (gb >= kStages &&
                        !mbar_wait(smem_u32(&bars.kv_empty[u]), ((gb / kStages) & 1) ^ 1, lim, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&bars.kv_full[u]);
                    mbar_arrive_expect_tx(fb, ((n < I.n_kv ? 1 : 0) + (n >= 1 ? 1 : 0)) * C::kTileBytes);
                    if (n < I.n_kv)
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d(smem_base + C::kOffK + u * C::kTileBytes + c * C::kChunkBytes, &tm_k,
                                        fb, c * C::kBoxX, n * kBN, I.bh_kv);
                    if (n >= 1)
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d(smem_base + C::kOffV + u * C::kTileBytes + c * C::kChunkBytes, &tm_v,
                                        fb, c * C::kBoxX, (n - 1) * kBN, I.bh_kv);
                }
            }
            if (!ok) record_timeout(args.ctl, &abort_flag);
            // drain: the last Q and the newest bundle of every slot have landed before exit
            if (kq > 0) mbar_wait(qf, (kq - 1) & 1, kDrainWaitNs, &never);
            for (int n = max(0, gb - kStages); n < gb; ++n)
                mbar_wait(smem_u32(&bars.kv_full[n % kStages]), (n / kStages) & 1, kDrainWaitNs, &never);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t sQ0 = smem_base + C::kOffQ, sQ1 = sQ0 + C::kTileBytes;
            // Operand descriptors: the low words of Q_t and of stage 0 of the K and V rings
            // are computed once; each MMA adds its K step's offset (see sdesc_sw128_lo).
            constexpr uint32_t kDescHi = sdesc_sw128_hi(1024);
            const uint32_t q_lo0 = sdesc_sw128_lo(sQ0, 16), q_lo1 = sdesc_sw128_lo(sQ1, 16);
            const uint32_t k_lo = sdesc_sw128_lo(smem_base + C::kOffK, 16);
            const uint32_t v_lo = sdesc_sw128_lo(smem_base + C::kOffV, C::kChunkBytes);
            auto issue_s = [&](uint32_t q_lo, int s, uint32_t col) {
                const uint32_t kl = k_lo + s * (C::kTileBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < D / C::kKStep; ++kk) {
                    const uint32_t off16 = ((kk * C::kStepBytes) / 128 * C::kChunkBytes +
                                            (kk * C::kStepBytes) % 128) >> 4;
                    if (kk == 0)
                        mma_ss_w<FP8, -1>(tmem + col, q_lo, kl, kDescHi, C::kIdescS, 0u);
                    else
                        mma_ss_w<FP8, 1>(tmem + col, q_lo + off16, kl + off16, kDescHi, C::kIdescS);
                }
            };
            auto issue_pv = [&](uint32_t colP, int s, uint32_t colO, bool acc) {
                const uint32_t vl = v_lo + s * (C::kTileBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < kBN / C::kKStep; ++kk) {
                    if (kk == 0)
                        mma_ts_w<FP8, -1>(tmem + colO, tmem + colP, vl, kDescHi, C::kIdescO, acc ? 1u : 0u);
                    else
                        mma_ts_w<FP8, 1>(tmem + colO, tmem + colP + kk * 8, vl + ((kk * C::kKStep * 128) >> 4),
                                         kDescHi, C::kIdescO);
                }
            };
            // kPsmem: O_t += P_t V with P_t from its shared-memory tile (K-major, 128-byte rows)
            const uint32_t p_lo0 = sdesc_sw128_lo(smem_base + C::kOffP, 16);
            auto issue_pv_s = [&](uint32_t p_lo, int s, uint32_t colO, bool acc) {
                const uint32_t vl = v_lo + s * (C::kTileBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < kBN / C::kKStep; ++kk) {
                    if (kk == 0)
                        mma_ss_w<FP8, -1>(tmem + colO, p_lo, vl, kDescHi, C::kIdescO, acc ? 1u : 0u);
                    else
                        mma_ss_w<FP8, 1>(tmem + colO, p_lo + ((kk * C::kStepBytes) >> 4),
                                         vl + ((kk * C::kKStep * 128) >> 4), kDescHi, C::kIdescO);
                }
            };
            int gb = 0;  // bundle index of the current item's bundle 0, over all items
            int c0 = 0, c1 = 0;  // K/V blocks of tile 0 / tile 1 before the current item
            bool ok = true;
            // One K/V block j of the current item.  MORE (compile-time): a block j+1 follows,
            // so S_t(j+1) is issued; otherwise o_done is committed.  LAST2: block j+1 is the
            // item's last, so S_1(j+1) is the item's last read of Q (q_free).  The item's last
            // two blocks run outside the loop, which keeps its body free of these branches.
            //  - bf16: one wait for bundle j+1 (V_j and K_{j+1}, slot u of both rings), P_t V_j
            //    then S_t(j+1) per tile, one release commit after S_1(j+1).
            //  - E4M3 (kPsmem): S_0(j+1) and S_1(j+1) as soon as the softmax warps have read
            //    S_t(j) out of TMEM, then O_t += P_t(j) V_j as each P_t(j) is published; the
            //    bundle is released after P_1(j) V_j.
            // g1: index of bundle j+1 over all items; p0, p1: parity of block j's per-block
            // barriers of tile 0 and tile 1 (passed by value, so the running counters stay out
            // of the loop body)
            auto block = [&](int j, int g1, uint32_t p0, uint32_t p1, auto more_c, auto last2_c) -> bool {
                constexpr bool more = decltype(more_c)::value, last2 = decltype(last2_c)::value;
                const int u = g1 % kStages;
                const uint32_t phu = (g1 / kStages) & 1;
                if constexpr (C::kPsmem) {
                    if (!mbar_wait(smem_u32(&bars.kv_full[u]), phu, lim, &abort_flag)) return false;
                    if constexpr (more) {
                        if (!mbar_wait(smem_u32(&bars.s_free[0]), p0, lim, &abort_flag)) return false;
                        tc_fence_after();
                        issue_s(q_lo0, u, C::kColS0);
                        mma_commit(smem_u32(&bars.s_full[0]));
                        if (!mbar_wait(smem_u32(&bars.s_free[1]), p1, lim, &abort_flag)) return false;
                        tc_fence_after();
                        issue_s(q_lo1, u, C::kColS1);
                        mma_commit(smem_u32(&bars.s_full[1]));
                        if constexpr (last2) mma_commit(smem_u32(&bars.q_free));
                    }
                    if (!mbar_wait(smem_u32(&bars.p_full[0]), p0, lim, &abort_flag)) return false;
                    tc_fence_after();
                    issue_pv_s(p_lo0, u, C::kColO0, j > 0);
                    mma_commit(smem_u32(&bars.pv_done[0]));
                    if constexpr (!more) mma_commit(smem_u32(&bars.o_done[0]));
                    if (!mbar_wait(smem_u32(&bars.p_full[1]), p1, lim, &abort_flag)) return false;
                    tc_fence_after();
                    issue_pv_s(p_lo0 + (C::kPBytes >> 4), u, C::kColO1, j > 0);
                    mma_commit(smem_u32(&bars.pv_done[1]));
                    if constexpr (!more) mma_commit(smem_u32(&bars.o_done[1]));
                } else {
                    if (!mbar_wait(smem_u32(&bars.kv_full[u]), phu, lim, &abort_flag)) return false;
                    if (!mbar_wait(smem_u32(&bars.p_full[0]), p0, lim, &abort_flag)) return false;
                    tc_fence_after();
                    issue_pv(C::kColS0, u, C::kColO0, j > 0);
                    if constexpr (more) {
                        issue_s(q_lo0, u, C::kColS0);
                        mma_commit(smem_u32(&bars.s_full[0]));
                    } else {
                        mma_commit(smem_u32(&bars.o_done[0]));
                    }
                    if (!mbar_wait(smem_u32(&bars.p_full[1]), p1, lim, &abort_flag)) return false;
                    tc_fence_after();
                    issue_pv(C::kColS1, u, C::kColO1, j > 0);
                    if constexpr (more) {
                        issue_s(q_lo1, u, C::kColS1);
                        mma_commit(smem_u32(&bars.s_full[1]));
                        if constexpr (last2) mma_commit(smem_u32(&bars.q_free));
                    } else {
                        mma_commit(smem_u32(&bars.o_done[1]));
                    }
                }
                mma_commit(smem_u32(&bars.kv_empty[u]));  // bundle j+1 read
                return true;
            };
            using T = std::true_type;
            using F = std::false_type;
            int kq = 0;  // items with at least one key block done
            for (int k = 0; ok && k < kItemsMax; ++k) {
                const int x = item_x(k);
                if (x >= n_items) break;
                const Item I = item_at(x);
                if (I.n_kv == 0) continue;  // no key reaches these queries
                ok = mbar_wait(smem_u32(&bars.q_full), kq & 1, lim, &abort_flag);
                if (!ok) break;
                // the item's first scores: bundle 0 holds K_0; with P in shared memory the
                // previous item's last S_t must have been read out of TMEM first
                ok = mbar_wait(smem_u32(&bars.kv_full[gb % kStages]), (gb / kStages) & 1, lim, &abort_flag);
                if (ok && C::kPsmem && c0 > 0) {
                    ok = mbar_wait(smem_u32(&bars.s_free[0]), (c0 - 1) & 1, lim, &abort_flag);
                    if (ok) ok = mbar_wait(smem_u32(&bars.s_free[1]), (c1 - 1) & 1, lim, &abort_flag);
                }
                if (!ok) break;
                tc_fence_after();
                if (kSolo && I.solo) {
                    // One query tile (Q_0); key block b belongs to softmax warpgroup b % 2, whose
                    // S, P and O columns it uses.  Bundle n = {K_n, V_{n-1}}: first S_{n%2}(n)
                    // (those columns held P(n-2), whose P V went out with the previous bundle and
                    // runs first), then P(n-1) V_{n-1} once warpgroup (n-1) % 2 has published it.
                    const int u0 = gb % kStages;
                    issue_s(q_lo0, u0, C::kColS0);
                    mma_commit(smem_u32(&bars.s_full[0]));
                    if (I.n_kv == 1) mma_commit(smem_u32(&bars.q_free));
                    mma_commit(smem_u32(&bars.kv_empty[u0]));  // bundle 0 read
                    for (int n = 1; ok && n <= I.n_kv; ++n) {
                        const int g = gb + n, u = g % kStages;
                        ok = mbar_wait(smem_u32(&bars.kv_full[u]), (g / kStages) & 1, lim, &abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        if (n < I.n_kv) {
                            const int ts = n & 1;
                            issue_s(q_lo0, u, ts ? C::kColS1 : C::kColS0);
                            mma_commit(smem_u32(&bars.s_full[ts]));
                            if (n == I.n_kv - 1) mma_commit(smem_u32(&bars.q_free));
                        }
                        const int b = n - 1, tb = b & 1;
                        ok = mbar_wait(smem_u32(&bars.p_full[tb]), ((tb ? c1 : c0) + b / 2) & 1, lim, &abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(tb ? C::kColS1 : C::kColS0, u, tb ? C::kColO1 : C::kColO0, b >= 2);
                        if (b + 2 >= I.n_kv) mma_commit(smem_u32(&bars.o_done[tb]));  // tile tb's last
                        mma_commit(smem_u32(&bars.kv_empty[u]));  // bundle n read
                    }
                    c0 += (I.n_kv + 1) / 2;
                    c1 += I.n_kv / 2;
                } else {
                    issue_s(q_lo0, gb % kStages, C::kColS0);
                    mma_commit(smem_u32(&bars.s_full[0]));
                    issue_s(q_lo1, gb % kStages, C::kColS1);
                    mma_commit(smem_u32(&bars.s_full[1]));
                    if (I.n_kv == 1) mma_commit(smem_u32(&bars.q_free));
                    mma_commit(smem_u32(&bars.kv_empty[gb % kStages]));  // bundle 0 read
                    const int g0 = gb, a0 = c0, a1 = c1, n = I.n_kv;
                    int j = 0;
                    for (; j + 2 < n && ok; ++j) ok = block(j, g0 + j + 1, (a0 + j) & 1, (a1 + j) & 1, T{}, F{});
                    if (ok && n >= 2) ok = block(n - 2, g0 + n - 1, (a0 + n - 2) & 1, (a1 + n - 2) & 1, T{}, T{});
                    if (ok) ok = block(n - 1, g0 + n, (a0 + n - 1) & 1, (a1 + n - 1) & 1, F{}, F{});
                    c0 += n;
                    c1 += n;
                }
                gb += I.n_kv + 1;
                ++kq;
            }
            if (!ok) record_timeout(args.ctl, &abort_flag);
            // drain every MMA this thread issued before TMEM is released
            mma_commit(smem_u32(&bars.drain));
            const volatile int never = 0;
            mbar_wait(smem_u32(&bars.drain), 0, kDrainWaitNs, &never);
        }
    }
    // warps 2-3 have no role
    } else {
        regs_inc<184>();
        // ================================================================ softmax warpgroups
        const int t = (warp - 4) / 4;              // query tile 0 or 1
        const int wq = warp % 4;                   // TMEM lane quarter
        const int row_in_tile = wq * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t colS = t ? C::kColS1 : C::kColS0;
        const uint32_t colO = t ? C::kColO1 : C::kColO0;
        int gj = 0;  // K/V blocks this warpgroup processed before the current item
        int kd = 0;  // items in which this warpgroup processed at least one key block
        int ns = 0;  // solo items merged
        bool ok = true;
        for (int k = 0; ok && k < kItemsMax; ++k) {
            const int x = item_x(k);
            if (x >= n_items) break;
            const Item I = item_at(x);
            const int n_kv = I.n_kv;
            // solo item: both warpgroups hold the tile's rows, warpgroup t taking key blocks
            // t, t + 2, ...; a solo tile past N has no rows and no keys
            const bool solo = kSolo && I.solo;
            if (solo && n_kv == 0) continue;
            const int tile_r0 = I.r0 + (solo ? 0 : t * kBM);
            const int qrow = tile_r0 + row_in_tile;
            // per-head FP8 descales fold into the score constant and the output scale
            float c = args.c_log2, o_scale = args.o_scale;
            // per-block FP8 descales: this tile's Q factor folds into c, key block j's K factor
            // into c_j = c * kd_j.  V's factor vd_j cannot be applied after P V has been
            // accumulated, so it goes into P before the E4M3 rounding: P'_j = P_j vd_j / vd_max
            // (at most P_j), by adding log2(vd_j / vd_max) <= 0 to the exponent; the row sum
            // adds the block's sum times vd_max / vd_j, and O is scaled by vd_max at the end.
            // The ratio is held at >= 2^-100, where P' is still exact in fp32, so that a zero
            // factor keeps its block's mass in l.
            const float* kd_blk = nullptr;
            const float* vd_blk = nullptr;
            float lg_vmax = 0.f;
            if (PB) {
                const int n_kb = (N_kv + kBN - 1) / kBN;
                c *= args.qk_descale_q[static_cast<size_t>(I.bh) * ((N + kBM - 1) / kBM) + tile_r0 / kBM];
                kd_blk = args.qk_descale_k + static_cast<size_t>(I.bh_kv) * n_kb;
                vd_blk = args.v_descale + static_cast<size_t>(I.bh_kv) * n_kb;
                float vm = 0.f;
                for (int x = lane; x < n_kb; x += 32) vm = fmaxf(vm, vd_blk[x]);
    #pragma unroll
                for (int off = 16; off > 0; off >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
                o_scale = vm;
                lg_vmax = lg2_approx(vm);
            } else if (args.qk_descale_q) {
                c *= args.qk_descale_q[I.bh] * args.qk_descale_k[I.bh_kv];
                o_scale = args.v_descale[I.bh_kv];
            }
            const bool c_pos = c >= 0.f;
            // a masked score must become -inf after the multiply by c
            const uint32_t mask_bits = c_pos ? 0xff800000u : 0x7f800000u;
            float m_ref = -INFINITY;  // reference max in log2 units
            float l = 0.f;

            int i = 0;  // key blocks of this item done by this warpgroup
            for (int j = solo ? t : 0; j < n_kv; j += solo ? 2 : 1, ++i) {
                // key block j's factors (per-block FP8), loaded before the wait
                float cj = c, bj = 0.f, inv_rj = 1.f;
                if (PB) {
                    const float kdj = __ldg(kd_blk + j), vdj = __ldg(vd_blk + j);
                    cj = c * kdj;
                    bj = fmaxf(lg2_approx(vdj) - lg_vmax, -100.f);
                    inv_rj = ex2_approx(-bj);
                }
                ok = mbar_wait(smem_u32(&bars.s_full[t]), (gj + i) & 1, lim, &abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t r[128];
                tmem_ld32_at<0>(lane_base + colS, r);
                tmem_ld32_at<32>(lane_base + colS + 32, r);
                tmem_ld32_at<64>(lane_base + colS + 64, r);
                tmem_ld32_at<96>(lane_base + colS + 96, r);
                tmem_wait_ld_fence(r);
                if constexpr (C::kPsmem) {
                    // S_t(j) is in registers: its columns may take S_t(j+1)
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bars.s_free[t]));
                }

                const int kv0 = j * kBN;
                const int qlast = qrow + delta;  // last key this row reaches when causal
                if ((kv0 + kBN > N_kv) || (args.causal && kv0 + kBN - 1 > qlast)) {
                    // keys >= N_kv, and keys after this query row when causal, drop out
                    const int valid = min(N_kv - kv0, args.causal ? qlast - kv0 + 1 : kBN);
    #pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i >= valid) r[i] = mask_bits;
                }
                // block max of the scaled scores = c * (max of the raw scores) for c >= 0
                const float mt = cj * block_extreme(r, c_pos);
                // lazy rescale: move the reference only when the block max exceeds it by > kTau
                float alpha = 1.f;
                const bool bump = mt > m_ref + kTau;
                if (bump) {
                    alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mt);
                    m_ref = mt;
                    l *= alpha;
                }
                const float ref = (m_ref == -INFINITY) ? 0.f : m_ref;
                const float2 c2 = make_float2(cj, cj), nref2 = make_float2(bj - ref, bj - ref);
                if (C::kPsmem && i > 0) {
                    // P_t(j) replaces P_t(j-1), and O_t may be rescaled, once O_t += P_t(j-1) V
                    // has completed
                    ok = mbar_wait(smem_u32(&bars.pv_done[t]), (gj + i - 1) & 1, lim, &abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                }
                float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
                if (FP8) {
                    uint32_t pk[32];
    #pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 x01 = __ffma2_rn(
                            make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])), c2, nref2);
                        const float2 x23 = __ffma2_rn(
                            make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])), c2, nref2);
                        const float2 p01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
                        const float2 p23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
                        acc0 = __fadd2_rn(acc0, p01);
                        acc1 = __fadd2_rn(acc1, p23);
                        pk[i] = pack_e4m3x4(p01.x, p01.y, p23.x, p23.y);
                    }
                    if constexpr (C::kPsmem) {
                        // this row's 128 bytes in the 128-byte swizzle the MMA reads (16-byte
                        // granule g of row r at g ^ (r % 8)), then visible to the tensor core
                        const uint32_t prow = smem_base + C::kOffP + t * C::kPBytes + row_in_tile * 128;
    #pragma unroll
                        for (int g = 0; g < 8; ++g)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + ((g ^ (row_in_tile & 7)) * 16)),
                                         "r"(pk[4 * g]), "r"(pk[4 * g + 1]), "r"(pk[4 * g + 2]), "r"(pk[4 * g + 3])
                                         : "memory");
                        fence_proxy_async_smem();
                    } else {
                        tmem_st32(lane_base + colS, pk);
                    }
                } else {
    #pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[32];
    #pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int e = 64 * h + 2 * i;
                            const float2 x = __ffma2_rn(
                                make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), c2, nref2);
                            const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            if (i & 1)
                                acc1 = __fadd2_rn(acc1, p);
                            else
                                acc0 = __fadd2_rn(acc0, p);
                            pk[i] = pack_bf16x2(p.x, p.y);
                        }
                        tmem_st32(lane_base + colS + 32 * h, pk);
                    }
                }
                if (i > 0 && __any_sync(0xffffffffu, bump)) {
                    // O_t += P V of this warpgroup's previous block has completed (it precedes
                    // S_t(j) in issue order, or with P in shared memory pv_done said so above),
                    // so O_t can be rescaled in place before P_t(j) is published.
    #pragma unroll
                    for (int q4 = 0; q4 < D / 32; ++q4) {
                        uint32_t ov[32];
                        tmem_ld32(lane_base + colO + 32 * q4, ov);
    #pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(lane_base + colO + 32 * q4, ov);
                    }
                }
                const float rs = (acc0.x + acc0.y) + (acc1.x + acc1.y);
                l = (PB) ? fmaf(rs, inv_rj, l) : l + rs;
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars.p_full[t]));
            }
            gj += i;
            if (ok && i > 0) {
                ok = mbar_wait(smem_u32(&bars.o_done[t]), kd & 1, lim, &abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                ++kd;
            }
            if (!ok) {
                if (lane == 0) record_timeout(args.ctl, &abort_flag);
                break;
            }
            tc_fence_after();
            if (solo) {
                // Two states over disjoint key sets, each relative to its own reference max:
                // (m_0, l_0, O_0) and (m_1, l_1, O_1).  Combined: m = max(m_0, m_1),
                // l = 2^(m_0 - m) l_0 + 2^(m_1 - m) l_1, O = (2^(m_0 - m) O_0 + 2^(m_1 - m) O_1) / l.
                if (t == 1) {
                    merge_m[row_in_tile] = m_ref;
                    merge_l[row_in_tile] = l;
                    mbar_arrive(smem_u32(&bars.merge_ml));
                    // O_1 stays in TMEM until warpgroup 0 has read it
                    ok = mbar_wait(smem_u32(&bars.merge_done), ns & 1, lim, &abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    ++ns;
                    if (!ok) {
                        if (lane == 0) record_timeout(args.ctl, &abort_flag);
                        break;
                    }
                    continue;
                }
                ok = mbar_wait(smem_u32(&bars.merge_ml), ns & 1, lim, &abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                ++ns;
                if (!ok) {
                    if (lane == 0) record_timeout(args.ctl, &abort_flag);
                    break;
                }
                tc_fence_after();
                const float m1 = merge_m[row_in_tile], l1 = merge_l[row_in_tile];
                const float mm = fmaxf(m_ref, m1);
                const float a0 = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mm);
                const float a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - mm);
                const float lsum = a0 * l + a1 * l1;
                const float w0 = a0 * (o_scale / lsum), w1 = a1 * (o_scale / lsum);
                const bool has1 = n_kv >= 2;  // warpgroup 1 had key blocks: O_1 holds them
                const size_t orow = (static_cast<size_t>(I.bh) * N + qrow) * D;
#pragma unroll
                for (int q4 = 0; q4 < D / 32; ++q4) {
                    uint32_t ov[32];
                    tmem_ld32(lane_base + C::kColO0 + 32 * q4, ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * w0);
                    if (has1) {
                        uint32_t ow[32];
                        tmem_ld32(lane_base + C::kColO1 + 32 * q4, ow);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            ov[e] = __float_as_uint(fmaf(__uint_as_float(ow[e]), w1, __uint_as_float(ov[e])));
                    }
                    if (qrow < N) {
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(ov[2 * e]), __uint_as_float(ov[2 * e + 1]));
                        uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + orow + 32 * q4);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            out[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&bars.merge_done));
                if (qrow < N && args.lse != nullptr)
                    args.lse[static_cast<size_t>(I.bh) * N + qrow] = (mm + log2f(lsum)) * 0.69314718055994530942f;
                continue;
            }
            // A row that saw no key (l = 0; only in a causal key shard) gives O = 0 and
            // lse = -inf.  O_t is read before this warp publishes the next item's first P,
            // so the next item's first P V (which overwrites O_t) comes after these loads.
            const float inv = (!SHARD || l > 0.f) ? o_scale / l : 0.f;
            const size_t orow = (static_cast<size_t>(I.bh) * N + qrow) * D;
#pragma unroll
            for (int q4 = 0; q4 < D / 32; ++q4) {
                uint32_t ov[32];
                if (i > 0) {
                    tmem_ld32(lane_base + colO + 32 * q4, ov);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = 0u;
                }
                if (SHARD && qrow < N) {
                    float4* out = reinterpret_cast<float4*>(static_cast<float*>(args.o) + orow + 32 * q4);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        out[i] = make_float4(__uint_as_float(ov[4 * i]) * inv, __uint_as_float(ov[4 * i + 1]) * inv,
                                             __uint_as_float(ov[4 * i + 2]) * inv, __uint_as_float(ov[4 * i + 3]) * inv);
                } else if (qrow < N) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
                    uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + orow + 32 * q4);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        out[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
            if (qrow < N && args.lse != nullptr)
                args.lse[static_cast<size_t>(I.bh) * N + qrow] = (m_ref + log2f(l)) * 0.69314718055994530942f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool FP8, bool SHARD, bool PB = false>
int launch_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int H_kv, int N, int N_kv, int delta, float c_log2, float o_scale,
                const float* qd, const float* kd, const float* vd, int causal, DevCtl ctl,
                cudaStream_t s) {
    const int BH = B * H, BH_kv = B * H_kv;
    using C = Cfg<D, FP8>;
    const CUtensorMapDataType dt =
        FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv;
    int rc = make_map_3d(&tq, q, dt, C::kElem, D, N, BH, C::kBoxX, kBM);
    if (rc == 0) rc = make_map_3d(&tk, k, dt, C::kElem, D, N_kv, BH_kv, C::kBoxX, kBN);
    if (rc == 0) rc = make_map_3d(&tv, v, dt, C::kElem, D, N_kv, BH_kv, C::kBoxX, kBN);
    if (rc != 0) return rc;
    static uint64_t attr_set = 0;  // per template instance, one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(attr_set & (1ull << dev))) {
        cudaError_t e = cudaFuncSetAttribute(fwd_sm103_kernel<D, FP8, SHARD, PB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemAlloc);
        if (e != cudaSuccess) return static_cast<int>(e);
        if (dev < 64) attr_set |= 1ull << dev;
    }
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.N = N;
    a.N_kv = N_kv;
    a.delta = delta;
    a.n_pairs = (N + 2 * kBM - 1) / (2 * kBM);
    a.BH = BH;
    a.c_log2 = c_log2;
    a.o_scale = o_scale;
    a.causal = causal;
    a.H = H;
    a.H_kv = H_kv;
    a.qk_descale_q = qd;
    a.qk_descale_k = kd;
    a.v_descale = vd;
    a.ctl = ctl;
    // bf16: persistent, one CTA per SM (fewer if there are fewer items), each looping over
    // items.  E4M3: one CTA per item (its k-th item is then blockIdx.x alone), placed by the
    // hardware as SMs free up: its items are short, and dealing them statically measured
    // 4-8% slower than letting the next CTA take the first free SM.
    int sms = 152;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int pairs = a.n_pairs * BH;
    a.n_pair_items = pairs;
    a.n_items = pairs;
    int grid = pairs;
    if (!FP8) {
        // When the last round of pairs fills at most half the CTAs, its pairs are dealt as
        // twice as many single tiles, all in that last round (bf16 forward, not shards).
        // Causal items run heaviest first, so after a full round the last one holds the
        // lightest pairs, whose split measured slower: there, only a single round is split.
        const int rounds = (pairs + sms - 1) / sms;
        const int last = pairs - (rounds - 1) * sms;
        if (!SHARD && 2 * last <= sms && (!causal || rounds == 1)) {
            a.n_pair_items = pairs - last;
            a.n_items = pairs + last;
        }
        grid = rounds > 1 ? sms : a.n_items;
    }
    return static_cast<int>(launch_pdl(fwd_sm103_kernel<D, FP8, SHARD, PB>, dim3(grid), dim3(kThreads),
                                       C::kSmemAlloc, s, tq, tk, tv, a));
}

}  // namespace

int launch_fwd_sm103(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int H_kv, int N, int d, float c_log2, float o_scale, const float* qd,
                     const float* kd, const float* vd, int per_block, int causal, bool is_fp8,
                     DevCtl ctl, cudaStream_t s) {
    if (is_fp8 && per_block)
        return launch_impl<128, true, false, true>(q, k, v, o, lse, B, H, H_kv, N, N, 0, c_log2,
                                                   o_scale, qd, kd, vd, causal, ctl, s);
    if (is_fp8)
        return launch_impl<128, true, false>(q, k, v, o, lse, B, H, H_kv, N, N, 0, c_log2,
                                             o_scale, qd, kd, vd, causal, ctl, s);
    if (d == 64)
        return launch_impl<64, false, false>(q, k, v, o, lse, B, H, H_kv, N, N, 0, c_log2,
                                             o_scale, qd, kd, vd, causal, ctl, s);
    return launch_impl<128, false, false>(q, k, v, o, lse, B, H, H_kv, N, N, 0, c_log2, o_scale,
                                          qd, kd, vd, causal, ctl, s);
}

int launch_fwd_kv_shard(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                        int H, int H_kv, int N_q, int N_kv, int d, float c_log2, int causal,
                        int delta, DevCtl ctl, cudaStream_t s) {
    if (d == 64)
        return launch_impl<64, false, true>(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, delta, c_log2,
                                            1.0f, nullptr, nullptr, nullptr, causal, ctl, s);
    return launch_impl<128, false, true>(q, k, v, o, lse, B, H, H_kv, N_q, N_kv, delta, c_log2,
                                         1.0f, nullptr, nullptr, nullptr, causal, ctl, s);
}

}  // namespace fa
