// bwd_sm103.cu -- attention backward by recomputation on the sm_103a tensor core.
//
// The "FlashAttention-1" page (10.2.4) keeps only O and the softmax statistics
// from the forward and rebuilds P block by block:
//     P_ij = exp(S_ij - lse_i),  dV = P^T dO,  dP = dO V^T,
//     delta_i = dO_i . O_i,      dS = P o (dP - delta),
//     dQ = scale dS K,           dK = scale dS^T Q.
// (The page's rowsum(dP o P) form of the softmax backward is the same delta:
// rowsum(dP o P)_i = sum_j P_ij dO_i . V_j = dO_i . O_i.)
//
// Three kernels on one stream:
//   1. bwd_prep      delta_i (fp32), lse_i * log2(e) copied into a padded
//                    workspace row, and the fp32 dQ accumulator zeroed.
//   2. bwd_main      persistent, one CTA per SM working through (head, 128-key
//                    block j) items; per item it loops over all 128-row query
//                    blocks i, dK_j and dV_j accumulate in TMEM
//                    for the whole loop, dQ_i partials are added to the fp32
//                    accumulator by TMA bulk tensor reductions (d = 64).
//   3. bwd_dq_convert  dQ = bf16(scale * accumulator).
//
// bwd_main layout (d = 64), 16 warps:
//   warp 0      TMA producer: Q_i, dO_i, lse_i, delta_i in a 3-stage ring that runs
//               across item boundaries
//   warp 1      MMA issuer (dV, S, dK, dP) + TMEM owner
//   warp 2      second MMA issuer: dQ (d = 64 only)
//   warp 3      TMA producer: K_j (two buffers: the next item's K loads while this item
//               runs) and V_j (reloaded as soon as the item's last dP has read it)
//   warps 4-7   P/dS for query columns 0-63 of block i   (thread = key row)
//   warps 8-11  P/dS for query columns 64-127; at an item's end these 8 warps stage dV
//               and dK in the ring stage of the item's last block and warp 4 writes
//               them with TMA stores
//   warps 12-15 drain dQ_i from TMEM into the fp32 accumulator: each warp stages its
//               32 rows in the dS buffer that dQ_i has just consumed (128-byte
//               swizzled boxes) and adds them with TMA bulk tensor reductions
//   TMEM: S^T 0-127 (P^T bf16 over 0-31 and 64-95), dP^T 128-255 (dS^T bf16 over
//         128-159 and 192-223: each half writes only inside the columns it read),
//         dV 256-319, dK 320-383, dQ double buffer 384-447 / 448-511.
//   MMAs per query block i (M = 128 keys or queries), in issue order:
//     dV  += P^T dO_i         (TS, dO_i MN-major)          after P_i is in TMEM
//     S^T  = K_j Q_{i+1}^T    (SS, both K-major)           P_i lives on in registers
//     dK  += dS^T Q_i         (TS, Q_i MN-major)           after dS_i is in TMEM/smem
//     dP^T = V_j dO_{i+1}^T   (SS, both K-major)
//     dQ_i = dS_i K_j         (SS, dS from smem MN-major, K_j MN-major; warp 2)
//   so the next block's scores are ready when the P/dS warps finish dS_i.
#include <cmath>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

constexpr int kBlk = 128;            // keys per CTA, queries per inner step
constexpr float kLog2e = 1.4426950408889634f;

// Add a (32 x 32 fp32) box from shared memory into global memory through the
// tensor map (TMA reduction, f32 add), tracked by the thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                                  int z) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// Store a box from shared memory to global memory through the tensor map (TMA),
// tracked by the thread's bulk async-group; rows past the tensor's end are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// All of this thread's committed bulk operations have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// All of this thread's committed bulk operations have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// d = 64: dK, dV and dQ in one kernel (dQ partials added by TMA bulk reductions).
// d = 128: TMEM holds S^T, dP^T, dV and dK (4 x 128 columns) and nothing else, so
// this kernel computes dK and dV only; bwd_dq_kernel computes dQ.
template <int D>
struct BwdCfg {
    static constexpr bool kFusedDQ = (D == 64);
    static constexpr int kThreads = kFusedDQ ? 512 : 384;
    static constexpr int kQStages = kFusedDQ ? 3 : 2;
    static constexpr int kChunks = D / 64;                    // 128-byte swizzle columns per row
    static constexpr int kTile = kBlk * D * 2;                // bf16 128 x D tile
    // shared memory map (offsets from a 1 KB aligned base)
    // d = 64: two K buffers, so the next item's K loads while this item runs (V, read only
    // by dP, is released one block before the end of an item and reloads in place)
    static constexpr int kKBufs = kFusedDQ ? 2 : 1;
    static constexpr int kOffK = 0;                            // kKBufs
    static constexpr int kOffV = kOffK + kKBufs * kTile;
    static constexpr int kOffQ = kOffV + kTile;               // kQStages
    static constexpr int kOffDO = kOffQ + kQStages * kTile;   // kQStages
    static constexpr int kDSBytes = kBlk * kBlk * 2;
    static constexpr int kOffDS = kOffDO + kQStages * kTile;  // fused: 2 x 32 KB (two 64-query columns)
    static constexpr int kOffL = kOffDS + (kFusedDQ ? 2 * kDSBytes : 0);  // kQStages x 512 B
    static constexpr int kOffDelta = kOffL + kQStages * kBlk * 4;          // kQStages x 512 B
    static constexpr int kSmemBytes = kOffDelta + kQStages * kBlk * 4;
    static constexpr int kSmemAlloc = kSmemBytes + 1024;
    // TMEM columns
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    static constexpr uint32_t kColDQ = 384;                   // fused only
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kIdescSS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
    static constexpr uint32_t kIdescTS = idesc_bf16(128, D, false, true);     // dV, dK
    static constexpr uint32_t kIdescDQ = idesc_bf16(128, D, true, true);      // dQ (A MN-major)
};
static_assert(BwdCfg<64>::kSmemAlloc <= 232448 && BwdCfg<128>::kSmemAlloc <= 232448, "smem");

struct BwdArgs {
    const float* ws_delta;  // [BH][Np], negated: -delta_i
    const float* ws_lse2;   // [BH][Np], negated: -lse_i * log2(e)
    float* dq_acc;          // [BH][Np][d]
    void* dk;
    void* dv;
    int N, Np, n_kv, BH;    // BH: K/V heads (B * H_kv), the grid's head count
    int H, H_kv;            // query heads and K/V heads per batch; H_kv divides H
    int causal;             // 1: key j only reaches queries i >= j
    float c_log2;           // scale * log2(e)
    float scale;
    DevCtl ctl;
};

template <int NQ>
struct Bars {
    uint64_t k_full[2], k_empty[2];  // K buffer (item kc uses buffer kc % kKBufs)
    uint64_t v_full, v_empty;        // the V tile
    uint64_t q_full[NQ], q_empty[NQ];
    uint64_t s_full, dp_full, p_full;
    uint64_t ds_full[2];  // dS_i written (TMEM and dS buffer i % 2); one barrier per buffer
    uint64_t ds_empty[2];
    uint64_t dq_full[2], dq_free[2];
    uint64_t all_done;
    uint64_t epi_staged;  // d = 64: an item's dV, dK staged in shared memory
    uint64_t drain, drain2;
};

__device__ __forceinline__ void record_timeout(const DevCtl& ctl, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(ctl.status, kDevOk, kDevTimeout);
}

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv,
                    const BwdArgs args) {
    using C = BwdCfg<D>;
    constexpr int kD = D, kQStages = C::kQStages, kTile = C::kTile, kChunks = C::kChunks;
    constexpr int kOffK = C::kOffK, kOffV = C::kOffV, kOffQ = C::kOffQ, kOffDO = C::kOffDO;
    constexpr int kOffDS = C::kOffDS, kDSBytes = C::kDSBytes, kOffL = C::kOffL, kOffDelta = C::kOffDelta;
    constexpr uint32_t kColS = C::kColS, kColDP = C::kColDP, kColDV = C::kColDV, kColDK = C::kColDK;
    constexpr uint32_t kColDQ = C::kColDQ, kTmemCols = C::kTmemCols;
    constexpr uint32_t kIdescSS = C::kIdescSS, kIdescTS = C::kIdescTS, kIdescDQ = C::kIdescDQ;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) Bars<kQStages> bars;
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const uint32_t sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* const sb_ptr = smem_raw + (sb - smem_u32(smem_raw));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int N = args.N, Np = args.Np;
    const int n_q = Np / kBlk;
    const int G = args.H / args.H_kv;
    // Persistent: an item is one (K/V head bh, 128-key block kvb); causal items are
    // numbered heaviest first (kvb = 0 meets every query block).  This CTA takes item
    // x = k * gridDim.x + c in round k, with c = blockIdx.x in even rounds and
    // gridDim.x - 1 - blockIdx.x in odd ones: alternating the direction balances the
    // heavy-first causal work across CTAs about as well as dynamic dispatch, and every
    // role can compute the sequence on its own.  Every role numbers the query blocks
    // g = 0, 1, 2, ... across items: stages and barrier phases follow g, the K/V tile
    // and the dK/dV accumulators follow the item count.
    const int n_items = args.n_kv * args.BH;
    auto item_x = [&](int k) {
        const int c = (k & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
        return k * static_cast<int>(gridDim.x) + c;
    };
    struct Item {
        int bh, kvb, i0, n_loc, n_it;
    };
    auto item_at = [&](int x) {
        Item I;
        I.bh = args.causal ? x % args.BH : x / args.n_kv;
        I.kvb = args.causal ? x / args.BH : x % args.n_kv;
        // query blocks this key block meets: all of them, or (causal) blocks kvb..n_q-1;
        // with grouped-query attention, that range for each of the G query heads that
        // share this K/V head (dK, dV sum over all of them)
        I.i0 = args.causal ? I.kvb : 0;
        I.n_loc = n_q - I.i0;
        I.n_it = G * I.n_loc;
        return I;
    };
    auto q_head = [&](const Item& I, int it) {
        return (I.bh / args.H_kv) * args.H + (I.bh % args.H_kv) * G + it / I.n_loc;
    };
    auto q_blk = [&](const Item& I, int it) { return I.i0 + it % I.n_loc; };
    const uint64_t lim = args.ctl.wait_ns;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        // a K buffer is free again once every thread that reads it has committed (the
        // main MMA thread after the item's last S, the dQ thread after its last dQ); V once
        // the main thread's last dP of the item has completed
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars.k_full[b]), 1);
            mbar_init(smem_u32(&bars.k_empty[b]), C::kFusedDQ ? 2 : 1);
        }
        mbar_init(smem_u32(&bars.v_full), 1);
        mbar_init(smem_u32(&bars.v_empty), 1);
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(smem_u32(&bars.q_full[s]), 1);
            mbar_init(smem_u32(&bars.q_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars.ds_empty[s]), 4);  // the four dQ drain warps
            mbar_init(smem_u32(&bars.dq_full[s]), 1);
            mbar_init(smem_u32(&bars.dq_free[s]), 128);
        }
        mbar_init(smem_u32(&bars.s_full), 1);
        mbar_init(smem_u32(&bars.dp_full), 1);
        mbar_init(smem_u32(&bars.p_full), 256);
        mbar_init(smem_u32(&bars.ds_full[0]), 256);
        mbar_init(smem_u32(&bars.ds_full[1]), 256);
        mbar_init(smem_u32(&bars.all_done), 1);
        mbar_init(smem_u32(&bars.epi_staged), 256);
        mbar_init(smem_u32(&bars.drain), 1);
        mbar_init(smem_u32(&bars.drain2), 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        if (C::kFusedDQ) {
            tma_prefetch_desc(&tm_dq);
            tma_prefetch_desc(&tm_dk);
            tma_prefetch_desc(&tm_dv);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // launched while the delta pass may still run: its rows and the zeroed accumulator
    // are read only after it has completed; the pass after this one may start launching
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        // ================================================================ Q / dO producer
        // The ring runs across item boundaries: it waits only for its own stages.
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int k = 0, x = item_x(0); x < n_items && ok; x = item_x(++k)) {
                const Item I = item_at(x);
                for (int i = 0; i < I.n_it; ++i, ++g) {
                    const int s = g % kQStages;
                    const int qb = q_blk(I, i), qh = q_head(I, i);
                    if (g >= kQStages &&
                        !mbar_wait(smem_u32(&bars.q_empty[s]), ((g / kQStages) & 1) ^ 1, lim, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t qf = smem_u32(&bars.q_full[s]);
                    mbar_arrive_expect_tx(qf, 2 * kTile + 2 * kBlk * 4);
                    for (int c = 0; c < kChunks; ++c) {
                        tma_load_3d(sb + kOffQ + s * kTile + c * 16384, &tm_q, qf, 64 * c, qb * kBlk, qh);
                        tma_load_3d(sb + kOffDO + s * kTile + c * 16384, &tm_do, qf, 64 * c, qb * kBlk, qh);
                    }
                    const size_t row = static_cast<size_t>(qh) * Np + static_cast<size_t>(qb) * kBlk;
                    bulk_load(sb + kOffL + s * kBlk * 4, args.ws_lse2 + row, kBlk * 4, qf);
                    bulk_load(sb + kOffDelta + s * kBlk * 4, args.ws_delta + row, kBlk * 4, qf);
                }
            }
            if (!ok) record_timeout(args.ctl, &abort_flag);
            // drain: the newest load of every stage has landed
            const volatile int never = 0;
            for (int q = max(0, g - kQStages); q < g; ++q)
                mbar_wait(smem_u32(&bars.q_full[q % kQStages]), (q / kQStages) & 1, kDrainWaitNs, &never);
        }
    } else if (warp == 3) {
        // ================================================================ K / V producer
        // Item kc's K goes into buffer kc % kKBufs once that buffer's previous item has
        // released it (with two buffers: as soon as the item before this CTA's current one
        // ends); its V once the previous item's last dP has completed.
        if (lane == 0) {
            constexpr int kKB = C::kKBufs;
            int k_issued = 0, v_issued = 0;
            bool ok = true;
            for (int kc = 0, x = item_x(0); x < n_items; x = item_x(++kc)) {
                const Item I = item_at(x);
                const int b = kc % kKB, u = kc / kKB;
                if (u > 0 && !mbar_wait(smem_u32(&bars.k_empty[b]), (u - 1) & 1, lim, &abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t kf = smem_u32(&bars.k_full[b]);
                mbar_arrive_expect_tx(kf, kTile);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_3d(sb + kOffK + b * kTile + c * 16384, &tm_k, kf, 64 * c, I.kvb * kBlk, I.bh);
                k_issued = kc + 1;
                if (kc > 0 && !mbar_wait(smem_u32(&bars.v_empty), (kc - 1) & 1, lim, &abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t vf = smem_u32(&bars.v_full);
                mbar_arrive_expect_tx(vf, kTile);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_3d(sb + kOffV + c * 16384, &tm_v, vf, 64 * c, I.kvb * kBlk, I.bh);
                v_issued = kc + 1;
            }
            if (!ok) record_timeout(args.ctl, &abort_flag);
            // drain: the newest K load of each buffer and the newest V load have landed
            // (also loads for an item the consumers then gave up on)
            const volatile int never = 0;
            for (int kc = max(0, k_issued - kKB); kc < k_issued; ++kc)
                mbar_wait(smem_u32(&bars.k_full[kc % kKB]), (kc / kKB) & 1, kDrainWaitNs, &never);
            if (v_issued > 0) mbar_wait(smem_u32(&bars.v_full), (v_issued - 1) & 1, kDrainWaitNs, &never);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            // Operand descriptors as low words built once (see sdesc_sw128_lo): K-major
            // (leading byte offset 16) for S^T and dP^T, MN-major (16384) for dV and dK.
            // A stage's word is stage 0's plus s * kTile / 16; each MMA adds its K step's
            // offset / 16.
            constexpr uint32_t kDescHi = sdesc_sw128_hi(1024);
            constexpr uint32_t kStage16 = kTile >> 4;
            const uint32_t v_lo = sdesc_sw128_lo(sb + kOffV, 16);
            const uint32_t q_lo = sdesc_sw128_lo(sb + kOffQ, 16), q_mn = sdesc_sw128_lo(sb + kOffQ, 16384);
            const uint32_t do_lo = sdesc_sw128_lo(sb + kOffDO, 16), do_mn = sdesc_sw128_lo(sb + kOffDO, 16384);
            uint32_t k_lo = sdesc_sw128_lo(sb + kOffK, 16);  // this item's K buffer
            auto issue_s = [&](int s) {  // S^T = K_j Q^T into columns 0-127
                const uint32_t ql = q_lo + s * kStage16;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off16 = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    if (kk == 0)
                        mma_ss_w<false, -1>(tmem + kColS, k_lo, ql, kDescHi, kIdescSS, 0u);
                    else
                        mma_ss_w<false, 1>(tmem + kColS, k_lo + off16, ql + off16, kDescHi, kIdescSS);
                }
                mma_commit(smem_u32(&bars.s_full));
            };
            auto issue_dp = [&](int s) {  // dP^T = V_j dO^T into columns 128-255
                const uint32_t dl = do_lo + s * kStage16;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off16 = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    if (kk == 0)
                        mma_ss_w<false, -1>(tmem + kColDP, v_lo, dl, kDescHi, kIdescSS, 0u);
                    else
                        mma_ss_w<false, 1>(tmem + kColDP, v_lo + off16, dl + off16, kDescHi, kIdescSS);
                }
                mma_commit(smem_u32(&bars.dp_full));
            };
            int g = 0, kc = 0;
            bool ok = true;
            for (int k = 0, x = item_x(0); x < n_items && ok; x = item_x(++k), ++kc) {
                const Item I = item_at(x);
                const int kb = kc % C::kKBufs;
                k_lo = sdesc_sw128_lo(sb + kOffK + kb * kTile, 16);
                // the item's first scores; S and dP of the previous item's last block were
                // read by its dV and dK, issued before these by this thread.  K and V are
                // released after their last readers: K after the item's last S (and, d = 64,
                // the dQ thread's last dQ), V after its last dP.
                ok = mbar_wait(smem_u32(&bars.k_full[kb]), (kc / C::kKBufs) & 1, lim, &abort_flag);
                if (ok) ok = mbar_wait(smem_u32(&bars.q_full[g % kQStages]), (g / kQStages) & 1, lim, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_s(g % kQStages);
                if (I.n_it == 1) mma_commit(smem_u32(&bars.k_empty[kb]));
                ok = mbar_wait(smem_u32(&bars.v_full), kc & 1, lim, &abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_dp(g % kQStages);
                if (I.n_it == 1) mma_commit(smem_u32(&bars.v_empty));
                // One query block: dV_i, the next block's S, dK_i, the next block's dP.  MORE:
                // a next block exists; LAST2: that next block is the item's last, so this
                // block issues the item's last S and dP and releases K and V after them.
                // The two flags are compile-time: the item's last two blocks run outside the
                // loop, which keeps the loop body free of the release commits (a conditional
                // commit inside it measured ~100 cycles slower per block).
                auto block = [&](int i, auto more_c, auto last2_c) -> bool {
                    constexpr bool more = decltype(more_c)::value, last2 = decltype(last2_c)::value;
                    const int gi = g + i;
                    const int s = gi % kQStages;
                    const int s1 = (gi + 1) % kQStages;
                    const uint32_t qm = q_mn + s * kStage16, dm = do_mn + s * kStage16;
                    // The loads of block i+1 (ready blocks ahead) are checked together with
                    // P_i: every wait of an issuing thread can leave the tensor pipe idle.
                    // P of an item's first block is computed after the P/dS warps have read
                    // the previous item's dV and dK, so dV, dK may then be overwritten.
                    bool okb = mbar_wait(smem_u32(&bars.p_full), gi & 1, lim, &abort_flag);
                    if (okb && more)
                        okb = mbar_wait(smem_u32(&bars.q_full[s1]), ((gi + 1) / kQStages) & 1, lim, &abort_flag);
                    if (!okb) return false;
                    tc_fence_after();
                    // dV += P^T dO_i
#pragma unroll
                    for (int kk = 0; kk < kBlk / 16; ++kk) {
                        if (kk == 0)
                            mma_ts_w<false, -1>(tmem + kColDV, tmem + kColS, dm, kDescHi, kIdescTS, i > 0 ? 1u : 0u);
                        else
                            mma_ts_w<false, 1>(tmem + kColDV, tmem + kColS + 64 * (kk >> 2) + 8 * (kk & 3),
                                               dm + 128 * kk, kDescHi, kIdescTS);
                    }
                    // next block's scores: the P/dS warps keep P_i in registers
                    if constexpr (more) {
                        issue_s(s1);
                        if constexpr (last2) mma_commit(smem_u32(&bars.k_empty[kb]));  // K's last S
                    }
                    // one barrier per dS buffer: writing buffer gi % 2 again needs block gi's
                    // dK and dQ, so no waiter can fall two phases behind
                    if (!mbar_wait(smem_u32(&bars.ds_full[gi & 1]), (gi >> 1) & 1, lim, &abort_flag))
                        return false;
                    tc_fence_after();
                    // dK += dS^T Q_i
#pragma unroll
                    for (int kk = 0; kk < kBlk / 16; ++kk) {
                        if (kk == 0)
                            mma_ts_w<false, -1>(tmem + kColDK, tmem + kColDP, qm, kDescHi, kIdescTS, i > 0 ? 1u : 0u);
                        else
                            mma_ts_w<false, 1>(tmem + kColDK, tmem + kColDP + 64 * (kk >> 2) + 8 * (kk & 3),
                                               qm + 128 * kk, kDescHi, kIdescTS);
                    }
                    // Q_i, dO_i, lse_i, delta_i consumed.  At d = 64 the item's last block hands
                    // its ring stage to the epilogue instead, which stages dV and dK in it and
                    // releases it once the TMA stores have read them.
                    if constexpr (more || !C::kFusedDQ) mma_commit(smem_u32(&bars.q_empty[s]));
                    if constexpr (more) {
                        issue_dp(s1);
                        if constexpr (last2) mma_commit(smem_u32(&bars.v_empty));  // V's last dP
                    }
                    return true;
                };
                using T = std::true_type;
                using F = std::false_type;
                int i = 0;
                for (; i + 2 < I.n_it && ok; ++i) ok = block(i, T{}, F{});
                if (ok && I.n_it >= 2) ok = block(I.n_it - 2, T{}, T{});
                if (ok) ok = block(I.n_it - 1, F{}, F{});
                if (!ok) break;
                mma_commit(smem_u32(&bars.all_done));  // the item's dV, dK are final
                g += I.n_it;
            }
            if (!ok) record_timeout(args.ctl, &abort_flag);
            mma_commit(smem_u32(&bars.drain));
            const volatile int never = 0;
            mbar_wait(smem_u32(&bars.drain), 0, kDrainWaitNs, &never);
        }
    } else if (C::kFusedDQ && warp == 2) {
        // ================================================================ dQ MMA issuer
        // dQ_i = dS_i K_j (dS from its shared-memory buffer g % 2, K MN-major) into TMEM
        // buffer g % 2.  A second issuing thread: its waits (dS_i, the dQ buffer) do not
        // stall the main MMA chain, and its MMAs read nothing that chain writes (dS in
        // shared memory, K) and write only the dQ buffers.
        if (lane == 0) {
            int g = 0, kc = 0;
            bool ok = true;
            for (int k = 0, x = item_x(0); x < n_items && ok; x = item_x(++k), ++kc) {
                const Item I = item_at(x);
                const int kb = kc % C::kKBufs;
                constexpr uint32_t kDescHi = sdesc_sw128_hi(1024);
                const uint32_t k_mn = sdesc_sw128_lo(sb + kOffK + kb * kTile, 16384);
                ok = mbar_wait(smem_u32(&bars.k_full[kb]), (kc / C::kKBufs) & 1, lim, &abort_flag);
                for (int i = 0; i < I.n_it && ok; ++i) {
                    const int gi = g + i, b = gi & 1;
                    ok = mbar_wait(smem_u32(&bars.ds_full[b]), (gi >> 1) & 1, lim, &abort_flag);
                    if (ok && gi >= 2)
                        ok = mbar_wait(smem_u32(&bars.dq_free[b]), ((gi >> 1) & 1) ^ 1, lim, &abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t ds_mn = sdesc_sw128_lo(sb + kOffDS + b * kDSBytes, 16384);
#pragma unroll
                    for (int kk = 0; kk < kBlk / 16; ++kk) {
                        if (kk == 0)
                            mma_ss_w<false, -1>(tmem + kColDQ + 64 * b, ds_mn, k_mn, kDescHi, kIdescDQ, 0u);
                        else
                            mma_ss_w<false, 1>(tmem + kColDQ + 64 * b, ds_mn + 128 * kk, k_mn + 128 * kk,
                                               kDescHi, kIdescDQ);
                    }
                    mma_commit(smem_u32(&bars.dq_full[b]));  // also: dS buffer b consumed
                }
                if (!ok) break;
                mma_commit(smem_u32(&bars.k_empty[kb]));  // this thread's reads of K are done
                g += I.n_it;
            }
            if (!ok) record_timeout(args.ctl, &abort_flag);
            // drain this thread's MMAs before TMEM is released
            mma_commit(smem_u32(&bars.drain2));
            const volatile int never = 0;
            mbar_wait(smem_u32(&bars.drain2), 0, kDrainWaitNs, &never);
        }
    } else if (warp >= 4 && warp < 12) {
        static_assert(C::kThreads >= 384, "P/dS warpgroups are warps 4-11");
        // ================================================================ P / dS warpgroups
        const int half = (warp - 4) / 4;          // query columns 64*half .. 64*half+63
        const int wq = warp % 4;
        const int key_in_blk = wq * 32 + lane;
        const uint32_t lb = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float2 c2 = make_float2(args.c_log2, args.c_log2);
        int epi_stage = -1;  // warp 4 lane 0: the ring stage whose dV/dK stores are in flight
        bool ok = true;
        int g = 0, kc = 0;
        for (int k = 0, x = item_x(0); x < n_items && ok; x = item_x(++k), ++kc) {
            const Item I = item_at(x);
            for (int i = 0; i < I.n_it; ++i) {
                const int gi = g + i;
                const int s = gi % kQStages;
                // causal diagonal block: key k only reaches queries q >= k of the block
                const bool diag = args.causal && (q_blk(I, i) == I.kvb);
                ok = mbar_wait(smem_u32(&bars.q_full[s]), (gi / kQStages) & 1, lim, &abort_flag);
                if (ok) ok = mbar_wait(smem_u32(&bars.s_full), gi & 1, lim, &abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                // -lse_i * log2(e) and -delta_i of this block's 64 queries
                const float2* L2 = reinterpret_cast<const float2*>(sb_ptr + kOffL + s * kBlk * 4) + 32 * half;
                const float2* D2 = reinterpret_cast<const float2*>(sb_ptr + kOffDelta + s * kBlk * 4) + 32 * half;
                uint32_t pk[32];  // P^T row (64 queries) as bf16 pairs
                {
                    uint32_t r[2][32];
                    tmem_ld32_async(lb + kColS + 64 * half, r[0]);
                    tmem_ld32_async(lb + kColS + 64 * half + 32, r[1]);
                    tmem_wait_ld();
                    reg_fence(r[0]);
                    reg_fence(r[1]);
#pragma unroll
                    for (int x2 = 0; x2 < 32; ++x2) {
                        const uint32_t* rr = r[x2 / 16];
                        const int e = 2 * (x2 % 16);
                        float2 a = __ffma2_rn(make_float2(__uint_as_float(rr[e]), __uint_as_float(rr[e + 1])),
                                              c2, L2[x2]);
                        if (diag) {
                            const int q0 = 64 * half + 32 * (x2 / 16) + e;
                            if (key_in_blk > q0) a.x = -INFINITY;
                            if (key_in_blk > q0 + 1) a.y = -INFINITY;
                        }
                        pk[x2] = pack_bf16x2(ex2_approx(a.x), ex2_approx(a.y));
                    }
                }
                // P^T of this half goes inside the columns this half read (the other half's
                // scores may still be unread): queries 64h..64h+63 -> columns 64h..64h+31
                tmem_st32(lb + kColS + 64 * half, pk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars.p_full));

                // dS^T = P^T o (dP^T - delta)
                const int b = gi & 1;
                ok = mbar_wait(smem_u32(&bars.dp_full), gi & 1, lim, &abort_flag);
                if (C::kFusedDQ && ok && gi >= 2)
                    ok = mbar_wait(smem_u32(&bars.ds_empty[b]), ((gi >> 1) & 1) ^ 1, lim, &abort_flag);
                // the previous item's dV, dK stores: once they have read their ring stage,
                // hand it back to the producer (normally long done by now)
                if (C::kFusedDQ && warp == 4 && lane == 0 && epi_stage >= 0) {
                    bulk_wait_read_all();
                    mbar_arrive(smem_u32(&bars.q_empty[epi_stage]));
                    epi_stage = -1;
                }
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint8_t* dsrow = sb_ptr + kOffDS + b * kDSBytes + half * 16384 + key_in_blk * 128;
                // dP^T of this half's 64 queries in two 32-column loads; the second load runs
                // while the first 32 queries' dS is stored
                uint32_t r[32];
                tmem_ld32_async(lb + kColDP + 64 * half, r);
                tmem_wait_ld();
                reg_fence(r);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t w[16];
#pragma unroll
                    for (int x2 = 0; x2 < 16; ++x2) {
                        const uint32_t pp = pk[16 * h + x2];
                        const float2 p = make_float2(__uint_as_float(pp << 16), __uint_as_float(pp & 0xFFFF0000u));
                        const float2 gg = __fadd2_rn(make_float2(__uint_as_float(r[2 * x2]), __uint_as_float(r[2 * x2 + 1])),
                                                     D2[16 * h + x2]);
                        const float2 ds = __fmul2_rn(p, gg);
                        w[x2] = pack_bf16x2(ds.x, ds.y);
                    }
                    if (h == 0) tmem_ld32_async(lb + kColDP + 64 * half + 32, r);
                    tmem_st16(lb + kColDP + 64 * half + 16 * h, w);
                    if constexpr (C::kFusedDQ) {
                        // queries 64*half + 32h .. +31 of this key row -> MN-major swizzled A tile
                        // for dQ: column `half`, row = key, 16-byte granule ((query % 64) / 8) ^ (key % 8)
#pragma unroll
                        for (int g4 = 0; g4 < 4; ++g4) {
                            const int gran = (h * 4 + g4) ^ (key_in_blk & 7);
                            *reinterpret_cast<uint4*>(dsrow + gran * 16) =
                                make_uint4(w[4 * g4], w[4 * g4 + 1], w[4 * g4 + 2], w[4 * g4 + 3]);
                        }
                    }
                    if (h == 0) {
                        tmem_wait_ld();
                        reg_fence(r);
                    }
                }
                tmem_st_wait();
                if constexpr (C::kFusedDQ) fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars.ds_full[gi & 1]));
            }
            if (!ok) break;
            if constexpr (C::kFusedDQ) {
                // epilogue (d = 64): warps 4-7 stage dV, warps 8-11 dK (times scale) as
                // 128-byte swizzled 128 x 64 boxes in the Q/dO ring stage of the item's last
                // block (dV over its dO tile, dK over its Q tile), free once that block's dV
                // and dK have completed (all_done); one thread writes them with TMA stores of
                // whole lines and hands the stage back to the producer once the stores have
                // read it, at its next dS phase, so the stores' latency stays off the next
                // item's first blocks.
                const int sl = (g + I.n_it - 1) % kQStages;
                ok = mbar_wait(smem_u32(&bars.all_done), kc & 1, lim, &abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint32_t box = sb + (half ? kOffQ : kOffDO) + sl * kTile;
                const float sc = half ? args.scale : 1.0f;
                const uint32_t col = half ? kColDK : kColDV;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
                    tmem_ld32(lb + col + 32 * h, r);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int gran = (h * 4 + c4) ^ (key_in_blk & 7);
                        const float* f = reinterpret_cast<const float*>(r) + 8 * c4;
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(box + key_in_blk * 128 + gran * 16),
                                     "r"(pack_bf16x2(f[0] * sc, f[1] * sc)), "r"(pack_bf16x2(f[2] * sc, f[3] * sc)),
                                     "r"(pack_bf16x2(f[4] * sc, f[5] * sc)), "r"(pack_bf16x2(f[6] * sc, f[7] * sc))
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();  // generic-proxy writes -> visible to the TMA unit
                mbar_arrive(smem_u32(&bars.epi_staged));
                if (warp == 4 && lane == 0) {
                    if (mbar_wait(smem_u32(&bars.epi_staged), kc & 1, lim, &abort_flag)) {
                        tma_store_3d(&tm_dv, sb + kOffDO + sl * kTile, 0, I.kvb * kBlk, I.bh);
                        tma_store_3d(&tm_dk, sb + kOffQ + sl * kTile, 0, I.kvb * kBlk, I.bh);
                        bulk_commit_group();
                        epi_stage = sl;
                    } else {
                        ok = false;
                    }
                }
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                g += I.n_it;
                continue;
            }
            // epilogue (d = 128): warps 4-7 store dV, warps 8-11 store dK (times scale).
            // Their TMEM reads finish before these warps compute the next item's first P.
            ok = mbar_wait(smem_u32(&bars.all_done), kc & 1, lim, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int key = I.kvb * kBlk + key_in_blk;
            const float sc = half ? args.scale : 1.0f;
            void* dst = half ? args.dk : args.dv;
            const uint32_t col = half ? kColDK : kColDV;
            uint16_t* out = static_cast<uint16_t*>(dst) + (static_cast<size_t>(I.bh) * N + key) * kD;
#pragma unroll
            for (int h = 0; h < kD / 32; ++h) {
                uint32_t r[32];
                tmem_ld32(lb + col + 32 * h, r);
                if (key < N) {
                    uint4* o4 = reinterpret_cast<uint4*>(out + 32 * h);
#pragma unroll
                    for (int x2 = 0; x2 < 4; ++x2)
                        o4[x2] = make_uint4(
                            pack_bf16x2(__uint_as_float(r[8 * x2]) * sc, __uint_as_float(r[8 * x2 + 1]) * sc),
                            pack_bf16x2(__uint_as_float(r[8 * x2 + 2]) * sc, __uint_as_float(r[8 * x2 + 3]) * sc),
                            pack_bf16x2(__uint_as_float(r[8 * x2 + 4]) * sc, __uint_as_float(r[8 * x2 + 5]) * sc),
                            pack_bf16x2(__uint_as_float(r[8 * x2 + 6]) * sc, __uint_as_float(r[8 * x2 + 7]) * sc));
                }
            }
            g += I.n_it;
        }
        // d = 64: the dV, dK stores complete before the CTA's shared memory goes away
        if (C::kFusedDQ && warp == 4 && lane == 0) bulk_wait_all();
        if (!ok && lane == 0) record_timeout(args.ctl, &abort_flag);
    } else if (C::kFusedDQ && warp >= 12) {
        // ================================================================ dQ drain
        // dQ_i (fp32, TMEM) -> this warp's 32 rows staged in dS buffer b, which the dQ_i
        // MMA has finished reading once dq_full[b] completes -> two TMA reductions
        // (32 rows x 32 columns each) into the accumulator.  The staging uses the
        // 128-byte swizzle of the tensor map (16-byte chunk c of row r at chunk
        // c ^ (r % 8)), so the 32 lanes' row writes hit distinct banks.  Buffer b is
        // handed back to the P/dS warps (ds_empty[b]) once the reductions have read it.
        const int wq = warp % 4;
        const uint32_t lb = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        bool ok = true;
        int g = 0;
        for (int k = 0, x = item_x(0); x < n_items && ok; x = item_x(++k)) {
            const Item I = item_at(x);
            for (int i = 0; i < I.n_it; ++i) {
                const int gi = g + i, b = gi & 1;
                ok = mbar_wait(smem_u32(&bars.dq_full[b]), (gi >> 1) & 1, lim, &abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t r[2][32];
                tmem_ld32_async(lb + kColDQ + 64 * b, r[0]);
                tmem_ld32_async(lb + kColDQ + 64 * b + 32, r[1]);
                tmem_wait_ld();
                reg_fence(r[0]);
                reg_fence(r[1]);
                tc_fence_before();
                mbar_arrive(smem_u32(&bars.dq_free[b]));
                const uint32_t box0 = sb + kOffDS + b * kDSBytes + wq * 8192;  // two 4 KB boxes
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t dst = box0 + h * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                                     "r"(r[h][4 * c]), "r"(r[h][4 * c + 1]), "r"(r[h][4 * c + 2]),
                                     "r"(r[h][4 * c + 3])
                                     : "memory");
                    }
                fence_proxy_async_smem();  // generic-proxy writes -> visible to the TMA unit
                __syncwarp();
                if (lane == 0) {
                    const int y = q_blk(I, i) * kBlk + wq * 32;
                    tma_reduce_add_3d(&tm_dq, box0, 0, y, q_head(I, i));
                    tma_reduce_add_3d(&tm_dq, box0 + 4096, 32, y, q_head(I, i));
                    bulk_commit_group();
                    bulk_wait_read_all();
                    mbar_arrive(smem_u32(&bars.ds_empty[b]));
                }
                __syncwarp();
            }
            g += I.n_it;
        }
        // the reductions must complete before the CTA's shared memory goes away
        if (lane == 0) bulk_wait_all();
        if (!ok && lane == 0) record_timeout(args.ctl, &abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- pre / post passes
// -delta_i = -(dO_i . O_i) and -lse_i * log2(e) (rows past N: 0 and -inf, so
// that recomputed P is exactly 0 there), dQ accumulator zeroed.  Both are stored
// negated so the main kernel adds them with packed FMA/FADD.
// D/8 threads per row, each reading 16 bytes of O and dO.
template <int D>
__global__ void bwd_prep_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO,
                                const float* __restrict__ lse, float* __restrict__ ws_delta,
                                float* __restrict__ ws_lse2, float4* __restrict__ dq_acc, int BH,
                                int N, int Np, size_t acc_vec4) {
    griddep_wait();               // O, dO may come from the kernel before this one
    griddep_launch_dependents();  // the main kernel may launch and set up meanwhile
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t rows = static_cast<size_t>(BH) * Np;
    constexpr int kT = D / 8;  // threads per row (8 or 16): the shuffles stay inside a warp
    for (size_t base = tid; base < rows * kT; base += nthreads) {
        const size_t r = base / kT;
        const int part = static_cast<int>(base % kT);
        const int bh = static_cast<int>(r / Np), i = static_cast<int>(r % Np);
        float sum = 0.f;
        if (i < N) {
            const size_t src = (static_cast<size_t>(bh) * N + i) * kT + part;
            const uint4 a = o[src], b = dO[src];
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                sum = fmaf(__uint_as_float(av[x] << 16), __uint_as_float(bv[x] << 16), sum);
                sum = fmaf(__uint_as_float(av[x] & 0xFFFF0000u), __uint_as_float(bv[x] & 0xFFFF0000u), sum);
            }
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        if (kT == 16) sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        if (part == 0) {
            ws_delta[r] = -sum;
            ws_lse2[r] = (i < N) ? -lse[static_cast<size_t>(bh) * N + i] * kLog2e : -INFINITY;
        }
    }
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (size_t x = tid; x < acc_vec4; x += nthreads) dq_acc[x] = z;
}

// dQ = bf16(scale * accumulator) for rows < N (d = 64); 8 elements per thread.
__global__ void bwd_dq_convert_kernel(const float4* __restrict__ acc, uint4* __restrict__ dq,
                                      int N, int Np, size_t n_vec8, float scale) {
    griddep_wait();  // launched while the main kernel may still run
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
    constexpr int kVecPerRow = 64 / 8;
    for (size_t x = tid; x < n_vec8; x += nthreads) {
        const size_t row = x / kVecPerRow;  // row in [BH][N]
        const int part = static_cast<int>(x % kVecPerRow);
        const size_t bh = row / N, i = row % N;
        const size_t src = ((bh * Np + i) * kVecPerRow + part) * 2;
        const float4 a = acc[src], b = acc[src + 1];
        dq[x] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                           pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
    }
}

int grid_for(size_t work, int threads, int max_blocks) {
    size_t b = (work + threads - 1) / threads;
    if (b > static_cast<size_t>(max_blocks)) b = max_blocks;
    return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace

size_t bwd_workspace_bytes(int BH, int N, int d) {
    // -delta and -lse*log2(e) rows, plus the fp32 dQ accumulator when d = 64
    const size_t Np = static_cast<size_t>(round_up(N, kBlk));
    const size_t acc = (d == 64) ? static_cast<size_t>(BH) * Np * d : 0;
    return (2 * static_cast<size_t>(BH) * Np + acc) * sizeof(float);
}

namespace {

template <int D>
int launch_bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, void* workspace, int B, int H,
                    int H_kv, int N, float scale, int causal, DevCtl ctl, cudaStream_t s) {
    using C = BwdCfg<D>;
    const int BH = B * H, BH_kv = B * H_kv;  // query heads; K/V heads
    const int Np = round_up(N, kBlk);
    float* ws = static_cast<float*>(workspace);
    float* ws_delta = ws;
    float* ws_lse2 = ws + static_cast<size_t>(BH) * Np;
    float* dq_acc = C::kFusedDQ ? ws + 2 * static_cast<size_t>(BH) * Np : nullptr;

    int sms = 152, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t acc_vec4 = C::kFusedDQ ? static_cast<size_t>(BH) * Np * D / 4 : 0;
    cudaError_t e = launch_pdl(bwd_prep_kernel<D>, dim3(grid_for(static_cast<size_t>(BH) * Np * (D / 8), 256, sms * 8)),
                               dim3(256), 0, s, static_cast<const uint4*>(o), static_cast<const uint4*>(dO), lse,
                               ws_delta, ws_lse2, reinterpret_cast<float4*>(dq_acc), BH, N, Np, acc_vec4);
    if (e != cudaSuccess) return static_cast<int>(e);

    CUtensorMap tq, tk, tv, tdo;
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    int rc = make_map_3d(&tq, q, dt, 2, D, N, BH, 64, kBlk);
    if (rc == 0) rc = make_map_3d(&tk, k, dt, 2, D, N, BH_kv, 64, kBlk);
    if (rc == 0) rc = make_map_3d(&tv, v, dt, 2, D, N, BH_kv, 64, kBlk);
    if (rc == 0) rc = make_map_3d(&tdo, dO, dt, 2, D, N, BH, 64, kBlk);
    // fp32 accumulator [BH][Np][64], reduced into in 32 x 32 boxes (fused dQ only)
    CUtensorMap tdq = tq, tdk = tq, tdv = tq;
    if (rc == 0 && C::kFusedDQ)
        rc = make_map_3d(&tdq, dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, Np, BH, 32, 32);
    // dK, dV [BH_kv][N][64] bf16, written in (64 x 128) boxes (fused d = 64 epilogue)
    if (rc == 0 && C::kFusedDQ) rc = make_map_3d(&tdk, dk, dt, 2, D, N, BH_kv, 64, kBlk);
    if (rc == 0 && C::kFusedDQ) rc = make_map_3d(&tdv, dv, dt, 2, D, N, BH_kv, 64, kBlk);
    if (rc != 0) return rc;
    static uint64_t attr_set = 0;
    if (dev >= 64 || !(attr_set & (1ull << dev))) {
        e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemAlloc);
        if (e != cudaSuccess) return static_cast<int>(e);
        if (dev < 64) attr_set |= 1ull << dev;
    }
    BwdArgs a;
    a.ws_delta = ws_delta;
    a.ws_lse2 = ws_lse2;
    a.dq_acc = dq_acc;
    a.dk = dk;
    a.dv = dv;
    a.N = N;
    a.Np = Np;
    a.n_kv = Np / kBlk;
    a.BH = BH_kv;
    a.H = H;
    a.H_kv = H_kv;
    a.causal = causal ? 1 : 0;
    a.c_log2 = scale * kLog2e;
    a.scale = scale;
    a.ctl = ctl;
    // persistent: one CTA per SM (fewer if there are fewer items), each looping over items
    const int n_items = a.n_kv * BH_kv;
    const int grid = n_items < sms ? n_items : sms;
    // Non-causal: launched with programmatic serialization, so its set-up overlaps the
    // delta pass.  Causal: an ordinary launch.  The causal items are dealt heaviest first
    // on the assumption that every CTA starts together; under programmatic launch the
    // CTAs start as the delta pass drains from their SMs, and the staggered start left
    // the heavy items' CTAs ~10% behind (B4 H16 N2048 d64: 146 -> 133 us).
    if (causal) {
        bwd_main_kernel<D><<<grid, C::kThreads, C::kSmemAlloc, s>>>(tq, tk, tv, tdo, tdq, tdk, tdv, a);
        e = cudaGetLastError();
    } else {
        e = launch_pdl(bwd_main_kernel<D>, dim3(grid), dim3(C::kThreads), C::kSmemAlloc, s, tq, tk, tv,
                       tdo, tdq, tdk, tdv, a);
    }
    if (e != cudaSuccess) return static_cast<int>(e);

    if constexpr (C::kFusedDQ) {
        const size_t n_vec8 = static_cast<size_t>(BH) * N * D / 8;
        return static_cast<int>(launch_pdl(bwd_dq_convert_kernel, dim3(grid_for(n_vec8, 256, sms * 8)),
                                           dim3(256), 0, s, reinterpret_cast<const float4*>(dq_acc),
                                           static_cast<uint4*>(dq), N, Np, n_vec8, scale));
    } else {
        // dQ by its own query-parallel kernel: recompute S and dP per query block
        return launch_bwd_dq(q, k, v, dO, ws_lse2, ws_delta, dq, B, H, H_kv, N, D, scale, causal,
                             ctl, s);
    }
}

}  // namespace

int launch_bwd_sm103(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv, void* workspace, int B, int H,
                     int H_kv, int N, int d, float scale, int causal, DevCtl ctl, cudaStream_t s) {
    if (d == 64)
        return launch_bwd_impl<64>(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, H, H_kv, N, scale,
                                   causal, ctl, s);
    if (d == 128)
        return launch_bwd_impl<128>(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, H, H_kv, N,
                                    scale, causal, ctl, s);
    return -1;
}

}  // namespace fa
