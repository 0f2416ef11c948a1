// merge.cu -- combine attention outputs computed over disjoint key sets.
//
// The "FlashAttention-1" page (10.2.2) combines two partial softmax states
// (m1, l1) and (m2, l2) over disjoint key blocks through m = max(m1, m2) and
// l = e^(m1-m) l1 + e^(m2-m) l2, each partial output weighted the same way.  A
// key shard's output here is already normalised and carries lse_s = m_s + ln l_s,
// so the combination over S shards is
//     lse = ln sum_s exp(lse_s),    O = sum_s exp(lse_s - lse) O_s,
// computed with the row's largest lse_s subtracted first.  A shard in which a row
// saw no key has lse_s = -inf and weight 0; a row that saw no key in any shard
// gives O = 0 and lse = -inf.
//
// Bandwidth-bound: each partial row that a row's keys reached is read once
// (float32), the merged row written once.  A lane owns one float4 of a row (d / 4
// lanes per row, so a warp reads whole 512-byte row segments); the grid strides
// over rows.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kMaxParts = 16;  // parts per merge (a lane per part for the lse reduction)

// A row is owned by a group of D/4 lanes (one float4 each: the whole row); lane j of
// the group reads lse of part j, the group reduces max and sum with shuffles, and
// every lane then reads its float4 of each part that the row's keys reached, four
// parts' loads in flight at a time.
template <int D, bool OUT_F32>
__global__ void __launch_bounds__(256)
    lse_merge_kernel(const float4* __restrict__ o_parts, const float* __restrict__ lse_parts,
                     int n_parts, size_t rows, void* __restrict__ o, float* __restrict__ lse) {
    constexpr int kVec = D / 4;         // lanes per row
    constexpr int kGroups = 32 / kVec;  // rows per warp
    static_assert(kVec >= kMaxParts, "a lane per part");
    griddep_wait();  // the parts may come from the kernels just before this one
    const int lane = threadIdx.x & 31, j = lane % kVec, g = lane / kVec;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x / 32 * kGroups;
    // the loop bound is the warp's first row, so whole warps iterate together
    for (size_t row = warp * kGroups + g; row - g < rows; row += step) {
        const bool in = row < rows;
        const float l = (in && j < n_parts) ? __ldg(lse_parts + j * rows + row) : -INFINITY;
        float m = l;
#pragma unroll
        for (int off = kVec / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float w = (l == -INFINITY) ? 0.f : expf(l - m);  // exp(lse_j - max), 0 if unreached
        float tot = w;
#pragma unroll
        for (int off = kVec / 2; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s0 = 0; s0 < kMaxParts; s0 += 4) {
            if (s0 >= n_parts) break;  // uniform across the warp
            float ws[4];
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                ws[u] = __shfl_sync(0xffffffffu, w, g * kVec + s0 + u);  // 0 past n_parts
                v[u] = (ws[u] != 0.f) ? __ldcs(o_parts + ((s0 + u) * rows + row) * kVec + j)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc.x = fmaf(ws[u], v[u].x, acc.x);
                acc.y = fmaf(ws[u], v[u].y, acc.y);
                acc.z = fmaf(ws[u], v[u].z, acc.z);
                acc.w = fmaf(ws[u], v[u].w, acc.w);
            }
        }
        if (in) {
            const bool any = m != -INFINITY;
            const float inv = any ? 1.f / tot : 0.f;  // tot >= 1 when any part was reached
            acc.x *= inv;
            acc.y *= inv;
            acc.z *= inv;
            acc.w *= inv;
            if (OUT_F32) {
                reinterpret_cast<float4*>(o)[row * kVec + j] = acc;
            } else {
                reinterpret_cast<uint2*>(o)[row * kVec + j] =
                    make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
            }
            if (lse != nullptr && j == 0) lse[row] = any ? m + logf(tot) : -INFINITY;
        }
    }
}

template <int D, bool OUT_F32>
cudaError_t launch_merge_impl(const float* o_parts, const float* lse_parts, int n_parts,
                              size_t rows, void* o, float* lse, cudaStream_t s) {
    int sms = 152, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // one full wave of resident blocks; the grid strides over the rest
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lse_merge_kernel<D, OUT_F32>, 256,
                                                      0) != cudaSuccess || per_sm < 1)
        per_sm = 4;
    const size_t warps_needed = (rows + (128 / D) - 1) / (128 / D);
    size_t blocks = (warps_needed + 7) / 8;
    const size_t cap = static_cast<size_t>(sms) * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(lse_merge_kernel<D, OUT_F32>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                      reinterpret_cast<const float4*>(o_parts), lse_parts, n_parts, rows, o, lse);
}

}  // namespace

cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int n_parts,
                             size_t rows, int d, void* o, int o_f32, float* lse, cudaStream_t s) {
    if (d == 64)
        return o_f32 ? launch_merge_impl<64, true>(o_parts, lse_parts, n_parts, rows, o, lse, s)
                     : launch_merge_impl<64, false>(o_parts, lse_parts, n_parts, rows, o, lse, s);
    return o_f32 ? launch_merge_impl<128, true>(o_parts, lse_parts, n_parts, rows, o, lse, s)
                 : launch_merge_impl<128, false>(o_parts, lse_parts, n_parts, rows, o, lse, s);
}

}  // namespace fa
