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
// Bandwidth-bound: each partial row is read once (float32), the merged row written
// once.  A thread owns one float4 of a row (d / 4 threads per row, consecutive
// threads on consecutive 16-byte pieces of consecutive rows, so every warp reads
// whole 512-byte row segments); the grid strides over rows.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(256)
    lse_merge_kernel(const float4* __restrict__ o_parts, const float* __restrict__ lse_parts,
                     int n_parts, size_t rows, void* __restrict__ o, float* __restrict__ lse) {
    constexpr int kVec = D / 4;  // float4 pieces per row
    const size_t units = rows * kVec;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t x = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < units;
         x += stride) {
        const size_t row = x / kVec;
        const int c = static_cast<int>(x % kVec);
        float m = -INFINITY;
        for (int s = 0; s < n_parts; ++s) m = fmaxf(m, __ldg(lse_parts + s * rows + row));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float out_lse = -INFINITY;
        if (m != -INFINITY) {
            float tot = 0.f;
            for (int s = 0; s < n_parts; ++s) tot += expf(__ldg(lse_parts + s * rows + row) - m);
            const float inv = 1.f / tot;
#pragma unroll 4
            for (int s = 0; s < n_parts; ++s) {
                const float l = __ldg(lse_parts + s * rows + row);
                if (l == -INFINITY) continue;  // no key of this shard reached the row
                const float w = expf(l - m) * inv;
                const float4 v = __ldcs(o_parts + (s * rows + row) * kVec + c);
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
            out_lse = m + logf(tot);
        }
        if (OUT_F32) {
            reinterpret_cast<float4*>(o)[row * kVec + c] = acc;
        } else {
            reinterpret_cast<uint2*>(o)[row * kVec + c] =
                make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        }
        if (lse != nullptr && c == 0) lse[row] = out_lse;
    }
}

template <int D, bool OUT_F32>
cudaError_t launch_merge_impl(const float* o_parts, const float* lse_parts, int n_parts,
                              size_t rows, void* o, float* lse, cudaStream_t s) {
    int sms = 152, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t units = rows * (D / 4);
    size_t blocks = (units + 255) / 256;
    const size_t cap = static_cast<size_t>(sms) * 8;  // 8 blocks of 256 threads per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    lse_merge_kernel<D, OUT_F32><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        reinterpret_cast<const float4*>(o_parts), lse_parts, n_parts, rows, o, lse);
    return cudaGetLastError();
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
