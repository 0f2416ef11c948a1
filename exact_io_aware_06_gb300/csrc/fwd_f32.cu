// fwd_f32.cu -- exact fp32 forward on CUDA cores (FFMA + accurate expf).
//
// Follows the blocked online softmax of the "Flash Attention V1/V2/V3演进"
// page (V1分块原理 / 在线Softmax; Python demo: Q blocks outer, K/V blocks inner,
// running max m, running sum l, unnormalised output, one division at the end)
// with the page's block size of 32 x 32 ("FlashAttention-1", 10.2.3: Br = Bc =
// 32).  Tensor-core TF32 would not meet a 1e-5 bound, so this stays on FFMA.
//
// CTA = 32 query rows of one head, 8 threads per row; thread `sub` of a row
// owns the head dimensions {sub, sub+8, sub+16, ...} so that shared-memory
// reads of a K/V row hit 8 consecutive banks.
#include <cmath>

#include "internal.h"

namespace fa {
namespace {

constexpr int kBr = 32, kBc = 32, kTpr = 8;

template <int D>
__global__ void __launch_bounds__(kBr* kTpr)
    fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                   const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
                   int N, float scale, int causal) {
    constexpr int kDpt = D / kTpr;
    __shared__ float Ks[kBc][D];
    __shared__ float Vs[kBc][D];

    const int bh = blockIdx.y;
    const int r0 = blockIdx.x * kBr;
    const int row = threadIdx.x / kTpr, sub = threadIdx.x % kTpr;
    const int i = r0 + row;
    const size_t base = static_cast<size_t>(bh) * N * D;

    float qr[kDpt], acc[kDpt];
#pragma unroll
    for (int e = 0; e < kDpt; ++e) {
        qr[e] = (i < N) ? q[base + static_cast<size_t>(i) * D + e * kTpr + sub] : 0.f;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int jend = causal ? min(N, r0 + kBr) : N;

    for (int j0 = 0; j0 < jend; j0 += kBc) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kBc * D / 4; idx += kBr * kTpr) {
            const int r = idx / (D / 4), c4 = idx % (D / 4);
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (j0 + r < N) {
                kv = reinterpret_cast<const float4*>(k + base + static_cast<size_t>(j0 + r) * D)[c4];
                vv = reinterpret_cast<const float4*>(v + base + static_cast<size_t>(j0 + r) * D)[c4];
            }
            reinterpret_cast<float4*>(&Ks[r][0])[c4] = kv;
            reinterpret_cast<float4*>(&Vs[r][0])[c4] = vv;
        }
        __syncthreads();

        // scores of this row against the 32 keys of the block
        float s[kBc];
        float mblk = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBc; ++c) {
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < kDpt; ++e) part = fmaf(qr[e], Ks[c][e * kTpr + sub], part);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            const int j = j0 + c;
            const bool masked = (j >= N) || (causal && j > i);
            s[c] = masked ? -INFINITY : part * scale;
            mblk = fmaxf(mblk, s[c]);
        }
        // online update: rescale the old state by exp(m_old - m_new)
        const float m_new = fmaxf(m, mblk);
        const float ref = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - ref);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < kDpt; ++e) acc[e] *= alpha;
#pragma unroll
        for (int c = 0; c < kBc; ++c) {
            const float p = (s[c] == -INFINITY) ? 0.f : expf(s[c] - ref);
            l += p;
#pragma unroll
            for (int e = 0; e < kDpt; ++e) acc[e] = fmaf(p, Vs[c][e * kTpr + sub], acc[e]);
        }
        m = m_new;
    }
    if (i < N) {
        const float inv = 1.f / l;
#pragma unroll
        for (int e = 0; e < kDpt; ++e) o[base + static_cast<size_t>(i) * D + e * kTpr + sub] = acc[e] * inv;
        if (sub == 0 && lse != nullptr) lse[static_cast<size_t>(bh) * N + i] = m + logf(l);
    }
}

}  // namespace

cudaError_t launch_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                           int BH, int N, int d, float scale, int causal, cudaStream_t s) {
    dim3 grid((N + kBr - 1) / kBr, BH);
    dim3 block(kBr * kTpr);
    if (d == 64)
        fwd_f32_kernel<64><<<grid, block, 0, s>>>(q, k, v, o, lse, N, scale, causal);
    else
        fwd_f32_kernel<128><<<grid, block, 0, s>>>(q, k, v, o, lse, N, scale, causal);
    return cudaGetLastError();
}

}  // namespace fa
