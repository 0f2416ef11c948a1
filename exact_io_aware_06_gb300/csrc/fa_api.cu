// fa_api.cu -- the extern "C" entry points declared in include/fa.h:
// argument checks, the per-device status word, and dispatch to the kernels.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

__device__ int g_status;  // first device-side error since the last query (per device)

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_mu;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

// Address of this device's status word (looked up once per device).
int* status_word(int* err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = FA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) {
            *err = FA_ERR_CUDA;
            return nullptr;
        }
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 int B, int H, int N) {
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
    if (lse != nullptr && !aligned16(lse)) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (!sizes_supported(B, H, N)) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

int from_cuda(int rc) { return rc == 0 ? FA_OK : FA_ERR_CUDA; }

__global__ void wait_selftest_kernel(DevCtl ctl) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    // nobody arrives on this barrier: the bounded wait must give up
    if (!mbar_wait(smem_u32(&bar), 0, ctl.wait_ns, &abort_flag)) {
        if (threadIdx.x == 0) atomicCAS(ctl.status, kDevOk, kDevTimeout);
    }
}

}  // namespace

cudaError_t launch_wait_selftest(DevCtl ctl, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(ctl);
    return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

extern "C" {

__attribute__((visibility("default"))) const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
        default: return "FA_ERR_UNKNOWN";
    }
}

__attribute__((visibility("default"))) void fa_set_wait_timeout_ns(uint64_t ns) {
    g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns);
}

__attribute__((visibility("default"))) int fa_fwd(const void* q, const void* k, const void* v,
                                                  void* o, float* lse, int B, int H, int N, int d,
                                                  float scale, int causal, int dtype,
                                                  void* stream) {
    int rc = check_common(q, k, v, o, lse, B, H, N);
    if (rc != FA_OK) return rc;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F32 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int BH = B * H;
    if (dtype == FA_F32)
        return from_cuda(launch_fwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                        static_cast<const float*>(v), static_cast<float*>(o), lse,
                                        BH, N, d, scale, causal ? 1 : 0, s));
    int err = FA_OK;
    int* st = status_word(&err);
    if (st == nullptr) return err;
    DevCtl ctl{st, g_wait_ns.load()};
    const float c_log2 = scale * 1.4426950408889634f;
    return from_cuda(
        launch_fwd_sm103(q, k, v, o, lse, B, H, H, N, d, c_log2, 1.0f, nullptr, nullptr, nullptr, 0,
                         causal ? 1 : 0, false, ctl, s));
}

__attribute__((visibility("default"))) int fa_fwd_fp8(const void* q8, const void* k8,
                                                      const void* v8, void* o, float* lse,
                                                      float q_descale, float k_descale,
                                                      float v_descale, int B, int H, int N, int d,
                                                      float scale, int causal, void* stream) {
    int rc = check_common(q8, k8, v8, o, lse, B, H, N);
    if (rc != FA_OK) return rc;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    for (float x : {q_descale, k_descale, v_descale})
        if (!std::isfinite(x) || !(x > 0.f)) return FA_ERR_INVALID_ARG;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    int err = FA_OK;
    int* st = status_word(&err);
    if (st == nullptr) return err;
    DevCtl ctl{st, g_wait_ns.load()};
    const float c_log2 = scale * q_descale * k_descale * 1.4426950408889634f;
    return from_cuda(launch_fwd_sm103(q8, k8, v8, o, lse, B, H, H, N, d, c_log2, v_descale, nullptr,
                                      nullptr, nullptr, 0, causal ? 1 : 0, true, ctl,
                                      static_cast<cudaStream_t>(stream)));
}

__attribute__((visibility("default"))) int fa_fwd_gqa(const void* q, const void* k, const void* v,
                                                      void* o, float* lse, int B, int H, int H_kv,
                                                      int N, int d, float scale, int causal,
                                                      int dtype, void* stream) {
    int rc = check_common(q, k, v, o, lse, B, H, N);
    if (rc != FA_OK) return rc;
    if (!std::isfinite(scale) || H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F32 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 || (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
    int err = FA_OK;
    int* st = status_word(&err);
    if (st == nullptr) return err;
    DevCtl ctl{st, g_wait_ns.load()};
    const float c_log2 = scale * 1.4426950408889634f;
    return from_cuda(launch_fwd_sm103(q, k, v, o, lse, B, H, H_kv, N, d, c_log2, 1.0f, nullptr,
                                      nullptr, nullptr, 0, causal ? 1 : 0, false, ctl,
                                      static_cast<cudaStream_t>(stream)));
}

__attribute__((visibility("default"))) int fa_fwd_fp8_per_head(
    const void* q8, const void* k8, const void* v8, void* o, float* lse, const float* q_descale,
    const float* k_descale, const float* v_descale, int B, int H, int N, int d, float scale,
    int causal, void* stream) {
    int rc = check_common(q8, k8, v8, o, lse, B, H, N);
    if (rc != FA_OK) return rc;
    if (!std::isfinite(scale) || q_descale == nullptr || k_descale == nullptr ||
        v_descale == nullptr)
        return FA_ERR_INVALID_ARG;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    int err = FA_OK;
    int* st = status_word(&err);
    if (st == nullptr) return err;
    DevCtl ctl{st, g_wait_ns.load()};
    const float c_log2 = scale * 1.4426950408889634f;
    return from_cuda(launch_fwd_sm103(q8, k8, v8, o, lse, B, H, H, N, d, c_log2, 1.0f, q_descale,
                                      k_descale, v_descale, 0, causal ? 1 : 0, true, ctl,
                                      static_cast<cudaStream_t>(stream)));
}

__attribute__((visibility("default"))) int fa_fwd_fp8_per_block(
    const void* q8, const void* k8, const void* v8, void* o, float* lse, const float* q_descale,
    const float* k_descale, const float* v_descale, int B, int H, int N, int d, float scale,
    int causal, void* stream) {
    int rc = check_common(q8, k8, v8, o, lse, B, H, N);
    if (rc != FA_OK) return rc;
    if (!std::isfinite(scale) || q_descale == nullptr || k_descale == nullptr ||
        v_descale == nullptr)
        return FA_ERR_INVALID_ARG;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    int err = FA_OK;
    int* st = status_word(&err);
    if (st == nullptr) return err;
    DevCtl ctl{st, g_wait_ns.load()};
    const float c_log2 = scale * 1.4426950408889634f;
    return from_cuda(launch_fwd_sm103(q8, k8, v8, o, lse, B, H, H, N, d, c_log2, 1.0f, q_descale,
                                      k_descale, v_descale, 1, causal ? 1 : 0, true, ctl,
                                      static_cast<cudaStream_t>(stream)));
}

__attribute__((visibility("default"))) int fa_fwd_kv_shard(
    const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B, int H,
    int H_kv, int N_q, int N_kv, int d, float scale, int causal, long long q_offset,
    long long kv_offset, int dtype, void* stream) {
    int rc = check_common(q, k, v, o_part, lse_part, B, H, N_q);
    if (rc != FA_OK) return rc;
    if (lse_part == nullptr || N_kv < 1) return FA_ERR_INVALID_ARG;
    if (N_kv > (1 << 24)) return FA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F32 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 || (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
    // key j reaches query i iff kv_offset + j <= q_offset + i; beyond these bounds the
    // offset difference no longer changes which keys a row sees
    long long delta = q_offset - kv_offset;
    if (delta > N_kv) delta = N_kv;
    if (delta < -static_cast<long long>(N_q) - 1) delta = -static_cast<long long>(N_q) - 1;
    int err = FA_OK;
    int* st = status_word(&err);
    if (st == nullptr) return err;
    DevCtl ctl{st, g_wait_ns.load()};
    const float c_log2 = scale * 1.4426950408889634f;
    return from_cuda(launch_fwd_kv_shard(q, k, v, o_part, lse_part, B, H, H_kv, N_q, N_kv, d,
                                         c_log2, causal ? 1 : 0, static_cast<int>(delta), ctl,
                                         static_cast<cudaStream_t>(stream)));
}

__attribute__((visibility("default"))) int fa_lse_merge(const float* o_parts,
                                                        const float* lse_parts, int n_parts,
                                                        void* o, float* lse, int B, int H, int N,
                                                        int d, int dtype, void* stream) {
    if (o_parts == nullptr || lse_parts == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
    if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o)) return FA_ERR_INVALID_ARG;
    if (lse != nullptr && !aligned16(lse)) return FA_ERR_INVALID_ARG;
    if (n_parts < 1 || B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F32 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || n_parts > 16) return FA_ERR_UNSUPPORTED;
    const size_t rows = static_cast<size_t>(B) * H * N;
    if (rows * static_cast<size_t>(n_parts) > (static_cast<size_t>(1) << 40))
        return FA_ERR_UNSUPPORTED;
    return from_cuda(static_cast<int>(launch_lse_merge(o_parts, lse_parts, n_parts, rows, d, o,
                                                       dtype == FA_F32 ? 1 : 0, lse,
                                                       static_cast<cudaStream_t>(stream))));
}

__attribute__((visibility("default"))) size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    // the product B*H is formed only once it is known to fit (the same bounds the
    // backward itself enforces); sizes outside them have no workspace
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    if (!sizes_supported(B, H, N)) return 0;
    return bwd_workspace_bytes(B * H, N, d);
}

__attribute__((visibility("default"))) int fa_bwd_gqa(const void* q, const void* k,
                                                      const void* v, const void* o,
                                                      const float* lse, const void* dO, void* dq,
                                                      void* dk, void* dv, void* workspace,
                                                      size_t workspace_bytes, int B, int H,
                                                      int H_kv, int N, int d, float scale,
                                                      int causal, int dtype, void* stream) {
    int rc = check_common(q, k, v, o, lse, B, H, N);
    if (rc != FA_OK) return rc;
    if (lse == nullptr || dO == nullptr || dq == nullptr || dk == nullptr || dv == nullptr ||
        workspace == nullptr)
        return FA_ERR_INVALID_ARG;
    if (!aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(workspace))
        return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F32 && dtype != FA_BF16 && dtype != FA_E4M3) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 || (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
    if (workspace_bytes < bwd_workspace_bytes(B * H, N, d)) return FA_ERR_INVALID_ARG;
    int err = FA_OK;
    int* st = status_word(&err);
    if (st == nullptr) return err;
    DevCtl ctl{st, g_wait_ns.load()};
    return from_cuda(launch_bwd_sm103(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, H, H_kv, N, d,
                                      scale, causal ? 1 : 0, ctl, static_cast<cudaStream_t>(stream)));
}

__attribute__((visibility("default"))) int fa_bwd(const void* q, const void* k, const void* v,
                                                  const void* o, const float* lse, const void* dO,
                                                  void* dq, void* dk, void* dv, void* workspace,
                                                  size_t workspace_bytes, int B, int H, int N,
                                                  int d, float scale, int causal, int dtype,
                                                  void* stream) {
    return fa_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, H, H, N, d,
                      scale, causal, dtype, stream);
}

__attribute__((visibility("default"))) int fa_last_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    int err = FA_OK;
    if (status_word(&err) == nullptr) return err;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    return v;
}

// Launch a one-warp kernel whose only wait can never be satisfied; it must give
// up after the configured bound and record FA_ERR_DEVICE_TIMEOUT.  Exercises the
// device-side failure path without faulting or hanging the GPU.
__attribute__((visibility("default"))) int fa_selftest_wait_timeout(void* stream) {
    int err = FA_OK;
    int* st = status_word(&err);
    if (st == nullptr) return err;
    DevCtl ctl{st, g_wait_ns.load()};
    return from_cuda(static_cast<int>(launch_wait_selftest(ctl, static_cast<cudaStream_t>(stream))));
}

}  // extern "C"
