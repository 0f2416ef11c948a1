// bwd_noalloc.cu -- fa_bwd_noalloc: the backward pass with its scratch memory
// held inside the library instead of passed in by the caller.
//
// Some callers cannot allocate device memory at the moment they need the
// backward: a plug-in invoked from a host framework that owns the whole device
// memory budget and forbids allocations inside its execution hook, or code on a
// latency-critical path where cudaMalloc's implicit device synchronisation is
// not acceptable.  This entry point serves them: the caller still passes every
// input and output buffer, but the delta / lse / dQ-accumulator scratch lives in
// a fixed, file-scope __device__ array (kNoAllocScratchBytes), which every GPU
// that loads the library holds until the process exits.
//
// The array's name in host code is only a host-side stand-in for the symbol,
// not a device address; the device address comes from cudaGetSymbolAddress,
// looked up once per device (with that device current) on the first call made
// on that device.
#include <mutex>

#include "../../include/fa.h"
#include "internal.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB per device

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of this device's scratch array; nullptr on failure.
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace fa

extern "C" __attribute__((visibility("default"))) int fa_bwd_noalloc(
    const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
    void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int dtype,
    void* stream) {
    using namespace fa;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    // B*H is formed only within the bounds fa_bwd enforces, so it cannot overflow
    if (!sizes_supported(B, H, N)) return FA_ERR_UNSUPPORTED;
    // the sizes this scratch array cannot hold are refused before anything runs
    if (bwd_workspace_bytes(B * H, N, d) > kNoAllocScratchBytes) return FA_ERR_UNSUPPORTED;
    void* scratch = scratch_address();
    if (scratch == nullptr) return FA_ERR_CUDA;
    // Every region of the scratch that the kernels read is written earlier in the
    // same call (delta and lse rows, and the zeroed dQ accumulator), so the previous
    // call's contents never leak into this one.
    return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, N, d,
                  scale, causal, dtype, stream);
}
