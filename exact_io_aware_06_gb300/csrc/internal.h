// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

// Device-side error codes written into the per-device status word.
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 4;  // == FA_ERR_DEVICE_TIMEOUT

// A single wait that runs out after this long records kDevTimeout; draining a
// kernel's own in-flight copies / MMAs after that uses a fixed bound.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
constexpr uint64_t kDrainWaitNs = 1000000000ull;

// Sizes every entry point accepts: B*H heads and N rows each at most 2^24, and the
// kernels' work items -- (head, 128-row block) for the backward, (head, 256-row pair) for
// the forward -- countable in an int (B*H*ceil(N/128) <= 2^31 - 1).
inline bool sizes_supported(int B, int H, int N) {
    if (static_cast<int64_t>(B) * H > (1ll << 24) || N > (1 << 24)) return false;
    return static_cast<int64_t>(B) * H * ((static_cast<int64_t>(N) + 127) / 128) <= 0x7fffffffll;
}

struct DevCtl {
    int* status;       // per-device status word (first error wins)
    uint64_t wait_ns;  // bound on one wait
};

// Launch with programmatic stream serialization: the kernel may start while the
// previous kernel in the stream finishes (after a copy or an event it starts as
// usual).  Every kernel launched this way calls griddep_wait() (ptx.cuh) before it
// reads anything an earlier kernel may have written.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// fp32 exact forward on CUDA cores, d in {64, 128}.
cudaError_t launch_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                           int BH, int N, int d, float scale, int causal, cudaStream_t s);

// tcgen05 forward: bf16 (is_fp8 = false) or E4M3 inputs (is_fp8 = true, d = 128).
// K/V have B*H_kv heads (H_kv = H: plain attention; H_kv < H: grouped-query).
// qd/kd/vd: optional per-head FP8 descales on the device (null: use c_log2/o_scale only);
// with per_block = 1, one descale per 128-row block of each head ([head][ceil(N / 128)]).
// Returns 0 on success, or a CUDA / tensor-map error code (non-zero).
int launch_fwd_sm103(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int H_kv, int N, int d, float c_log2, float o_scale, const float* qd,
                     const float* kd, const float* vd, int per_block, int causal, bool is_fp8,
                     DevCtl ctl, cudaStream_t s);

// Forward over one shard of keys, bf16 inputs, d in {64, 128}: N_q queries against
// N_kv keys; when causal, key j reaches query i iff j <= i + delta (delta = the
// queries' global offset minus the keys').  O is written as float32 [B*H][N_q][d];
// rows that reach no key get O = 0 and lse = -inf.
int launch_fwd_kv_shard(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                        int H, int H_kv, int N_q, int N_kv, int d, float c_log2, int causal,
                        int delta, DevCtl ctl, cudaStream_t s);

// Merge of n_parts normalised partial outputs over disjoint key sets:
// lse = ln sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s.  o_parts float32
// [n_parts][rows][d], lse_parts [n_parts][rows], n_parts <= 16; o bf16 (o_f32 = 0) or float32
// [rows][d]; lse (optional) [rows].
cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int n_parts,
                             size_t rows, int d, void* o, int o_f32, float* lse, cudaStream_t s);

// Backward pieces.  Workspace layout (all float32, Np = N rounded up to 128):
//   [0, BH*Np)            -delta_i  (BH = B*H query heads) = -(dO_i . O_i)
//   [BH*Np, 2*BH*Np)      -lse_i * log2(e)   (both negated for packed FMA/FADD use)
//   [2*BH*Np, ...)        dQ accumulator [BH][Np][d] (d = 64 only; d = 128 computes dQ
//                         in a separate kernel without an accumulator)
size_t bwd_workspace_bytes(int BH, int N, int d);
// Q, O, dO, lse, dQ have B*H heads; K, V, dK, dV have B*H_kv heads (H_kv divides H;
// each K/V head's gradients sum over the H/H_kv query heads that share it).
int launch_bwd_sm103(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv, void* workspace, int B, int H,
                     int H_kv, int N, int d, float scale, int causal, DevCtl ctl, cudaStream_t s);

// dQ for d = 128 by a query-parallel kernel (recomputes S and dP per query block,
// accumulates dQ in TMEM, writes bf16 dQ = scale * dS K directly).  ws_nlse2 and
// ws_ndelta are the backward workspace's negated rows ([B*H][Np] each).
int launch_bwd_dq(const void* q, const void* k, const void* v, const void* dO,
                  const float* ws_nlse2, const float* ws_ndelta, void* dq, int B, int H, int H_kv,
                  int N, int d, float scale, int causal, DevCtl ctl, cudaStream_t s);

// A kernel that waits on a barrier nobody arrives at, with the bounded wait;
// it must record kDevTimeout and return.
cudaError_t launch_wait_selftest(DevCtl ctl, cudaStream_t s);

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace fa
