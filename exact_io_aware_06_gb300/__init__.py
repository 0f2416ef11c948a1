"""Exact IO-aware attention on GB300 (sm_103a): a thin ctypes binding over libfa.so.

Every entry point has the name and argument order of the C function declared
in ``include/fa.h``; this module only turns torch tensors into device pointers
and sizes, passes the current CUDA stream and raises ``FaError`` on a non-zero
status.  All arithmetic happens in the library's CUDA kernels.  PyTorch serves
as the allocator and stream provider only.

There is no fallback: if ``libfa.so`` has not been built, or no GPU is present,
the calls raise.
"""
import ctypes
import math
import os

__all__ = [
    "FaError", "FA_F32", "FA_BF16", "FA_E4M3", "lib", "fa_fwd", "fa_fwd_fp8", "fa_fwd_gqa",
    "fa_fwd_fp8_per_head", "fa_fwd_fp8_per_block", "fa_bwd",
    "fa_bwd_workspace_size", "fa_bwd_noalloc", "fa_last_device_error", "fa_set_wait_timeout_ns",
    "fa_selftest_wait_timeout", "fa_status_string", "attention_forward", "attention_backward",
]

FA_F32, FA_BF16, FA_E4M3 = 0, 1, 2
FA_OK = 0
FA_ERR_DEVICE_TIMEOUT = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libfa.so")
_LIB = None


class FaError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        super().__init__(f"{what}: {fa_status_string(self.status)} ({self.status})")


def lib():
    """Load libfa.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        L.fa_fwd.restype = i
        L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, f, f, f, i, i, i, i, f, i, vp]
        L.fa_fwd_fp8.restype = i
        L.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
        L.fa_fwd_gqa.restype = i
        L.fa_fwd_fp8_per_head.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_fwd_fp8_per_head.restype = i
        L.fa_fwd_fp8_per_block.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_fwd_fp8_per_block.restype = i
        ll = ctypes.c_longlong
        L.fa_fwd_kv_shard.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, ll, ll, i, vp]
        L.fa_fwd_kv_shard.restype = i
        L.fa_lse_merge.argtypes = [vp, vp, i, vp, vp, i, i, i, i, i, vp]
        L.fa_lse_merge.restype = i
        L.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        L.fa_bwd_workspace_size.restype = sz
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, i, vp]
        L.fa_bwd_gqa.restype = i
        L.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, i,
                                 vp]
        L.fa_bwd.restype = i
        L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        L.fa_bwd_noalloc.restype = i
        L.fa_last_device_error.argtypes = [vp]
        L.fa_last_device_error.restype = i
        L.fa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        L.fa_set_wait_timeout_ns.restype = None
        L.fa_selftest_wait_timeout.argtypes = [vp]
        L.fa_selftest_wait_timeout.restype = i
        L.fa_status_string.argtypes = [i]
        L.fa_status_string.restype = ctypes.c_char_p
        _LIB = L
    return _LIB


def fa_status_string(status):
    try:
        return lib().fa_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _shape(q):
    if q.dim() != 4 or not q.is_contiguous():
        raise ValueError("tensors must be contiguous [B, H, N, d]")
    return tuple(int(x) for x in q.shape)


def _check(status, what):
    if status != FA_OK:
        raise FaError(status, what)


def fa_fwd(q, k, v, o, lse, scale, causal, dtype, stream=None):
    """O (and lse, may be None) <- attention(q, k, v); tensors [B, H, N, d] on the GPU."""
    B, H, N, d = _shape(q)
    _check(lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                        int(bool(causal)), int(dtype), _stream(stream)), "fa_fwd")


def fa_fwd_fp8(q8, k8, v8, o, lse, q_descale, k_descale, v_descale, scale, causal, stream=None):
    """FP8 forward: q8/k8/v8 uint8 E4M3 codes [B, H, N, d]; o bfloat16."""
    B, H, N, d = _shape(q8)
    _check(lib().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(o), _ptr(lse), float(q_descale),
                            float(k_descale), float(v_descale), B, H, N, d, float(scale),
                            int(bool(causal)), _stream(stream)), "fa_fwd_fp8")


def fa_fwd_gqa(q, k, v, o, lse, scale, causal, dtype, stream=None):
    """Grouped-query forward: q, o [B, H, N, d]; k, v [B, H_kv, N, d] with H % H_kv == 0."""
    B, H, N, d = _shape(q)
    H_kv = _shape(k)[1]
    _check(lib().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, N, d,
                            float(scale), int(bool(causal)), int(dtype), _stream(stream)),
           "fa_fwd_gqa")


def fa_fwd_fp8_per_head(q8, k8, v8, o, lse, q_descale, k_descale, v_descale, scale, causal,
                        stream=None):
    """FP8 forward with per-(b, h) descales: float32 device tensors of B*H elements."""
    B, H, N, d = _shape(q8)
    for t in (q_descale, k_descale, v_descale):
        if t.numel() != B * H or t.dtype.itemsize != 4 or not t.is_contiguous():
            raise ValueError("per-head descales: contiguous float32, B*H elements")
    _check(lib().fa_fwd_fp8_per_head(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(o), _ptr(lse),
                                     _ptr(q_descale), _ptr(k_descale), _ptr(v_descale), B, H, N,
                                     d, float(scale), int(bool(causal)), _stream(stream)),
           "fa_fwd_fp8_per_head")


def fa_fwd_fp8_per_block(q8, k8, v8, o, lse, q_descale, k_descale, v_descale, scale, causal,
                         stream=None):
    """FP8 forward with one descale per 128-row block of each head: float32 device
    tensors of B*H*ceil(N/128) elements ([B][H][ceil(N/128)])."""
    B, H, N, d = _shape(q8)
    nb = (N + 127) // 128
    for t in (q_descale, k_descale, v_descale):
        if t.numel() != B * H * nb or t.dtype.itemsize != 4 or not t.is_contiguous():
            raise ValueError("per-block descales: contiguous float32, B*H*ceil(N/128) elements")
    _check(lib().fa_fwd_fp8_per_block(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(o), _ptr(lse),
                                      _ptr(q_descale), _ptr(k_descale), _ptr(v_descale), B, H, N,
                                      d, float(scale), int(bool(causal)), _stream(stream)),
           "fa_fwd_fp8_per_block")


def fa_fwd_kv_shard(q, k, v, o_part, lse_part, scale, causal, q_offset, kv_offset,
                    dtype=FA_BF16, stream=None):
    """Forward of q [B, H, N_q, d] over one key shard k, v [B, H_kv, N_kv, d] at the
    given global offsets; o_part float32 [B, H, N_q, d], lse_part [B, H, N_q]."""
    B, H, N_q, d = _shape(q)
    H_kv, N_kv = _shape(k)[1], _shape(k)[2]
    _check(lib().fa_fwd_kv_shard(_ptr(q), _ptr(k), _ptr(v), _ptr(o_part), _ptr(lse_part), B, H,
                                 H_kv, N_q, N_kv, d, float(scale), int(bool(causal)),
                                 int(q_offset), int(kv_offset), int(dtype), _stream(stream)),
           "fa_fwd_kv_shard")


def fa_lse_merge(o_parts, lse_parts, o, lse, dtype, stream=None):
    """Merge stacked shard outputs o_parts [S, B, H, N, d] (float32), lse_parts
    [S, B, H, N] into o [B, H, N, d] (bf16 or float32 per dtype) and lse (or None)."""
    S, B, H, N, d = (int(x) for x in o_parts.shape)
    if tuple(lse_parts.shape) != (S, B, H, N) or tuple(o.shape) != (B, H, N, d):
        raise ValueError("fa_lse_merge: shapes do not match")
    _check(lib().fa_lse_merge(_ptr(o_parts), _ptr(lse_parts), S, _ptr(o), _ptr(lse), B, H, N, d,
                              int(dtype), _stream(stream)), "fa_lse_merge")


def fa_bwd_workspace_size(B, H, N, d):
    return int(lib().fa_bwd_workspace_size(int(B), int(H), int(N), int(d)))


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, workspace, scale, causal, dtype, stream=None):
    """dq, dk, dv <- backward; workspace: a device buffer of fa_bwd_workspace_size bytes."""
    B, H, N, d = _shape(q)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                        _ptr(dk), _ptr(dv), _ptr(workspace), nbytes, B, H, N, d, float(scale),
                        int(bool(causal)), int(dtype), _stream(stream)), "fa_bwd")


def fa_bwd_gqa(q, k, v, o, lse, do, dq, dk, dv, workspace, scale, causal, dtype, stream=None):
    """Grouped-query backward: q, o, do, dq [B, H, N, d]; k, v, dk, dv [B, H_kv, N, d]."""
    B, H, N, d = _shape(q)
    H_kv = _shape(k)[1]
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                            _ptr(dk), _ptr(dv), _ptr(workspace), nbytes, B, H, H_kv, N, d,
                            float(scale), int(bool(causal)), int(dtype), _stream(stream)),
           "fa_bwd_gqa")


def fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale, causal, dtype, stream=None):
    """fa_bwd with the library's built-in scratch (no workspace, no allocation).
    For callers that cannot allocate device memory at call time; calls that
    overlap on the GPU race on the shared scratch."""
    B, H, N, d = _shape(q)
    _check(lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                int(bool(causal)), int(dtype), _stream(stream)), "fa_bwd_noalloc")


def fa_last_device_error(stream=None):
    """Synchronise the stream and return (and clear) the device status word."""
    return int(lib().fa_last_device_error(_stream(stream)))


def fa_set_wait_timeout_ns(ns):
    lib().fa_set_wait_timeout_ns(int(ns))


def fa_selftest_wait_timeout(stream=None):
    _check(lib().fa_selftest_wait_timeout(_stream(stream)), "fa_selftest_wait_timeout")


# ---------------------------------------------------------------- conveniences
def attention_forward(q, k, v, scale=None, causal=False, stream=None):
    """Allocate O and lse with torch and run fa_fwd; q, k, v fp32 or bf16."""
    import torch
    dtype = {torch.float32: FA_F32, torch.bfloat16: FA_BF16}[q.dtype]
    B, H, N, d = _shape(q)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    # k, v with fewer heads than q: grouped-query attention
    fn = fa_fwd if _shape(k)[1] == H else fa_fwd_gqa
    fn(q, k, v, o, lse, 1.0 / math.sqrt(d) if scale is None else scale, causal, dtype, stream)
    return o, lse


def attention_backward(q, k, v, o, lse, do, scale=None, causal=False, stream=None):
    import torch
    B, H, N, d = _shape(q)
    ws = torch.empty(fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    # k, v with fewer heads than q: grouped-query attention
    fn = fa_bwd if _shape(k)[1] == H else fa_bwd_gqa
    fn(q, k, v, o, lse, do, dq, dk, dv, ws, 1.0 / math.sqrt(d) if scale is None else scale,
       causal, FA_BF16, stream)
    return dq, dk, dv
