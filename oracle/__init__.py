"""fp64 CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference leg may import this package.  The product library
(``exact_io_aware_06_gb300``) never imports, links or runs it, and the two
share no code.

Functions (numpy in, numpy out; every array is promoted to float64):

* ``attn_fwd(q, k, v, scale, causal)`` -- standard attention written out
  (S = scale QK^T, stable row softmax, O = PV, lse = m + ln l), following the
  "FlashAttention-1" page, 10.2.1, and the Python demo's ``softmax_attention``
  on the "Flash Attention V1/V2/V3" page.
* ``attn_fwd_rows(q, k, v, rows, scale, causal)`` -- the same for selected
  rows of one head (rows are independent in the forward).
* ``attn_fwd_tiled(q, k, v, Br, Bc, scale, causal)`` -- online softmax over
  blocks ("Flash Attention V1/V2/V3" page, Python demo; "5.4 FlashAttention"
  page, listing 3-1), used only for block-size invariance checks.
* ``attn_bwd(q, k, v, do, scale, causal)`` -- analytic backward
  ("FlashAttention-1" page, 10.2.4): dV = P^T dO, dP = dO V^T,
  dS = P o (dP - delta), delta_i = dO_i . O_i, dQ = scale dS K,
  dK = scale dS^T Q.
* ``attn_fwd_gqa`` / ``attn_bwd_gqa`` -- grouped-query attention ("5.4
  FlashAttention" page, GQA heading): each K/V head repeated for its group of
  query heads; dK, dV summed over the group (chain rule through the shared
  operand).
* ``attn_fwd_kv_shard(q, k, v, scale, causal, q_offset, kv_offset)`` -- the
  forward restricted to one shard of keys (numpy), rows with no key: O = 0,
  lse = -inf; ``lse_merge(o_parts, lse_parts)`` -- the two-state combination
  of "FlashAttention-1" 10.2.2 applied to normalised partial outputs.
* ``e4m3_decode(codes, descale)`` / ``e4m3_encode(x)`` -- OCP FP8 E4M3.
* ``e4m3_decode_blocks(codes, descales, block)`` -- E4M3 with one dequantisation
  factor per block of rows (the finer scale factors of the "Flash Attention
  V1/V2/V3" page, V3 section); the attention of the decoded values is
  ``attn_fwd``.

Tensors are ``[..., N, d]``; leading dimensions are flattened into heads.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def lib():
    """The oracle library.  ORACLE_LIB names another build of oracle.c to load
    instead (the mutation test uses it to run the pins against planted bugs)."""
    global _LIB
    if _LIB is None:
        path = os.environ.get("ORACLE_LIB") or _build.LIB
        if path == _build.LIB and (not os.path.exists(path) or not _build.up_to_date()):
            _build.build()
        L = ctypes.CDLL(path)
        L.oracle_fwd.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                 ctypes.c_double, ctypes.c_int, _dp, _dp, ctypes.c_int]
        L.oracle_fwd_rows.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                      ctypes.c_double, ctypes.c_int, _lp, ctypes.c_long, _dp, _dp,
                                      ctypes.c_int]
        L.oracle_fwd_tiled.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                       ctypes.c_double, ctypes.c_int, ctypes.c_long,
                                       ctypes.c_long, _dp, _dp]
        L.oracle_bwd.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                 ctypes.c_double, ctypes.c_int, _dp, _dp, _dp, ctypes.c_int]
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_f64.restype = ctypes.c_double
        L.oracle_f64_to_e4m3.argtypes = [ctypes.c_double]
        L.oracle_f64_to_e4m3.restype = ctypes.c_uint8
        L.oracle_e4m3_decode.argtypes = [_u8p, ctypes.c_long, ctypes.c_double, _dp]
        L.oracle_e4m3_encode.argtypes = [_dp, ctypes.c_long, _u8p]
        L.oracle_max_threads.restype = ctypes.c_int
        _LIB = L
    return _LIB


def max_threads():
    return int(lib().oracle_max_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, t=_dp):
    return a.ctypes.data_as(t)


def _heads(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.shape != k.shape or q.shape != v.shape or q.ndim < 2:
        raise ValueError("q, k, v must share one shape [..., N, d]")
    N, d = q.shape[-2], q.shape[-1]
    BH = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    return q, k, v, BH, N, d


def attn_fwd(q, k, v, scale, causal=False, nthreads=0):
    """Return (O, lse): O has q's shape, lse has q.shape[:-1]."""
    q, k, v, BH, N, d = _heads(q, k, v)
    o = np.empty_like(q)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    lib().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(scale), int(bool(causal)),
                     _ptr(o), _ptr(lse), int(nthreads))
    return o, lse


def attn_fwd_rows(q, k, v, rows, scale, causal=False, nthreads=0):
    """One head ([N, d] each); rows: query indices.  Returns (O[rows], lse[rows])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 2:
        raise ValueError("attn_fwd_rows takes one head: [N, d]")
    N, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).astype(np.int_)
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise ValueError("row index out of range")
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    lib().oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), N, d, float(scale), int(bool(causal)),
                          _ptr(rows, _lp), rows.size, _ptr(o), _ptr(lse), int(nthreads))
    return o, lse


def attn_fwd_tiled(q, k, v, Br, Bc, scale, causal=False):
    q, k, v, BH, N, d = _heads(q, k, v)
    if Br < 1 or Bc < 1:
        raise ValueError("block sizes must be >= 1")
    o = np.empty_like(q)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    lib().oracle_fwd_tiled(_ptr(q), _ptr(k), _ptr(v), BH, N, d, float(scale),
                           int(bool(causal)), int(Br), int(Bc), _ptr(o), _ptr(lse))
    return o, lse


def attn_bwd(q, k, v, do, scale, causal=False, nthreads=0):
    """Return (dQ, dK, dV) of L = <dO, O(q, k, v)>."""
    q, k, v, BH, N, d = _heads(q, k, v)
    do = _f64(do)
    if do.shape != q.shape:
        raise ValueError("dO must have q's shape")
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    lib().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), BH, N, d, float(scale),
                     int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv), int(nthreads))
    return dq, dk, dv


def _group(q, k, v):
    """[B, H, N, d] queries against [B, H_kv, N, d] keys/values: the group size."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.shape != v.shape or k.ndim != 4 or q.shape[0] != k.shape[0] \
            or q.shape[2:] != k.shape[2:] or k.shape[1] < 1 or q.shape[1] % k.shape[1]:
        raise ValueError("grouped-query: q [B, H, N, d], k and v [B, H_kv, N, d], H_kv | H")
    return q, k, v, q.shape[1] // k.shape[1]


def attn_fwd_gqa(q, k, v, scale, causal=False, nthreads=0):
    """Grouped-query forward ("5.4 FlashAttention" page, the GQA heading): query
    head h reads K/V head h // (H / H_kv).  Each K/V head is repeated for its group
    and the plain forward runs per query head."""
    q, k, v, g = _group(q, k, v)
    return attn_fwd(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), scale, causal, nthreads)


def attn_bwd_gqa(q, k, v, do, scale, causal=False, nthreads=0):
    """Gradients of L = <dO, O> for grouped-query attention.  K/V head j enters
    the forward of every query head of its group, so by the chain rule its dK, dV
    are the sums of the per-query-head gradients ("FlashAttention-1" page, 10.2.4,
    per head) over the group; dQ is per query head."""
    q, k, v, g = _group(q, k, v)
    dq, dk, dv = attn_bwd(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), do, scale, causal,
                          nthreads)
    B, H_kv, N, d = k.shape
    return (dq, dk.reshape(B, H_kv, g, N, d).sum(axis=2),
            dv.reshape(B, H_kv, g, N, d).sum(axis=2))


def attn_fwd_kv_shard(q, k, v, scale, causal=False, q_offset=0, kv_offset=0):
    """Attention of queries at global positions q_offset + i against one shard of
    keys at global positions kv_offset + j ([..., N_q, d] against [..., N_kv, d]).

    Standard attention written out ("FlashAttention-1" page, 10.2.1) on the keys
    the shard holds: S = scale Q K^T, causal mask kv_offset + j > q_offset + i,
    stable softmax, O = P V, lse = m + ln l.  A row that sees no key of the shard
    has l = 0: it returns O = 0 and lse = -inf, so that it drops out of the merge.
    Returns (O [..., N_q, d], lse [..., N_q])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if k.shape != v.shape or q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1]:
        raise ValueError("q [..., N_q, d]; k and v [..., N_kv, d] with the same leading dims")
    S = scale * np.matmul(q, np.swapaxes(k, -1, -2))
    Nq, Nkv = q.shape[-2], k.shape[-2]
    if causal:
        masked = (kv_offset + np.arange(Nkv))[None, :] > (q_offset + np.arange(Nq))[:, None]
        S = np.where(masked, -np.inf, S)
    m = S.max(axis=-1, initial=-np.inf)
    seen = np.isfinite(m)
    P = np.exp(S - np.where(seen, m, 0.0)[..., None])
    l = P.sum(axis=-1)
    o = np.matmul(P, v) / np.where(seen, l, 1.0)[..., None]
    lse = np.where(seen, m + np.log(np.where(seen, l, 1.0)), -np.inf)
    return o, lse


def lse_merge(o_parts, lse_parts):
    """Merge attention outputs computed over disjoint key sets ("FlashAttention-1"
    page, 10.2.2: two partial softmax states combine through their maxima and
    sums).  With each part normalised, part s carries l_s = exp(lse_s) of the
    total, so lse = ln sum_s exp(lse_s) and O = sum_s exp(lse_s - lse) O_s.
    o_parts [S, ..., d], lse_parts [S, ...].  Parts with lse = -inf contribute
    nothing; if every part is -inf the row is O = 0, lse = -inf."""
    o, L = _f64(o_parts), _f64(lse_parts)
    m = L.max(axis=0)
    seen = np.isfinite(m)
    mm = np.where(seen, m, 0.0)
    w = np.exp(L - mm[None])
    tot = w.sum(axis=0)
    lse = np.where(seen, mm + np.log(np.where(seen, tot, 1.0)), -np.inf)
    out = (w[..., None] * o).sum(axis=0) / np.where(seen, tot, 1.0)[..., None]
    return out, lse


def e4m3_decode(codes, descale=1.0):
    """uint8 E4M3 codes -> float64 values times descale."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_decode(_ptr(c, _u8p), c.size, float(descale), _ptr(out))
    return out


def e4m3_decode_blocks(codes, descales, block=128):
    """uint8 E4M3 codes [..., N, d] -> float64 values in which row i carries the
    factor descales[..., i // block] (one per block of rows; the last block may be
    short).  descales has shape [..., ceil(N / block)]."""
    x = e4m3_decode(codes)
    f = np.asarray(descales, dtype=np.float64)
    N = x.shape[-2]
    if f.shape != x.shape[:-2] + (-(-N // block),):
        raise ValueError("descales: [..., ceil(N / block)] for codes [..., N, d]")
    return x * f[..., np.arange(N) // block][..., None]


def e4m3_encode(x):
    """float64 values -> uint8 E4M3 codes (round to nearest even, saturate at 448)."""
    x = _f64(x)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode(_ptr(x), x.size, _ptr(out, _u8p))
    return out
