"""Shared helpers for the GPU parity tests: build once, move seeded inputs to
the device, and promote anything to float64 numpy for the oracle."""
import math

import numpy as np
import torch

import exact_io_aware_06_gb300 as fa
from exact_io_aware_06_gb300 import inputs

# tolerances (max abs error against the fp64 oracle)
TOL_F32_O = 1e-5
TOL_BF16_O = 2e-2
TOL_BF16_GRAD = 5e-2
TOL_FP8_O = 1e-1
TOL_LSE_F32 = 1e-5
TOL_LSE_BF16 = 1e-3
TOL_LSE_FP8 = 1e-2


_BUILT = False


def ensure_built():
    global _BUILT
    if not _BUILT:
        import __graft_entry__
        __graft_entry__.build()
        _BUILT = True
    if not torch.cuda.is_available():
        raise RuntimeError("these tests need a CUDA GPU")


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def max_err(a, b):
    return float(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)).max())


def scale_for(d):
    return 1.0 / math.sqrt(d)


def device_inputs(B, H, N, d, dtype, with_do=False, seeds=None):
    kw = {} if seeds is None else {"seeds": seeds}
    x = inputs.attention_inputs(B, H, N, d, dtype, with_do=with_do, **kw)
    dev = {n: (t.cuda() if torch.is_tensor(t) else t) for n, t in x.items()}
    return x, dev


def check_status():
    st = fa.fa_last_device_error()
    assert st == 0, f"device status {fa.fa_status_string(st)}"


def sample_rows(N, n_random=48, seed=0):
    """First/last rows, tile edges, and a few random rows."""
    edges = {0, 1, N - 1, N - 2}
    for t in (127, 128, 255, 256, 4095, 4096, 8191, 8192):
        if t < N:
            edges.add(t)
    rng = np.random.default_rng(seed)
    rnd = set(rng.integers(0, N, size=min(n_random, N)).tolist())
    return sorted(r for r in edges | rnd if 0 <= r < N)


def head_rows(N, seed, n_random=4):
    """Rows to check in every head of a large forward: the first and last row of the
    first, middle and last 128-row query tiles (so both tiles of a CTA's pair and the
    ragged end), plus a few random rows."""
    last = (N - 1) // 128
    mid = last // 2
    edges = {0, 127, 128 * mid, 128 * mid + 127, 128 * last, N - 1}
    rng = np.random.default_rng(1000 + seed)
    rnd = set(rng.integers(0, N, size=min(n_random, N)).tolist())
    return sorted(r for r in edges | rnd if 0 <= r < N)
