"""Device-side failure detection without a GPU fault: a kernel whose wait can
never be satisfied gives up after the bound and reports FA_ERR_DEVICE_TIMEOUT,
and the context stays usable afterwards."""
import time

import pytest
import torch

import exact_io_aware_06_gb300 as fa
from gpu_util import TOL_BF16_O, check_status, device_inputs, ensure_built, f64, max_err, scale_for
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_bounded_wait_reports_timeout_and_context_survives():
    assert fa.fa_last_device_error() == 0
    fa.fa_set_wait_timeout_ns(2_000_000)  # 2 ms
    try:
        t0 = time.time()
        fa.fa_selftest_wait_timeout()
        st = fa.fa_last_device_error()
        elapsed = time.time() - t0
    finally:
        fa.fa_set_wait_timeout_ns(0)
    assert st == fa.FA_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0
    assert fa.fa_last_device_error() == 0  # cleared by the read
    # the context still works: a normal forward afterwards is correct
    x, dev = device_inputs(1, 1, 256, 64, "bf16")
    s = scale_for(64)
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], s)
    check_status()
    o_ref, _ = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O


# ---------------------------------------------------------------- production kernels
def _fwd(B, H, N, d, causal):
    x, dev = device_inputs(B, H, N, d, "bf16")
    s = scale_for(d)
    return lambda: fa.attention_forward(dev["q"], dev["k"], dev["v"], s, causal)


def _fwd_fp8(B, H, N, causal):
    x, dev = device_inputs(B, H, N, 128, "e4m3")
    o = torch.empty((B, H, N, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    return lambda: fa.fa_fwd_fp8(dev["q"], dev["k"], dev["v"], o, lse, x["q_descale"],
                                 x["k_descale"], x["v_descale"], scale_for(128), causal)


def _bwd(B, H, N, d, causal):
    x, dev = device_inputs(B, H, N, d, "bf16", with_do=True)
    s = scale_for(d)
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], s, causal)
    check_status()
    return lambda: fa.attention_backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, causal)


ABORT_CASES = {
    "forward bf16 d128": lambda: _fwd(1, 16, 4096, 128, False),
    "forward bf16 d64 causal": lambda: _fwd(4, 16, 2048, 64, True),
    "forward e4m3": lambda: _fwd_fp8(2, 16, 4096, False),
    "backward d64 (delta, main, convert)": lambda: _bwd(4, 16, 2048, 64, False),
    "backward d64 causal": lambda: _bwd(4, 16, 2048, 64, True),
    "backward d128 (dK/dV kernel, dQ kernel)": lambda: _bwd(1, 8, 4096, 128, True),
}


def test_production_kernels_abort_on_a_short_wait_limit():
    # With a wait limit far below the time the kernels' loads and MMAs take, their waits
    # run out: the kernel records FA_ERR_DEVICE_TIMEOUT, every role drains its own
    # in-flight copies and MMAs, TMEM is freed and the kernel returns.  Each call must
    # come back well within a second with FA_OK (nothing ran out) or the timeout status;
    # then, with the default limit restored, the same context computes correct results.
    runs = {name: make() for name, make in ABORT_CASES.items()}
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    seen = {}
    try:
        for limit_ns in (1, 300):
            fa.fa_set_wait_timeout_ns(limit_ns)
            for name, run in runs.items():
                for _ in range(2):
                    t0 = time.time()
                    run()
                    st = fa.fa_last_device_error()
                    elapsed = time.time() - t0
                    assert st in (fa.FA_OK, fa.FA_ERR_DEVICE_TIMEOUT), (name, st)
                    assert elapsed < 5.0, (name, elapsed)
                    seen.setdefault(name, []).append(st)
    finally:
        fa.fa_set_wait_timeout_ns(0)
    print({name: sts.count(fa.FA_ERR_DEVICE_TIMEOUT) for name, sts in seen.items()})
    # the abort path was taken (some wait ran out in most launches this size)
    assert sum(sts.count(fa.FA_ERR_DEVICE_TIMEOUT) for sts in seen.values()) > 0, seen
    assert fa.fa_last_device_error() == 0
    # the context still works: a normal forward and backward are correct
    x, dev = device_inputs(1, 2, 300, 64, "bf16", with_do=True)
    s = scale_for(64)
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], s, True)
    dq, dk, dv = fa.attention_backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], s, True)
    check_status()
    o_ref, _ = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s, True)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O
    g_ref = oracle.attn_bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), s, True)
    for g, r in zip((dq, dk, dv), g_ref):
        assert max_err(f64(g), r) <= 5e-2
