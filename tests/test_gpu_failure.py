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
