"""FP8 (E4M3) forward parity: the oracle runs on the dequantised inputs
(codes decoded by the oracle's own E4M3 decoder, times the descale)."""
import numpy as np
import pytest
import torch

import exact_io_aware_06_gb300 as fa
import oracle
from gpu_util import (head_rows, TOL_FP8_O, TOL_LSE_FP8, check_status, device_inputs, ensure_built, f64,
                      max_err, sample_rows, scale_for)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def dequant(x, name):
    return oracle.e4m3_decode(x[name].numpy(), x[name + "_descale"])


def run_fp8(x, dev, scale, causal):
    B, H, N, d = dev["q"].shape
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa.fa_fwd_fp8(dev["q"], dev["k"], dev["v"], o, lse, x["q_descale"], x["k_descale"],
                  x["v_descale"], scale, causal)
    check_status()
    return o, lse


@pytest.mark.parametrize("N", [1, 100, 128, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_small(N, causal):
    x, dev = device_inputs(1, 2, N, 128, "e4m3")
    s = scale_for(128)
    o, lse = run_fp8(x, dev, s, causal)
    o_ref, lse_ref = oracle.attn_fwd(dequant(x, "q"), dequant(x, "k"), dequant(x, "v"), s, causal)
    assert max_err(f64(o), o_ref) <= TOL_FP8_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_FP8


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_config_b4_h16_n4096_d128_every_head(causal):
    # the FP8 workload at full size (and its causal form); rows are independent in the
    # forward, so the tile-edge and random rows of every head are checked exactly
    B, H, N, d = 4, 16, 4096, 128
    x, dev = device_inputs(B, H, N, d, "e4m3")
    s = scale_for(d)
    o, lse = run_fp8(x, dev, s, causal)
    o_c, lse_c = f64(o), f64(lse)
    assert np.isfinite(o_c).all()
    for b in range(B):
        for h in range(H):
            rows = head_rows(N, b * H + h)
            qh = oracle.e4m3_decode(x["q"][b, h].numpy(), x["q_descale"])
            kh = oracle.e4m3_decode(x["k"][b, h].numpy(), x["k_descale"])
            vh = oracle.e4m3_decode(x["v"][b, h].numpy(), x["v_descale"])
            o_ref, lse_ref = oracle.attn_fwd_rows(qh, kh, vh, rows, s, causal)
            assert max_err(o_c[b, h, rows], o_ref) <= TOL_FP8_O, f"b{b} h{h}"
            assert max_err(lse_c[b, h, rows], lse_ref) <= TOL_LSE_FP8, f"b{b} h{h}"
    if causal:
        # row 0 sees only key 0: O_0 = V_0 up to the bf16 output rounding
        v0 = oracle.e4m3_decode(x["v"][:, :, 0].numpy(), x["v_descale"])
        assert max_err(o_c[:, :, 0], v0) <= 2 ** -8 * np.abs(v0).max() + 1e-6
