"""FP8 (E4M3) forward parity: the oracle runs on the dequantised inputs
(codes decoded by the oracle's own E4M3 decoder, times the descale)."""
import numpy as np
import pytest
import torch

import exact_io_aware_06_gb300 as fa
import oracle
from gpu_util import (TOL_FP8_O, TOL_LSE_FP8, check_status, device_inputs, ensure_built, f64,
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


def test_fp8_config_b4_h16_n4096_d128_sampled():
    B, H, N, d = 4, 16, 4096, 128
    x, dev = device_inputs(B, H, N, d, "e4m3")
    s = scale_for(d)
    o, lse = run_fp8(x, dev, s, False)
    o_c, lse_c = f64(o), f64(lse)
    assert np.isfinite(o_c).all()
    errs = []
    for b, h in ((0, 0), (1, 7), (3, 15)):
        rows = sample_rows(N, 24, seed=b * 16 + h)
        qh = oracle.e4m3_decode(x["q"][b, h].numpy(), x["q_descale"])
        kh = oracle.e4m3_decode(x["k"][b, h].numpy(), x["k_descale"])
        vh = oracle.e4m3_decode(x["v"][b, h].numpy(), x["v_descale"])
        o_ref, lse_ref = oracle.attn_fwd_rows(qh, kh, vh, rows, s)
        errs.append(max_err(o_c[b, h, rows], o_ref))
        assert max_err(lse_c[b, h, rows], lse_ref) <= TOL_LSE_FP8
    assert max(errs) <= TOL_FP8_O
