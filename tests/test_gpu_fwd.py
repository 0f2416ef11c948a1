"""Forward parity through the C ABI against the fp64 oracle: the exact fp32
kernel and the tcgen05 bf16 kernel, small ragged shapes element by element and
the full-size workloads on sampled rows."""
import numpy as np
import pytest
import torch

import exact_io_aware_06_gb300 as fa
import oracle
from gpu_util import (head_rows, TOL_BF16_O, TOL_F32_O, TOL_LSE_BF16, TOL_LSE_F32, check_status,
                      device_inputs, ensure_built, f64, max_err, sample_rows, scale_for)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def run_fwd(dev, dtype_code, scale, causal):
    q = dev["q"]
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    fa.fa_fwd(q, dev["k"], dev["v"], o, lse, scale, causal, dtype_code)
    check_status()
    return o, lse


# ---------------------------------------------------------------- fp32 (exact) kernel
def test_f32_worked_config_n128_d64():
    # single head, N=128, d=64, the pages' fp32 check (block 32 x 32)
    x, dev = device_inputs(1, 1, 128, 64, "f32")
    s = scale_for(64)
    o, lse = run_fwd(dev, fa.FA_F32, s, False)
    o_ref, lse_ref = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s)
    assert max_err(f64(o), o_ref) <= TOL_F32_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_F32


@pytest.mark.parametrize("N", [1, 17, 33, 130, 257])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_f32_ragged(N, d, causal):
    x, dev = device_inputs(2, 1, N, d, "f32")
    s = scale_for(d)
    o, lse = run_fwd(dev, fa.FA_F32, s, causal)
    o_ref, lse_ref = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s, causal)
    assert max_err(f64(o), o_ref) <= TOL_F32_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_F32


# ---------------------------------------------------------------- bf16 tcgen05 kernel
@pytest.mark.parametrize("N", [1, 17, 128, 130, 255, 256, 300, 513])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_small(N, d, causal):
    x, dev = device_inputs(1, 3, N, d, "bf16")
    s = scale_for(d)
    o, lse = run_fwd(dev, fa.FA_BF16, s, causal)
    o_ref, lse_ref = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s, causal)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_BF16


def test_bf16_large_scores_trigger_rescale():
    # scores grow along the sequence so the running max keeps moving: exercises
    # the lazy O rescale path many times
    B, H, N, d = 1, 2, 1024, 64
    x, dev = device_inputs(B, H, N, d, "bf16")
    ramp = torch.linspace(0.2, 4.0, N).view(1, 1, N, 1)
    k = (x["k"].float() * ramp).to(torch.bfloat16)
    q = (x["q"].float() * 3).to(torch.bfloat16)
    dev = {"q": q.cuda(), "k": k.cuda(), "v": dev["v"]}
    s = scale_for(d)
    for causal in (False, True):
        o, lse = run_fwd(dev, fa.FA_BF16, s, causal)
        o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(x["v"]), s, causal)
        assert max_err(f64(o), o_ref) <= TOL_BF16_O
        assert max_err(f64(lse), lse_ref) <= 5 * TOL_LSE_BF16


def test_bf16_config_b4_h16_n1024_d64_full():
    # the whole forward workload compared element by element
    B, H, N, d = 4, 16, 1024, 64
    x, dev = device_inputs(B, H, N, d, "bf16")
    s = scale_for(d)
    o, lse = run_fwd(dev, fa.FA_BF16, s, False)
    o_ref, lse_ref = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_BF16


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_config_b1_h32_n16384_d128_sampled(causal):
    # the long-sequence workload at full size; rows are independent in the
    # forward, so sampled rows are checked exactly against the oracle
    B, H, N, d = 1, 32, 16384, 128
    x, dev = device_inputs(B, H, N, d, "bf16")
    s = scale_for(d)
    o, lse = run_fwd(dev, fa.FA_BF16, s, causal)
    o_c, lse_c = f64(o), f64(lse)
    assert np.isfinite(o_c).all()
    # every head: the tile edges (first and last rows of the first, middle and last
    # query tiles and tile pairs) and a few random rows
    for h in range(H):
        rows = head_rows(N, h)
        o_ref, lse_ref = oracle.attn_fwd_rows(f64(x["q"][0, h]), f64(x["k"][0, h]),
                                              f64(x["v"][0, h]), rows, s, causal)
        assert max_err(o_c[0, h, rows], o_ref) <= TOL_BF16_O, f"head {h}"
        assert max_err(lse_c[0, h, rows], lse_ref) <= TOL_LSE_BF16, f"head {h}"
    if causal:
        # row 0 sees only key 0
        assert max_err(o_c[0, :, 0], f64(x["v"][0, :, 0])) <= 1e-2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_many_heads_ragged_n_every_head(d, causal):
    # Many more (head, query-tile pair) items than SMs, each with a ragged last tile
    # (N = 1000: four pairs, the last one 232 rows): every CTA of the forward works
    # through several items, carrying its TMEM, barriers and K/V ring from one to the
    # next, and items of different lengths (causal) follow each other.  Every head's
    # tile edges and random rows against the oracle.
    B, H, N = 2, 96, 1000
    x, dev = device_inputs(B, H, N, d, "bf16")
    s = scale_for(d)
    o, lse = run_fwd(dev, fa.FA_BF16, s, causal)
    o_c, lse_c = f64(o), f64(lse)
    for b in range(B):
        for h in range(H):
            rows = head_rows(N, b * H + h, n_random=2)
            o_ref, lse_ref = oracle.attn_fwd_rows(f64(x["q"][b, h]), f64(x["k"][b, h]),
                                                  f64(x["v"][b, h]), rows, s, causal)
            assert max_err(o_c[b, h, rows], o_ref) <= TOL_BF16_O, f"batch {b} head {h}"
            assert max_err(lse_c[b, h, rows], lse_ref) <= TOL_LSE_BF16, f"batch {b} head {h}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_single_tile_items_between_pairs(d, causal):
    # N = 300: each head has one whole tile pair and a last pair whose second tile lies
    # past N, which runs as a single-tile item (its key blocks alternate between the two
    # softmax warpgroups, whose halves are merged at the end).  400 items on the persistent
    # CTAs, so each CTA works through pairs and single tiles in turn, and the two tiles'
    # per-block barrier counts drift apart.  Whole tensors against the oracle.
    B, H, N = 2, 100, 300
    x, dev = device_inputs(B, H, N, d, "bf16")
    s = scale_for(d)
    o, lse = run_fwd(dev, fa.FA_BF16, s, causal)
    o_ref, lse_ref = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s, causal)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_BF16


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_last_round_as_single_tiles(d, causal):
    # 40 heads x 4 pairs = 160 pairs: one full round on 152 CTAs; without the causal mask the
    # 8 pairs left for the second round are dealt as 16 single tiles (causal runs keep the
    # pairs there).  Whole tensors against the oracle.
    B, H, N = 1, 40, 1024
    x, dev = device_inputs(B, H, N, d, "bf16")
    s = scale_for(d)
    o, lse = run_fwd(dev, fa.FA_BF16, s, causal)
    o_ref, lse_ref = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s, causal)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_BF16


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_fewer_pairs_than_sms_run_as_single_tiles(d, causal):
    # 4 heads x 16 pairs = 64 pairs, fewer than half the SMs: every pair is dealt as two
    # single-tile items, and each warpgroup sweeps 16 of the 32 key blocks.  Whole tensors
    # against the oracle.
    B, H, N = 1, 4, 4096
    x, dev = device_inputs(B, H, N, d, "bf16")
    s = scale_for(d)
    o, lse = run_fwd(dev, fa.FA_BF16, s, causal)
    o_ref, lse_ref = oracle.attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), s, causal)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_BF16


def test_bf16_deterministic_and_lse_optional():
    x, dev = device_inputs(1, 2, 700, 128, "bf16")
    s = scale_for(128)
    o1, l1 = run_fwd(dev, fa.FA_BF16, s, True)
    o2, l2 = run_fwd(dev, fa.FA_BF16, s, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3 = torch.empty_like(o1)
    fa.fa_fwd(dev["q"], dev["k"], dev["v"], o3, None, s, True, fa.FA_BF16)
    check_status()
    assert torch.equal(o1, o3)


# ---------------------------------------------------------------- back-to-back launches
@pytest.mark.parametrize("d", [64, 128])
def test_chained_forwards_ping_pong_without_host_sync(d):
    # Kernels here may start while the one before them in the stream finishes (their
    # set-up overlaps its tail), and must not read its output or overwrite what it reads
    # until it has completed.  Stage t reads buffer A as Q and writes B; stage t + 1 reads
    # B and writes A, which stage t was reading: both orders are exercised, on one stream,
    # with no host synchronisation in between.  The oracle runs the same chain on its own
    # outputs, rounded to bf16 between stages as the kernel's outputs are.
    from exact_io_aware_06_gb300 import inputs
    B, H, N = 2, 3, 300
    s = scale_for(d)
    q0 = inputs.cast(inputs.normal((B, H, N, d), 80), "bf16")
    k = inputs.cast(inputs.normal((B, H, N, d), 81), "bf16")
    v = inputs.cast(inputs.normal((B, H, N, d), 82), "bf16")
    kd, vd = k.cuda(), v.cuda()
    bufs = [q0.cuda(), torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")]
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    stages = [False, True, False, True]  # causal flags
    for t, causal in enumerate(stages):
        fa.fa_fwd(bufs[t % 2], kd, vd, bufs[(t + 1) % 2], lse, s, causal, fa.FA_BF16)
    check_status()
    got = f64(bufs[len(stages) % 2])
    ref = q0
    for causal in stages:
        o_ref, _ = oracle.attn_fwd(f64(ref), f64(k), f64(v), s, causal)
        ref = torch.from_numpy(o_ref).to(torch.bfloat16)
    assert max_err(got, f64(ref)) <= TOL_BF16_O
