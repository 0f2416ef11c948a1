"""Sequence sharding through the C ABI: the forward over one key shard
(fa_fwd_kv_shard) against the oracle's shard forward, the lse merge
(fa_lse_merge) against the oracle's merge, and shards + merge against the
oracle's forward over the whole sequence."""
import numpy as np
import pytest
import torch

import exact_io_aware_06_gb300 as fa
import oracle
from exact_io_aware_06_gb300 import inputs
from gpu_util import (TOL_BF16_O, TOL_LSE_BF16, check_status, ensure_built, f64, max_err,
                      sample_rows, scale_for)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def bf16(shape, seed):
    return inputs.cast(inputs.normal(shape, seed), "bf16")


def shard_fwd(q, k, v, s, causal, q_off, kv_off):
    B, H, Nq, d = q.shape
    o = torch.empty((B, H, Nq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    fa.fa_fwd_kv_shard(q, k, v, o, lse, s, causal, q_off, kv_off)
    check_status()
    return o, lse


def check_rows(o, lse, o_ref, lse_ref):
    """Rows that saw no key must be exactly O = 0, lse = -inf; the rest within the
    bf16 tolerances."""
    o, lse = f64(o), f64(lse)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(o[empty] == 0)
    if (~empty).any():
        assert max_err(o[~empty], o_ref[~empty]) <= TOL_BF16_O
        assert max_err(lse[~empty], lse_ref[~empty]) <= TOL_LSE_BF16


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nkv,q_off,kv_off", [
    (130, 300, 0, 0),          # more keys than queries
    (300, 77, 500, 200),       # keys wholly before the queries: all visible under causal
    (257, 200, 100, 150),      # partial overlap: rows < 50 see nothing under causal
    (128, 128, 0, 4096),       # keys wholly after the queries: causal rows see nothing
    (1, 1, 0, 0),
])
@pytest.mark.parametrize("causal", [False, True])
def test_kv_shard_forward(d, Nq, Nkv, q_off, kv_off, causal):
    B, H = 2, 3
    q, k, v = bf16((B, H, Nq, d), 42), bf16((B, H, Nkv, d), 43), bf16((B, H, Nkv, d), 44)
    s = scale_for(d)
    o, lse = shard_fwd(q.cuda(), k.cuda(), v.cuda(), s, causal, q_off, kv_off)
    o_ref, lse_ref = oracle.attn_fwd_kv_shard(f64(q), f64(k), f64(v), s, causal, q_off, kv_off)
    check_rows(o, lse, o_ref, lse_ref)


def test_kv_shard_grouped_query():
    # 8 query heads on 2 K/V heads, causal shard with an offset
    B, H, H_kv, Nq, Nkv, d = 1, 8, 2, 260, 390, 128
    q, k, v = bf16((B, H, Nq, d), 50), bf16((B, H_kv, Nkv, d), 51), bf16((B, H_kv, Nkv, d), 52)
    s = scale_for(d)
    o, lse = shard_fwd(q.cuda(), k.cuda(), v.cuda(), s, True, 300, 100)
    rep = H // H_kv
    o_ref, lse_ref = oracle.attn_fwd_kv_shard(f64(q), np.repeat(f64(k), rep, axis=1),
                                              np.repeat(f64(v), rep, axis=1), s, True, 300, 100)
    check_rows(o, lse, o_ref, lse_ref)


def random_parts(S, B, H, N, d, seed, with_empty=True):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn((S, B, H, N, d), generator=g)
    lse = torch.randn((S, B, H, N), generator=g) * 4.0
    if with_empty:
        # some parts saw nothing for some rows; row 3 saw nothing anywhere
        lse[0, :, :, ::5] = -float("inf")
        o[0, :, :, ::5] = 0.0
        lse[:, :, :, 3] = -float("inf")
        o[:, :, :, 3] = 0.0
    return o, lse


@pytest.mark.parametrize("S", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_lse_merge_against_oracle(S, d, out):
    B, H, N = 2, 3, 257
    o_p, lse_p = random_parts(S, B, H, N, d, seed=S * 10 + d)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    o = torch.empty((B, H, N, d), dtype=dt, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa.fa_lse_merge(o_p.cuda(), lse_p.cuda(), o, lse, fa.FA_F32 if out == "f32" else fa.FA_BF16)
    check_status()
    o_ref, lse_ref = oracle.lse_merge(f64(o_p), f64(lse_p))
    got_o, got_l = f64(o), f64(lse)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(got_l), empty) and np.all(got_o[empty] == 0)
    # fp32 arithmetic: a few ulp of |O| <= ~5 (f32), or the bf16 output rounding
    tol = 1e-5 if out == "f32" else 2.0 ** -8 * max(1.0, float(np.abs(o_ref).max()))
    assert max_err(got_o, o_ref) <= tol
    assert max_err(got_l[~empty], lse_ref[~empty]) <= 1e-5


def run_sharded(q, k, v, s, causal, cuts, out=fa.FA_BF16):
    """Every query against key shards [cuts[i], cuts[i+1]); merged."""
    B, H, N, d = q.shape
    parts = [shard_fwd(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous(), s, causal, 0, a)
             for a, b in zip(cuts[:-1], cuts[1:])]
    o_p = torch.stack([p[0] for p in parts]).contiguous()
    lse_p = torch.stack([p[1] for p in parts]).contiguous()
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16 if out == fa.FA_BF16 else torch.float32,
                    device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa.fa_lse_merge(o_p, lse_p, o, lse, out)
    check_status()
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cuts", [(0, 128, 700), (0, 300, 301, 555, 700), (0, 700)])
def test_key_shards_merge_to_full_forward(d, causal, cuts):
    B, H, N = 1, 2, 700
    q, k, v = bf16((B, H, N, d), 60), bf16((B, H, N, d), 61), bf16((B, H, N, d), 62)
    s = scale_for(d)
    o, lse = run_sharded(q.cuda(), k.cuda(), v.cuda(), s, causal, list(cuts))
    o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), s, causal)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_BF16


def test_ring_style_query_and_key_shards_causal():
    # four ranks' worth of work on one GPU: rank r holds rows [r*n, (r+1)*n) of Q, K, V;
    # its output merges its queries against key shards 0..r (later shards are masked)
    B, H, N, d, R = 1, 4, 1024, 128, 4
    n = N // R
    q, k, v = bf16((B, H, N, d), 70), bf16((B, H, N, d), 71), bf16((B, H, N, d), 72)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    s = scale_for(d)
    o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), s, True)
    for r in range(R):
        qr = qd[:, :, r * n:(r + 1) * n].contiguous()
        parts = [shard_fwd(qr, kd[:, :, t * n:(t + 1) * n].contiguous(),
                           vd[:, :, t * n:(t + 1) * n].contiguous(), s, True, r * n, t * n)
                 for t in range(r + 1)]
        o_p = torch.stack([p[0] for p in parts]).contiguous()
        lse_p = torch.stack([p[1] for p in parts]).contiguous()
        o = torch.empty((B, H, n, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, H, n), dtype=torch.float32, device="cuda")
        fa.fa_lse_merge(o_p, lse_p, o, lse, fa.FA_BF16)
        check_status()
        assert max_err(f64(o), o_ref[:, :, r * n:(r + 1) * n]) <= TOL_BF16_O
        assert max_err(f64(lse), lse_ref[:, :, r * n:(r + 1) * n]) <= TOL_LSE_BF16


def test_sharded_b1_h32_n16384_d128_causal_sampled_rows():
    # the long-sequence forward split into 4 key shards of 4096; rows are independent,
    # so sampled rows are checked against the oracle over the whole sequence
    B, H, N, d = 1, 32, 16384, 128
    x = inputs.attention_inputs(B, H, N, d, "bf16")
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    s = scale_for(d)
    o, lse = run_sharded(q, k, v, s, True, [0, 4096, 8192, 12288, 16384])
    o, lse = f64(o), f64(lse)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = sample_rows(N, n_random=24)
    for h in (0, 31):
        o_ref, lse_ref = oracle.attn_fwd_rows(f64(x["q"][0, h]), f64(x["k"][0, h]),
                                              f64(x["v"][0, h]), rows, s, True)
        assert max_err(o[0, h, rows], o_ref) <= TOL_BF16_O
        assert max_err(lse[0, h, rows], lse_ref) <= TOL_LSE_BF16


@pytest.mark.parametrize("causal", [False, True])
def test_key_shards_on_side_streams_merge_to_full_forward(causal):
    # The shards are independent: launched on four streams side by side (as they would run
    # on four GPUs) after the launch stream's work, then merged on the launch stream once
    # all four have finished.  The result is the forward over the whole sequence.
    B, H, N, d, S = 1, 4, 2048, 128, 4
    n = N // S
    q, k, v = (bf16((B, H, N, d), 42 + i).cuda() for i in range(3))
    s = scale_for(d)
    ks = [k[:, :, t * n:(t + 1) * n].contiguous() for t in range(S)]
    vs = [v[:, :, t * n:(t + 1) * n].contiguous() for t in range(S)]
    o_p = torch.empty((S, B, H, N, d), dtype=torch.float32, device="cuda")
    l_p = torch.empty((S, B, H, N), dtype=torch.float32, device="cuda")
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    main = torch.cuda.current_stream()
    side = [torch.cuda.Stream() for _ in range(S)]
    start, done = torch.cuda.Event(), [torch.cuda.Event() for _ in range(S)]
    start.record(main)
    for t in range(S):
        side[t].wait_event(start)
        fa.fa_fwd_kv_shard(q, ks[t], vs[t], o_p[t], l_p[t], s, causal, 0, t * n, fa.FA_BF16, side[t])
        done[t].record(side[t])
    for t in range(S):
        main.wait_event(done[t])
    fa.fa_lse_merge(o_p, l_p, o, lse, fa.FA_BF16, main)
    check_status()
    o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), s, causal)
    assert max_err(f64(o), o_ref) <= TOL_BF16_O
    assert max_err(f64(lse), lse_ref) <= TOL_LSE_BF16
