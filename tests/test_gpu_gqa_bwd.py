"""Grouped-query backward through the C ABI against the fp64 oracle: dQ per
query head, dK and dV summed over the query heads that share each K/V head."""
import numpy as np
import pytest
import torch

import exact_io_aware_06_gb300 as fa
import oracle
from exact_io_aware_06_gb300 import inputs
from gpu_util import TOL_BF16_GRAD, check_status, ensure_built, f64, max_err, scale_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def gqa_inputs(B, H, H_kv, N, d, seed=0):
    q = inputs.cast(inputs.normal((B, H, N, d), 42 + seed), "bf16")
    k = inputs.cast(inputs.normal((B, H_kv, N, d), 43 + seed), "bf16")
    v = inputs.cast(inputs.normal((B, H_kv, N, d), 44 + seed), "bf16")
    do = inputs.cast(inputs.normal((B, H, N, d), 45 + seed), "bf16")
    return q, k, v, do


def run(q, k, v, do, s, causal):
    q, k, v, do = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention_forward(q, k, v, s, causal)      # grouped forward
    B, H, N, d = q.shape
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd_gqa(q, k, v, o, lse, do, dq, dk, dv, ws, s, causal, fa.FA_BF16)
    check_status()
    return dq, dk, dv


@pytest.mark.parametrize("H,H_kv", [(8, 2), (4, 1), (3, 3)])
@pytest.mark.parametrize("N", [1, 130, 300])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_bwd_small(H, H_kv, N, d, causal):
    q, k, v, do = gqa_inputs(2, H, H_kv, N, d)
    s = scale_for(d)
    got = run(q, k, v, do, s, causal)
    ref = oracle.attn_bwd_gqa(f64(q), f64(k), f64(v), f64(do), s, causal)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert g.shape == r.shape
        # dK and dV are sums over the group: the bound scales with its size
        tol = TOL_BF16_GRAD * (1 if name == "dq" else max(1.0, (H // H_kv) ** 0.5))
        assert max_err(f64(g), r) <= tol, name


@pytest.mark.parametrize("d", [64, 128])
def test_gqa_bwd_b2_h16_hkv4_n2048_sampled_kv_heads(d):
    # a grouped backward at a production-like size; whole K/V heads (with their
    # four query heads) against the oracle
    B, H, H_kv, N = 2, 16, 4, 2048
    q, k, v, do = gqa_inputs(B, H, H_kv, N, d, seed=3)
    s = scale_for(d)
    dq, dk, dv = (f64(t) for t in run(q, k, v, do, s, False))
    for t in (dq, dk, dv):
        assert np.isfinite(t).all()
    g = H // H_kv
    for b, j in ((0, 0), (1, 3)):
        hs = slice(j * g, (j + 1) * g)
        rq, rk, rv = oracle.attn_bwd_gqa(f64(q[b:b + 1, hs]), f64(k[b:b + 1, j:j + 1]),
                                         f64(v[b:b + 1, j:j + 1]), f64(do[b:b + 1, hs]), s)
        assert max_err(dq[b:b + 1, hs], rq) <= TOL_BF16_GRAD
        assert max_err(dk[b:b + 1, j:j + 1], rk) <= 2 * TOL_BF16_GRAD
        assert max_err(dv[b:b + 1, j:j + 1], rv) <= 2 * TOL_BF16_GRAD
    # sum_j dV_j over a K/V head = sum over its group's query heads of sum_i dO_i
    want = f64(do).reshape(B, H_kv, g, N, d).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(2), want, atol=1.0)


def test_gqa_bwd_dq_equals_plain_backward_on_repeated_heads():
    # d = 128 computes dQ without atomics: per query head it is the same arithmetic
    # as the plain backward with the K/V heads repeated, so identical bits
    B, H, H_kv, N, d = 1, 8, 2, 700, 128
    q, k, v, do = gqa_inputs(B, H, H_kv, N, d, seed=7)
    s = scale_for(d)
    dq1, dk1, dv1 = run(q, k, v, do, s, True)
    kr = k.repeat_interleave(H // H_kv, dim=1).contiguous()
    vr = v.repeat_interleave(H // H_kv, dim=1).contiguous()
    dq2, dk2, dv2 = run(q, kr, vr, do, s, True)
    assert torch.equal(dq1, dq2)
    # the grouped dK/dV sum in fp32 on chip; the repeated-head ones are rounded to
    # bf16 before the sum: close, not equal
    g = H // H_kv
    dk2s = dk2.float().view(B, H_kv, g, N, d).sum(2)
    dv2s = dv2.float().view(B, H_kv, g, N, d).sum(2)
    assert max_err(f64(dk1), f64(dk2s)) <= 5e-2
    assert max_err(f64(dv1), f64(dv2s)) <= 5e-2
