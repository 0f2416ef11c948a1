"""fa_bwd_noalloc: the backward with the library's own fixed scratch array, for
callers that cannot allocate device memory when they call it (a plug-in whose
host framework owns the memory budget, a latency-critical path that cannot
take cudaMalloc's device synchronisation).

Its results must match the workspace-taking fa_bwd on the same inputs, call
after call.  The calls run back to back on the one shared scratch array, and
each changes something the previous call left behind: other inputs (seeds), a
smaller and ragged N after a full-size one (so stale delta / lse rows and dQ
partials from the previous call would sit exactly where this call reads), the
d = 128 path (whose scratch holds no dQ accumulator and whose separate dQ kernel
reads the delta and lse rows) and the causal schedule.  The small cases are also
checked against the fp64 oracle.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import pytest
import torch

import exact_io_aware_06_gb300 as fa
import oracle
from gpu_util import TOL_BF16_GRAD, check_status, device_inputs, ensure_built, f64, max_err, scale_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def grads_with_workspace(dev, o, lse, scale, causal):
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["do"]
    B, H, N, d = q.shape
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=q.device)
    out = [torch.empty_like(q) for _ in range(3)]
    fa.fa_bwd(q, k, v, o, lse, do, *out, ws, scale, causal, fa.FA_BF16)
    check_status()
    return out


def grads_no_alloc(dev, o, lse, scale, causal):
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["do"]
    out = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.fa_bwd_noalloc(q, k, v, o, lse, do, *out, scale, causal, fa.FA_BF16)
    check_status()
    return out


# (B, H, N, d, causal, first seed) in call order; each case is called twice in a row
# with different inputs, so every call follows one whose scratch contents differ.
SEQUENCE = [
    (4, 16, 2048, 64, False, 42),   # the full backward configuration (34.6 MB of scratch)
    (1, 2, 300, 64, True, 142),     # ragged and causal, after a larger call
    (1, 3, 520, 128, False, 242),   # d = 128: no accumulator; the dQ kernel reads the rows
    (1, 2, 390, 128, True, 342),
    (2, 3, 1000, 64, False, 442),   # d = 64 again after d = 128
]


def test_no_alloc_matches_workspace_entry_call_after_call():
    for B, H, N, d, causal, seed0 in SEQUENCE:
        s = scale_for(d)
        for call in range(2):
            seed = seed0 + 10 * call
            x, dev = device_inputs(B, H, N, d, "bf16", with_do=True,
                                   seeds=(seed, seed + 1, seed + 2, seed + 3))
            o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], s, causal=causal)
            got = grads_no_alloc(dev, o, lse, s, causal)
            ref = grads_with_workspace(dev, o, lse, s, causal)
            what = f"B{B} H{H} N{N} d{d} causal={causal} call {call}"
            for name, g, r in zip(("dq", "dk", "dv"), got, ref):
                assert max_err(f64(g), f64(r)) <= TOL_BF16_GRAD, f"{name}: {what}"
            # dK and dV use no atomics (nor, at d = 128, does dQ): identical results
            assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2]), what
            if d == 128:
                assert torch.equal(got[0], ref[0]), what
            if B * H * N <= 6 * 1000:
                g_ref = oracle.attn_bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), s,
                                        causal=causal)
                for name, g, r in zip(("dq", "dk", "dv"), got, g_ref):
                    assert max_err(f64(g), r) <= TOL_BF16_GRAD, f"{name} vs oracle: {what}"


def test_no_alloc_refuses_sizes_beyond_its_scratch():
    # B*H*N rows whose workspace exceeds the 64 MiB array: refused before launch
    B, H, N, d = 8, 16, 4096, 64
    assert fa.fa_bwd_workspace_size(B, H, N, d) > 64 << 20
    P = 0x10000
    L = fa.lib()
    st = L.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, B, H, N, d, 0.125, 0, fa.FA_BF16, None)
    assert st == 2  # FA_ERR_UNSUPPORTED
    # B*H beyond the backward's bound is refused without forming an overflowing product
    st = L.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, 1 << 16, 1 << 16, 128, d, 0.125, 0,
                          fa.FA_BF16, None)
    assert st == 2
