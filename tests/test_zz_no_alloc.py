"""fa_bwd_noalloc: the backward with the library's own fixed scratch array, for
callers that cannot allocate device memory when they call it (a plug-in whose
host framework owns the memory budget, a latency-critical path that cannot
take cudaMalloc's device synchronisation).  Its results must match the
workspace-taking fa_bwd on the same inputs, on two calls in a row (the second
call finds the first call's leftovers in the shared scratch).

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import pytest
import torch

import exact_io_aware_06_gb300 as fa
from gpu_util import TOL_BF16_GRAD, check_status, device_inputs, ensure_built, f64, max_err, scale_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def grads_with_workspace(dev, o, lse, scale):
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["do"]
    B, H, N, d = q.shape
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=q.device)
    out = [torch.empty_like(q) for _ in range(3)]
    fa.fa_bwd(q, k, v, o, lse, do, *out, ws, scale, False, fa.FA_BF16)
    check_status()
    return out


def grads_no_alloc(dev, o, lse, scale):
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["do"]
    out = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.fa_bwd_noalloc(q, k, v, o, lse, do, *out, scale, False, fa.FA_BF16)
    check_status()
    return out


@pytest.mark.parametrize("B,H,N", [(1, 2, 300), (4, 16, 2048)])
def test_no_alloc_matches_workspace_entry_twice(B, H, N):
    d = 64
    s = scale_for(d)
    x, dev = device_inputs(B, H, N, d, "bf16", with_do=True)
    o, lse = fa.attention_forward(dev["q"], dev["k"], dev["v"], s)
    ref = grads_with_workspace(dev, o, lse, s)
    for _ in range(2):
        got = grads_no_alloc(dev, o, lse, s)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert max_err(f64(g), f64(r)) <= TOL_BF16_GRAD, name
        # dK and dV do not depend on atomics: identical to the other entry point
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def test_no_alloc_refuses_sizes_beyond_its_scratch():
    # B*H*N rows whose workspace exceeds the 64 MiB array: refused before launch
    B, H, N, d = 8, 16, 4096, 64
    assert fa.fa_bwd_workspace_size(B, H, N, d) > 64 << 20
    P = 0x10000
    L = fa.lib()
    st = L.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, B, H, N, d, 0.125, 0, fa.FA_BF16, None)
    assert st == 2  # FA_ERR_UNSUPPORTED
