"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/fa.h declares, and rejects bad arguments on the host before touching
the device.  CPU only: no kernel is launched here."""
import ctypes
import os
import re

import pytest

import exact_io_aware_06_gb300 as fa
from exact_io_aware_06_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(fa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return fa.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_fwd", "fa_fwd_fp8", "fa_bwd", "fa_bwd_workspace_size",
                     "fa_last_device_error", "fa_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_only_declared_symbols_are_exported(L):
    # hidden visibility: nothing but the C ABI leaks out of the library
    out = os.popen(f"nm -D --defined-only {fa.LIB_PATH}").read()
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert {n for n in exported if n.startswith("fa_")} == set(declared_functions())


def test_status_strings(L):
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(1) == "FA_ERR_INVALID_ARG"
    assert fa.fa_status_string(2) == "FA_ERR_UNSUPPORTED"
    assert fa.fa_status_string(3) == "FA_ERR_CUDA"
    assert fa.fa_status_string(4) == "FA_ERR_DEVICE_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


def test_workspace_size(L):
    # delta + lse2 ([BH][Np]) and the fp32 dQ accumulator ([BH][Np][d]), Np = ceil128(N)
    B, H, N, d = 4, 16, 2048, 64
    assert fa.fa_bwd_workspace_size(B, H, N, d) == (2 * B * H * N + B * H * N * d) * 4
    # d = 128 computes dQ without an accumulator: only the two row vectors
    assert fa.fa_bwd_workspace_size(B, H, N, 128) == 2 * B * H * N * 4
    Np = 256
    assert fa.fa_bwd_workspace_size(1, 3, 130, 64) == (2 * 3 * Np + 3 * Np * 64) * 4
    assert fa.fa_bwd_workspace_size(0, 1, 1, 64) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 0, 64) == 0


P = ctypes.c_void_p(0x10000)        # aligned, never dereferenced: rejected first
MIS = ctypes.c_void_p(0x10008)      # misaligned


def fwd(L, q=P, o=P, B=1, H=1, N=128, d=64, dtype=1, lse=None, scale=0.125):
    return L.fa_fwd(q, P, P, o, lse, B, H, N, d, scale, 0, dtype, None)


def test_fwd_argument_errors(L):
    assert fwd(L, q=None) == 1
    assert fwd(L, o=None) == 1
    assert fwd(L, q=MIS) == 1
    assert fwd(L, lse=MIS) == 1
    assert fwd(L, N=0) == 1
    assert fwd(L, B=0) == 1
    assert fwd(L, H=-1) == 1
    assert fwd(L, dtype=2) == 1          # E4M3 goes through fa_fwd_fp8
    assert fwd(L, dtype=7) == 1
    assert fwd(L, scale=float("nan")) == 1
    assert fwd(L, d=96) == 2
    assert fwd(L, d=256) == 2


def test_size_limits(L):
    # B*H and N each at most 2^24, and B*H*ceil(N/128) work items at most 2^31 - 1
    assert fwd(L, B=1 << 12, H=1 << 13) == 2            # B*H = 2^25
    assert fwd(L, N=(1 << 24) + 1) == 2
    assert fwd(L, B=1 << 12, H=1 << 12, N=1 << 24) == 2  # 2^24 heads x 2^17 blocks
    assert fwd(L, B=1 << 8, H=1 << 8, N=1 << 22) == 2    # exactly 2^31 blocks
    # the workspace query applies the same limits, at the boundary on both sides
    assert fa.fa_bwd_workspace_size(1 << 8, 1 << 8, 1 << 22, 128) == 0
    ok = fa.fa_bwd_workspace_size(1 << 8, 1 << 8, (1 << 22) - 128, 128)
    assert ok == 2 * (1 << 16) * ((1 << 22) - 128) * 4
    assert fa.fa_bwd_workspace_size(1, 1, (1 << 24) + 1, 64) == 0
    # the allocation-free backward refuses them before looking at its scratch
    assert L.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, 1 << 8, 1 << 8, 1 << 22, 64, 0.125, 0,
                            1, None) == 2


def test_fp8_argument_errors(L):
    def f(qd=1.0, d=128, N=128, scale=0.1):
        return L.fa_fwd_fp8(P, P, P, P, None, qd, 1.0, 1.0, 1, 1, N, d, scale, 0, None)
    assert f(qd=0.0) == 1
    assert f(qd=-1.0) == 1
    assert f(qd=float("inf")) == 1
    assert f(qd=float("nan")) == 1
    assert f(N=0) == 1
    assert f(scale=float("nan")) == 1
    assert f(d=64) == 2


def test_gqa_forward_argument_errors(L):
    def g(H=4, H_kv=2, d=64, dtype=1, scale=0.125):
        return L.fa_fwd_gqa(P, P, P, P, None, 1, H, H_kv, 128, d, scale, 0, dtype, None)
    assert g(H_kv=0) == 1
    assert g(H_kv=3) == 1                # 4 % 3 != 0
    assert g(scale=float("inf")) == 1
    assert g(dtype=2) == 1               # E4M3 goes through the fp8 entry points
    assert g(dtype=0) == 2               # fp32 inputs: not on this path
    assert g(d=96) == 2


@pytest.mark.parametrize("name", ["fa_fwd_fp8_per_head", "fa_fwd_fp8_per_block"])
def test_fp8_descale_array_argument_errors(L, name):
    fn = getattr(L, name)

    def f(qd=P, kd=P, vd=P, d=128, N=128, scale=0.1):
        return fn(P, P, P, P, None, qd, kd, vd, 1, 1, N, d, scale, 0, None)
    assert f(qd=None) == 1
    assert f(kd=None) == 1
    assert f(vd=None) == 1
    assert f(N=0) == 1
    assert f(scale=float("nan")) == 1
    assert f(d=64) == 2


def test_bwd_argument_errors(L):
    ws = fa.fa_bwd_workspace_size(1, 1, 128, 64)

    def b(dtype=1, d=64, causal=0, ws_bytes=ws, dq=P, lse=P):
        return L.fa_bwd(P, P, P, P, lse, P, dq, P, P, P, ws_bytes, 1, 1, 128, d, 0.125, causal,
                        dtype, None)
    assert b(dq=None) == 1
    assert b(lse=None) == 1
    assert b(ws_bytes=ws - 4) == 1
    assert b(dtype=9) == 1
    assert b(dtype=0) == 2
    assert b(dtype=2) == 2               # no E4M3 backward
    assert b(d=96) == 2


def test_bwd_gqa_argument_errors(L):
    ws = fa.fa_bwd_workspace_size(1, 4, 128, 64)

    def b(H=4, H_kv=2, d=64, ws_bytes=ws):
        return L.fa_bwd_gqa(P, P, P, P, P, P, P, P, P, P, ws_bytes, 1, H, H_kv, 128, d, 0.125, 0,
                            1, None)
    assert b(H_kv=0) == 1
    assert b(H_kv=3) == 1                # 4 % 3 != 0
    assert b(ws_bytes=ws - 4) == 1
    assert b(d=96) == 2


def test_kv_shard_argument_errors(L):
    def f(lse=P, Nkv=128, H_kv=1, d=64, dtype=1):
        return L.fa_fwd_kv_shard(P, P, P, P, lse, 1, 2, H_kv, 128, Nkv, d, 0.125, 1, 0, 0, dtype,
                                 None)
    assert f(lse=None) == 1            # the merge needs lse
    assert f(Nkv=0) == 1
    assert f(H_kv=3) == 1
    assert f(dtype=0) == 2             # fp32 inputs: not on this path
    assert f(d=96) == 2
    assert f(Nkv=(1 << 24) + 1) == 2   # keys per shard beyond 2^24


def test_lse_merge_argument_errors(L):
    def m(op=P, lp=P, o=P, S=2, d=64, dtype=1, lse=None, B=1, H=1, N=128):
        return L.fa_lse_merge(op, lp, S, o, lse, B, H, N, d, dtype, None)
    assert m(op=None) == 1
    assert m(lp=MIS) == 1
    assert m(lse=MIS) == 1
    assert m(S=0) == 1
    assert m(N=0) == 1
    assert m(dtype=2) == 1
    assert m(d=32) == 2
    assert m(S=17) == 2                # at most 16 parts
    # B*H*N rows times parts beyond 2^40 elements are refused, not wrapped
    assert m(B=1 << 10, H=1 << 10, N=1 << 21) == 2
    assert m(S=17) == 2
