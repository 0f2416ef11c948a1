"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws numbers and casts
them.  The workloads on the pages are random N(0,1) matrices (the
"Flash Attention V1/V2/V3" page's demo seeds numpy with 42; the
"FlashAttention-1" page draws ``torch.randn``), so every tensor here is iid
N(0,1) from a CPU ``torch.Generator`` with a fixed seed, then cast:

* ``f32``  -- kept as float32;
* ``bf16`` -- rounded to bfloat16 (round to nearest even, torch's cast);
* ``e4m3`` -- per-tensor FP8: ``descale = amax(|x|) / 448`` (448 is the largest
  finite E4M3 value; descale 1 if amax is 0) and
  ``codes = e4m3(clamp(x / descale, -448, 448))`` with torch's
  ``float8_e4m3fn`` cast.

Default seeds: Q 42, K 43, V 44, dO 45.
"""
import torch

SEED_Q, SEED_K, SEED_V, SEED_DO = 42, 43, 44, 45
E4M3_MAX = 448.0


def normal(shape, seed):
    """iid N(0,1) float32 CPU tensor from a generator seeded with ``seed``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32)


def cast(x, dtype):
    if dtype == "f32":
        return x.to(torch.float32).contiguous()
    if dtype == "bf16":
        return x.to(torch.bfloat16).contiguous()
    raise ValueError(f"unknown dtype {dtype!r}")


def quantize_e4m3(x):
    """Per-tensor amax quantisation. Returns (uint8 codes tensor, float descale)."""
    amax = float(x.abs().max()) if x.numel() else 0.0
    descale = amax / E4M3_MAX if amax > 0 else 1.0
    descale = float(torch.tensor(descale, dtype=torch.float32))  # an fp32 scale factor
    y = (x / descale).clamp(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return codes, descale


def quantize_e4m3_per_head(x):
    """Per-(batch, head) amax quantisation of a [B, H, N, d] tensor.
    Returns (uint8 codes, float32 descales of shape [B, H])."""
    B, H = x.shape[0], x.shape[1]
    codes = torch.empty(x.shape, dtype=torch.uint8)
    descale = torch.empty((B, H), dtype=torch.float32)
    for b in range(B):
        for h in range(H):
            codes[b, h], descale[b, h] = quantize_e4m3(x[b, h])
    return codes, descale


def quantize_e4m3_per_block(x, block=128):
    """Per-(batch, head, 128-row block) amax quantisation of a [B, H, N, d] tensor.
    Returns (uint8 codes, float32 descales of shape [B, H, ceil(N / block)])."""
    B, H, N = x.shape[0], x.shape[1], x.shape[2]
    nb = (N + block - 1) // block
    codes = torch.empty(x.shape, dtype=torch.uint8)
    descale = torch.empty((B, H, nb), dtype=torch.float32)
    for b in range(B):
        for h in range(H):
            for j in range(nb):
                rows = slice(j * block, min(N, (j + 1) * block))
                codes[b, h, rows], descale[b, h, j] = quantize_e4m3(x[b, h, rows])
    return codes, descale


def attention_inputs(B, H, N, d, dtype="bf16", with_do=False,
                     seeds=(SEED_Q, SEED_K, SEED_V, SEED_DO)):
    """CPU tensors [B, H, N, d] for q, k, v (and do).  For ``e4m3`` the dict
    holds uint8 codes plus ``q_descale``/``k_descale``/``v_descale``."""
    shape = (B, H, N, d)
    raw = {n: normal(shape, s) for n, s in zip(("q", "k", "v"), seeds[:3])}
    if with_do:
        raw["do"] = normal(shape, seeds[3])
    out = {}
    if dtype == "e4m3":
        for n in ("q", "k", "v"):
            out[n], out[n + "_descale"] = quantize_e4m3(raw[n])
        if with_do:
            out["do"] = cast(raw["do"], "bf16")
        return out
    for n, x in raw.items():
        out[n] = cast(x, dtype)
    return out
