"""Throughput of the exact-attention hot path on GB300 (TFLOP/s and % of peak).

One step runs every stage of the path once, each on its own synthetic batch
(iid N(0,1) inputs, seeds 42-45, scale 1/sqrt(d)):

  fwd   bf16  B=1  H=32 N=16384 d=128  non-causal   (long-sequence forward)
  fwd   bf16  B=1  H=32 N=16384 d=128  causal
  fwd   bf16  B=4  H=16 N=1024  d=64   non-causal
  fwd+bwd bf16 B=4 H=16 N=2048  d=64   non-causal   (forward, then delta / dK dV dQ / dQ convert)
  fwd   e4m3  B=4  H=16 N=4096  d=128  non-causal   (per-tensor descales, bf16 O)

FLOP counts: forward 4 B H N^2 d, backward 10 B H N^2 d, halved when causal.
``value`` is the step's total FLOP over its device time (CUDA events on the
launch stream, inputs resident in HBM); ``parts`` gives each stage alone.
``e2e`` times the same step through the public API with pinned host buffers:
inputs copied in and outputs copied out inside the timed region, each part's copies
on their own streams so that they overlap the other parts' compute.

``extras`` times the variant rows alone, after the step and outside ``value``
(the median of 20 launches each, after 3 warm-ups): backward at d=128 and causal, FP8 causal
and per-head and per-128-row-block scale factors, grouped-query forward/backward (32 query heads on 8 K/V heads),
and the forward sharded over 4 key blocks of the sequence (the shards on 4 streams side
by side, as they would run on 4 GPUs) plus the lse merge (with the merge kernel's achieved
HBM bandwidth).

``--impl reference`` times the fp64 CPU oracle instead (the comparison arm) on a
bounded sample of the same workload, on this machine's host cores.

Multi-GPU: the stages shard by head with no exchange, so N ranks run N
independent replicas (weak scaling); rank 0 prints the line.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd/bwd attention TFLOP/s on 1 GB300 and % of dense tensor-core peak"
UNIT = "TFLOP/s"

PARTS = [
    # name, kind, dtype, B, H, N, d, causal
    ("fwd_bf16_b1h32n16384d128", "fwd", "bf16", 1, 32, 16384, 128, False),
    ("fwd_bf16_b1h32n16384d128_causal", "fwd", "bf16", 1, 32, 16384, 128, True),
    ("fwd_bf16_b4h16n1024d64", "fwd", "bf16", 4, 16, 1024, 64, False),
    ("fwdbwd_bf16_b4h16n2048d64", "fwdbwd", "bf16", 4, 16, 2048, 64, False),
    ("fwd_e4m3_b4h16n4096d128", "fwd8", "e4m3", 4, 16, 4096, 128, False),
]
WORKLOAD = ("bf16 fwd B1 H32 N16384 d128 (non-causal + causal) + bf16 fwd B4 H16 N1024 d64 "
            "+ bf16 fwd+bwd B4 H16 N2048 d64 + e4m3 fwd B4 H16 N4096 d128")
LAUNCHES = {"fwd": 1, "fwd8": 1, "fwdbwd": 4}  # our kernels per part per step


def flops(kind, B, H, N, d, causal):
    f = {"fwd": 4, "fwd8": 4, "fwdbwd": 14}[kind] * B * H * N * N * d
    return f / 2 if causal else f


def recorded_traffic(key):
    """DRAM bytes per launch of one kernel (or one call's kernels) from the committed
    ncu capture record ``profiles/roofline_traffic.json[key]``, or None if there is no
    record or the sources it was taken on have changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(key)
    if rec is None:
        return None
    h = hashlib.sha256()
    for f in rec["source_files"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return rec["traffic_bytes_per_launch"] if h.hexdigest() == rec["source_sha256"] else None


def roofline_record(kernel, achieved, peak, peak_source, traffic_key, algorithmic_bytes):
    """Roofline entry of a tensor-bound launch: achieved = algorithmic FLOP per launch over
    its CUDA-event duration, against the measured peak of its dtype."""
    return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_source": peak_source,
            "traffic": recorded_traffic(traffic_key),
            "traffic_unit": "bytes per launch (ncu dram read+write)",
            "algorithmic_bytes": algorithmic_bytes}


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings over the process group (the slowest rank
    sets the job's time); the values unchanged when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tflops(world, step_flop, ms_step):
    """Whole-job throughput: each of `world` replicas runs one step in ms_step."""
    return world * step_flop / (ms_step * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"bf16": p["bf16_tflops"], "bf16_sustained": p.get("bf16_tflops_sustained"),
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = str(index)
        try:  # address the GPU by UUID: robust to CUDA_VISIBLE_DEVICES remapping
            import torch
            self.index = "GPU-" + str(torch.cuda.get_device_properties(index).uuid)
        except Exception:  # noqa: BLE001
            pass
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.index, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for ln in (self.out or "").splitlines():
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, f in zip(names, flags)
                          if f.lower() == "active"})
        loaded = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- our arm
_INPUT_CACHE = {}


def make_part(torch, fa, inputs, part, dev):
    name, kind, dt, B, H, N, d, causal = part
    key = (kind, dt, B, H, N, d)
    if key not in _INPUT_CACHE:  # parts with equal shapes share one input batch
        x = inputs.attention_inputs(B, H, N, d, dt, with_do=(kind == "fwdbwd"))
        host = {n: t.pin_memory() for n, t in x.items() if torch.is_tensor(t)}
        _INPUT_CACHE[key] = (x, host, {n: t.to(dev) for n, t in host.items()})
    x, host, dev_in = _INPUT_CACHE[key]
    P = {"part": part, "host": host, "scale": 1.0 / math.sqrt(d), "dev": dev_in}
    out_dtype = torch.bfloat16
    P["o"] = torch.empty((B, H, N, d), dtype=out_dtype, device=dev)
    P["lse"] = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    outs = {"o": P["o"]}
    if kind == "fwd8":
        P["descales"] = (x["q_descale"], x["k_descale"], x["v_descale"])
    if kind == "fwdbwd":
        P["ws"] = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
        for g in ("dq", "dk", "dv"):
            P[g] = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
            outs[g] = P[g]
    P["outs"] = outs
    P["host_out"] = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in outs.items()}
    P["flop"] = flops(kind, B, H, N, d, causal)
    P["h2d"] = sum(t.numel() * t.element_size() for t in host.values())
    P["d2h"] = sum(t.numel() * t.element_size() for t in outs.values())
    return P


def run_part(fa, P, stream, mid_event=None):
    name, kind, dt, B, H, N, d, causal = P["part"]
    D = P["dev"]
    if kind == "fwd8":
        qd, kd, vd = P["descales"]
        fa.fa_fwd_fp8(D["q"], D["k"], D["v"], P["o"], P["lse"], qd, kd, vd, P["scale"], causal,
                      stream)
    else:
        fa.fa_fwd(D["q"], D["k"], D["v"], P["o"], P["lse"], P["scale"], causal, fa.FA_BF16, stream)
    if kind == "fwdbwd":
        if mid_event is not None:
            mid_event.record(stream)
        fa.fa_bwd(D["q"], D["k"], D["v"], P["o"], P["lse"], D["do"], P["dq"], P["dk"], P["dv"],
                  P["ws"], P["scale"], False, fa.FA_BF16, stream)


class E2EPipeline:
    """The step through the public API with its host<->device copies, pipelined:
    inputs are copied in on one stream, the parts run on the launch stream, outputs
    are copied out on a third, so the copies of one part overlap the compute of
    others.  Device inputs are double-buffered across steps (the next step's copies
    run during this step's compute); events order every buffer's reuse.  Parts that
    share one input batch (same shapes) copy it once per step."""

    def __init__(self, torch, fa, parts, stream):
        self.torch, self.fa, self.parts, self.stream = torch, fa, parts, stream
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        self.groups = {}
        for i, P in enumerate(parts):
            key = id(P["dev"])
            if key not in self.groups:
                spare = {n: torch.empty_like(t) for n, t in P["dev"].items()}
                self.groups[key] = {"host": P["host"], "devs": [P["dev"], spare],
                                    "ready": [ev(), ev()], "free": [ev(), ev()], "first": i}
            self.groups[key]["last"] = i
            P["group"] = key
        for P in parts:
            P["done"], P["out_copied"] = ev(), ev()
        self.k = 0
        self.h2d = sum(t.numel() * t.element_size() for g in self.groups.values()
                       for t in g["host"].values())
        self.d2h = sum(P["d2h"] for P in parts)

    def step(self):
        torch, stream, b = self.torch, self.stream, self.k % 2
        for i, P in enumerate(self.parts):
            g = self.groups[P["group"]]
            if g["first"] == i:
                self.s_in.wait_event(g["free"][b])     # the step before last is done with it
                with torch.cuda.stream(self.s_in):
                    for n, t in g["host"].items():
                        g["devs"][b][n].copy_(t, non_blocking=True)
                g["ready"][b].record(self.s_in)
            stream.wait_event(g["ready"][b])
            stream.wait_event(P["out_copied"])        # last step's outputs have left
            P["dev"] = g["devs"][b]
            run_part(self.fa, P, stream)
            P["done"].record(stream)
            if g["last"] == i:
                g["free"][b].record(stream)
            self.s_out.wait_event(P["done"])
            with torch.cuda.stream(self.s_out):
                for n, t in P["outs"].items():
                    P["host_out"][n].copy_(t, non_blocking=True)
            P["out_copied"].record(self.s_out)
        self.k += 1

    def join(self):
        """Make the launch stream wait for every copy issued so far."""
        for P in self.parts:
            self.stream.wait_event(P["out_copied"])


# ---------------------------------------------------------------- extras
# The widened rows, each timed alone after the main step (not part of `value`):
# name, what, B, H, H_kv, N, d, causal
EXTRAS = [
    ("bwd_bf16_b1h32n16384d128", "bwd", 1, 32, 32, 16384, 128, False),
    ("bwd_bf16_b1h32n16384d128_causal", "bwd", 1, 32, 32, 16384, 128, True),
    ("bwd_bf16_b4h16n2048d64_causal", "bwd", 4, 16, 16, 2048, 64, True),
    ("fwd_e4m3_b4h16n4096d128_causal", "fwd8", 4, 16, 16, 4096, 128, True),
    ("fwd_e4m3_per_head_b4h16n4096d128", "fwd8h", 4, 16, 16, 4096, 128, False),
    ("fwd_e4m3_per_block_b4h16n4096d128", "fwd8b", 4, 16, 16, 4096, 128, False),
    ("fwd_gqa_bf16_b1h32hkv8n16384d128_causal", "gqa_fwd", 1, 32, 8, 16384, 128, True),
    ("bwd_gqa_bf16_b1h32hkv8n16384d128_causal", "gqa_bwd", 1, 32, 8, 16384, 128, True),
    ("fwd_seq4shards_bf16_b1h32n16384d128_causal", "shard4", 1, 32, 32, 16384, 128, True),
]


def make_extra(torch, fa, inputs, ex, dev, stream):
    """Inputs on the device and a closure that runs the row once on `stream`.
    Returns (run, flop, sub) where sub names event-split pieces (or None)."""
    name, what, B, H, H_kv, N, d, causal = ex
    s = 1.0 / math.sqrt(d)
    bf = lambda shape, seed: inputs.cast(inputs.normal(shape, seed), "bf16").to(dev)
    f_fwd = flops("fwd", B, H, N, d, causal)
    f_bwd = flops("fwdbwd", B, H, N, d, causal) - f_fwd
    if what == "fwd8b":  # one E4M3 factor per 128-row block of each head
        qb = [inputs.quantize_e4m3_per_block(inputs.normal((B, H, N, d), 42 + i)) for i in range(3)]
        q8, k8, v8 = (c.to(dev) for c, _ in qb)
        bd = [f.to(dev) for _, f in qb]
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        return (lambda: fa.fa_fwd_fp8_per_block(q8, k8, v8, o, lse, *bd, s, causal, stream)), f_fwd, None
    if what in ("fwd8", "fwd8h"):
        x = inputs.attention_inputs(B, H, N, d, "e4m3")
        q8, k8, v8 = x["q"].to(dev), x["k"].to(dev), x["v"].to(dev)
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        if what == "fwd8":
            ds = (x["q_descale"], x["k_descale"], x["v_descale"])
            return (lambda: fa.fa_fwd_fp8(q8, k8, v8, o, lse, *ds, s, causal, stream)), f_fwd, None
        hd = [torch.full((B * H,), float(x[n + "_descale"]), device=dev) for n in "qkv"]
        return (lambda: fa.fa_fwd_fp8_per_head(q8, k8, v8, o, lse, *hd, s, causal, stream)), f_fwd, None
    q, do = bf((B, H, N, d), 42), bf((B, H, N, d), 45)
    k, v = bf((B, H_kv, N, d), 43), bf((B, H_kv, N, d), 44)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    if what == "gqa_fwd":
        return (lambda: fa.fa_fwd_gqa(q, k, v, o, lse, s, causal, fa.FA_BF16, stream)), f_fwd, None
    if what in ("bwd", "gqa_bwd"):
        (fa.fa_fwd if H == H_kv else fa.fa_fwd_gqa)(q, k, v, o, lse, s, causal, fa.FA_BF16, stream)
        ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fn = fa.fa_bwd if H == H_kv else fa.fa_bwd_gqa
        return (lambda: fn(q, k, v, o, lse, do, dq, dk, dv, ws, s, causal, fa.FA_BF16, stream)), \
            f_bwd, None
    # sequence sharded: every query against 4 key shards, then the lse merge
    S = 4
    n = N // S
    ks = [k[:, :, t * n:(t + 1) * n].contiguous() for t in range(S)]
    vs = [v[:, :, t * n:(t + 1) * n].contiguous() for t in range(S)]
    o_p = torch.empty((S, B, H, N, d), dtype=torch.float32, device=dev)
    l_p = torch.empty((S, B, H, N), dtype=torch.float32, device=dev)
    mid = torch.cuda.Event(enable_timing=True)
    # the shards are independent (on several GPUs they would run side by side): each runs
    # on its own stream after the launch stream's prior work, and the merge waits for all
    side = [torch.cuda.Stream(device=dev) for _ in range(S)]
    start, done = torch.cuda.Event(), [torch.cuda.Event() for _ in range(S)]

    def run():
        start.record(stream)
        for t in range(S):
            side[t].wait_event(start)
            fa.fa_fwd_kv_shard(q, ks[t], vs[t], o_p[t], l_p[t], s, causal, 0, t * n,
                               fa.FA_BF16, side[t])
            done[t].record(side[t])
        for t in range(S):
            stream.wait_event(done[t])
        mid.record(stream)
        fa.fa_lse_merge(o_p, l_p, o, lse, fa.FA_BF16, stream)
    # algorithmic bytes of the merge: every part's lse, the O rows of the parts whose
    # keys a row reached (under the causal mask, key shard t reaches rows >= t*n
    # only; the rest carry lse = -inf and are not read), the merged O (bf16) and lse
    rows = B * H * N
    reached = B * H * (sum(N - t * n for t in range(S)) if causal else S * N)
    merge_bytes = S * rows * 4 + reached * 4 * d + rows * (2 * d + 4)
    return run, f_fwd, {"mid": mid, "merge_bytes": merge_bytes, "launches": S + 1}


def time_extras(torch, fa, inputs, dev, stream, pk, iters=20, warmup=3):
    out = {}
    for ex in EXTRAS:
        name, what = ex[0], ex[1]
        run, fl, sub = make_extra(torch, fa, inputs, ex, dev, stream)
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        ms, merge_ms = [], []
        for _ in range(iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
            if sub is not None:
                merge_ms.append(sub["mid"].elapsed_time(e1))
        st = fa.fa_last_device_error()
        if st != 0:
            raise RuntimeError(f"{name}: device status {fa.fa_status_string(st)}")
        med = statistics.median(ms)
        tf = fl / (med * 1e-3) / 1e12
        rec = {"ms": round(med, 4), "mean_ms": round(sum(ms) / len(ms), 4), "tflops": round(tf, 1), "flop": fl}
        if what.startswith("fwd8"):
            rec["dtype"] = "e4m3"
        else:
            rec["pct_of_peak"] = round(100 * tf / pk["bf16"], 1)
        if sub is not None:
            mm = statistics.median(merge_ms)
            gbs = sub["merge_bytes"] / (mm * 1e-3) / 1e9
            rec["merge"] = {"kernel": "lse_merge_kernel<128,bf16>", "bound": "hbm", "ms": round(mm, 4),
                            "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                            "frac": round(gbs / pk["hbm_gbs"], 4),
                            "algorithmic_bytes": sub["merge_bytes"]}
        out[name] = rec
        del run, sub
        torch.cuda.empty_cache()
    return out


def fp8_peak(torch, dev):
    """Dense e4m3 GEMM throughput (torch._scaled_mm, 8192^3, best of 10)."""
    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.tensor(1.0, device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return 2 * n ** 3 / (best * 1e-3) / 1e12, "measured: torch._scaled_mm e4m3 8192^3 best of 10"
    except Exception as ex:  # noqa: BLE001 - report and fall back
        return None, f"unmeasured ({type(ex).__name__})"


def cpu_sample(oracle, inputs, budget_s):
    """Time the fp64 oracle on a bounded sample of the step's workload.
    Returns (metric FLOP of the sample, seconds, description)."""
    import numpy as np
    f64 = lambda t: t.float().numpy().astype(np.float64)
    units = []
    # rows of the long-sequence forward (non-causal and causal), one head each
    big = inputs.attention_inputs(1, 1, 16384, 128, "bf16")
    qb, kb, vb = f64(big["q"][0, 0]), f64(big["k"][0, 0]), f64(big["v"][0, 0])
    rng = np.random.default_rng(0)
    for causal in (False, True):
        rows = np.sort(rng.choice(16384, 32, replace=False))
        fl = sum(4 * ((r + 1) if causal else 16384) * 128 for r in rows)
        units.append((lambda rows=rows, c=causal: oracle.attn_fwd_rows(
            qb, kb, vb, rows, 1 / math.sqrt(128), c), fl))
    # one head of the fwd+bwd workload
    m = inputs.attention_inputs(1, 1, 2048, 64, "bf16", with_do=True)
    qm, km, vm, dm = (f64(m[n][0, 0]) for n in ("q", "k", "v", "do"))
    units.append((lambda: (oracle.attn_fwd(qm, km, vm, 1 / 8.0),
                           oracle.attn_bwd(qm, km, vm, dm, 1 / 8.0)), 14 * 2048 * 2048 * 64))
    # rows of the e4m3 forward on dequantised inputs
    e = inputs.attention_inputs(1, 1, 4096, 128, "e4m3")
    qe = oracle.e4m3_decode(e["q"][0, 0].numpy(), e["q_descale"])
    ke = oracle.e4m3_decode(e["k"][0, 0].numpy(), e["k_descale"])
    ve = oracle.e4m3_decode(e["v"][0, 0].numpy(), e["v_descale"])
    rows8 = np.arange(0, 4096, 64)
    units.append((lambda: oracle.attn_fwd_rows(qe, ke, ve, rows8, 1 / math.sqrt(128)),
                  4 * len(rows8) * 4096 * 128))
    total_f, reps = 0.0, 0
    t0 = time.perf_counter()
    while True:
        for fn, fl in units:
            fn()
            total_f += fl
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    desc = (f"{reps} x [32 rows non-causal + 32 rows causal of one N=16384 d=128 head, one "
            f"N=2048 d=64 head fwd+bwd, 64 rows of one N=4096 d=128 e4m3 head]")
    return total_f, dt, desc


def cpu_single_thread(oracle, inputs, seconds=2.0):
    """The oracle on one host thread over the whole fp32 worked configuration (B=H=1,
    N=128, d=64, non-causal), repeated for about `seconds`."""
    import numpy as np
    x = inputs.attention_inputs(1, 1, 128, 64, "f32")
    q, k, v = (x[n].numpy().astype(np.float64) for n in "qkv")
    fl, reps, t0 = 4 * 128 * 128 * 64, 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle.attn_fwd(q, k, v, 1 / 8.0, nthreads=1)
        reps += 1
    dt = time.perf_counter() - t0
    return {"value": round(reps * fl / dt / 1e9, 3), "unit": "GFLOP/s", "cores": 1,
            "sample": f"{reps} x fp32 forward B1 H1 N128 d64 (4.19 MFLOP each)",
            "ms_per_call": round(1e3 * dt / reps, 3)}


def bench_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import exact_io_aware_06_gb300 as fa
    from exact_io_aware_06_gb300 import inputs

    stream = torch.cuda.current_stream()
    chosen = [p for p in PARTS if not args.only or p[0] in args.only]
    if not chosen:
        raise SystemExit(f"--only names no part; parts are {[p[0] for p in PARTS]}")
    parts = [make_part(torch, fa, inputs, p, dev) for p in chosen]
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def step_timed(events, mids):
        for i, P in enumerate(parts):
            events[i].record(stream)
            run_part(fa, P, stream, mids[i])
        events[-1].record(stream)

    for _ in range(args.warmup):
        for P in parts:
            run_part(fa, P, stream)
    st = fa.fa_last_device_error()
    if st != 0:
        raise RuntimeError(f"device status {fa.fa_status_string(st)}")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(K)]
    # an extra event between the forward and the backward of the fwd+bwd part
    mids = [[torch.cuda.Event(enable_timing=True) if P["part"][1] == "fwdbwd" else None
             for P in parts] for _ in range(K)]
    barrier()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for k in range(K):
            step_timed(evs[k], mids[k])
        t_end.record(stream)
        barrier()
    total_ms = t_start.elapsed_time(t_end)
    st = fa.fa_last_device_error()
    if st != 0:
        raise RuntimeError(f"device status {fa.fa_status_string(st)}")
    part_ms = [[evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K)] for i in range(len(parts))]
    split_ms = {i: ([evs[k][i].elapsed_time(mids[k][i]) for k in range(K)],
                    [mids[k][i].elapsed_time(evs[k][i + 1]) for k in range(K)])
                for i, P in enumerate(parts) if P["part"][1] == "fwdbwd"}

    # e2e: same step with pinned host buffers, copies inside the timed region; at least
    # 10 steps whatever K is, so that the figure is stable at short runs
    Ke = max(10, K // 10)
    pipe = E2EPipeline(torch, fa, parts, stream)
    pipe.step()
    pipe.join()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.s_in.wait_stream(stream)   # the first copies start inside the timed region
    for _ in range(Ke):
        pipe.step()
    pipe.join()
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / Ke

    ms_step = total_ms / K
    ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms], dev)
    step_flop = sum(P["flop"] for P in parts)
    value = job_tflops(world, step_flop, ms_step)
    pk = peaks()
    fp8_tf, fp8_how = fp8_peak(torch, dev)
    extras = None if args.no_extras else time_extras(torch, fa, inputs, dev, stream, pk)
    if extras:
        for rec in extras.values():
            if rec.get("dtype") == "e4m3" and fp8_tf:
                rec["pct_of_fp8_peak"] = round(100 * rec["tflops"] / fp8_tf, 1)

    part_out = {}
    for P, ms in zip(parts, part_ms):
        name, kind, dt = P["part"][0], P["part"][1], P["part"][2]
        mean = sum(ms) / len(ms)
        tf = P["flop"] / (mean * 1e-3) / 1e12
        peak = (fp8_tf or 2 * pk["bf16"]) if dt == "e4m3" else pk["bf16"]
        part_out[name] = {"ms": round(mean, 4), "best_ms": round(min(ms), 4),
                          "tflops": round(tf, 1), "pct_of_peak": round(100 * tf / peak, 1),
                          "peak_tflops": round(peak, 1), "flop": P["flop"]}

    for i, (fms, bms) in split_ms.items():
        name, kind, dt, B, H, N, d, causal = parts[i]["part"]
        for sub, ms, f in (("fwd", fms, flops("fwd", B, H, N, d, causal)),
                           ("bwd", bms, flops("fwdbwd", B, H, N, d, causal) - flops("fwd", B, H, N, d, causal))):
            mean = sum(ms) / len(ms)
            tf = f / (mean * 1e-3) / 1e12
            part_out[name][sub] = {"ms": round(mean, 4), "tflops": round(tf, 1),
                                   "pct_of_peak": round(100 * tf / pk["bf16"], 1)}

    # The step mixes bf16 and e4m3 stages: its peak is the FLOP-weighted one, i.e. the
    # step's FLOP over the time every stage would take at its own dtype's peak.
    peak_of = lambda dt: (fp8_tf or 2 * pk["bf16"]) if dt == "e4m3" else pk["bf16"]
    ideal_s = sum(P["flop"] / (peak_of(P["part"][2]) * 1e12) for P in parts)
    step_peak = step_flop / ideal_s / 1e12
    dtypes = sorted({P["part"][2] for P in parts}, key=lambda t: t != "bf16")

    rooflines = {}
    if "fwd_bf16_b1h32n16384d128" in part_out:
        rec = part_out["fwd_bf16_b1h32n16384d128"]
        rooflines["fwd_bf16_b1h32n16384d128"] = roofline_record(
            "fwd_sm103_kernel<128,bf16> (B1 H32 N16384 d128 non-causal), one launch",
            rec["tflops"], pk["bf16"], f"{pk['source']} bf16 burst (sustained {pk['bf16_sustained']})",
            "fwd_bf16_b1h32n16384d128", 4 * 1 * 32 * 16384 * 128 * 2 + 32 * 16384 * 4)
    if "fwdbwd_bf16_b4h16n2048d64" in part_out:
        rec = part_out["fwdbwd_bf16_b4h16n2048d64"]["bwd"]
        n_elt = 4 * 16 * 2048 * 64
        rooflines["bwd_bf16_b4h16n2048d64"] = roofline_record(
            "fa_bwd d64 (B4 H16 N2048, non-causal): bwd_prep + bwd_main_kernel<64> + bwd_dq_convert",
            rec["tflops"], pk["bf16"], f"{pk['source']} bf16 burst", "bwd_bf16_b4h16n2048d64",
            8 * n_elt * 2 + 4 * 16 * 2048 * 4)
    if "fwd_e4m3_b4h16n4096d128" in part_out and fp8_tf:
        rec = part_out["fwd_e4m3_b4h16n4096d128"]
        n_elt = 4 * 16 * 4096 * 128
        rooflines["fwd_e4m3_b4h16n4096d128"] = roofline_record(
            "fwd_sm103_kernel<128,e4m3> (B4 H16 N4096 d128 non-causal), one launch",
            rec["tflops"], fp8_tf, "e4m3 torch._scaled_mm 8192^3 measured in this run",
            "fwd_e4m3_b4h16n4096d128", 3 * n_elt + 2 * n_elt + 4 * 16 * 4096 * 4)
    dominant = next(iter(rooflines.values()), None)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "+".join(dtypes), "data": "synthetic",
        "config": {"workload": WORKLOAD if not args.only else " + ".join(p[0] for p in chosen),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2: each part follows a part that streams >129 MB"},
        "pct_of_peak": round(100 * value / world / step_peak, 1),
        "pct_of_peak_basis": (f"of the FLOP-weighted peak {step_peak:.1f} TFLOP/s: bf16 stages at "
                              f"the measured bf16 burst {pk['bf16']}, e4m3 stages at the e4m3 peak "
                              f"measured in this run ({None if fp8_tf is None else round(fp8_tf, 1)})"),
        "parts": part_out,
        "extras": extras,
        "fp8_peak_tflops": None if fp8_tf is None else round(fp8_tf, 1), "fp8_peak_how": fp8_how,
        "roofline": dominant,
        "rooflines": rooflines,
        "e2e": {"value": round(job_tflops(world, step_flop, e2e_ms), 1), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 3), "steps": Ke,
                "h2d_bytes_per_step": pipe.h2d, "d2h_bytes_per_step": pipe.d2h,
                "copies": "pipelined: inputs in on one stream (double-buffered across steps), "
                          "outputs out on another, overlapping compute"},
        "gpu_launches": K * sum(LAUNCHES[P["part"][1]] for P in parts),
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        fl, dt, desc = cpu_sample(oracle, inputs, args.cpu_seconds)
        result["cpu_baseline"] = {"value": round(fl / dt / 1e12, 6), "unit": UNIT,
                                  "cores": oracle.max_threads(), "kind": "oracle",
                                  "sample": desc, "seconds": round(dt, 2),
                                  "single_thread_fp32_config": cpu_single_thread(oracle, inputs)}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


# ---------------------------------------------------------------- reference arm
def bench_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from exact_io_aware_06_gb300 import inputs
    for _ in range(args.warmup):
        cpu_sample(oracle, inputs, 0.0)
    total_f, total_t = 0.0, 0.0
    desc = None
    for _ in range(args.steps):
        fl, dt, desc = cpu_sample(oracle, inputs, 0.0)
        total_f += fl
        total_t += dt
    value = total_f / total_t / 1e12
    cores = oracle.max_threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_t / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": "single"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--only", nargs="+", default=None, metavar="PART",
                    help="run only these parts of the step (for profiling one kernel)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the separately timed variant rows (``extras``)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
