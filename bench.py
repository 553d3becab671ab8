"""Benchmark of the fused norm / SwiGLU + FP8 quantisation path on GB300.

One step = the whole hot path once over the prefill-stress workload: residual
add + Gemma RMSNorm + MXFP8 + bf16 copy at M=8192, H=6144, then OAI SwiGLU +
MXFP8 at M=8192, I=3072 (inputs N(0,1) with 0.1% outliers x100 and 1% zero
32-blocks). `value` is algorithmic HBM bytes per step / device time, in GB/s.

Also reported: µs per launch at decode sizes (M = 8 .. 192, CUDA graph of 200
back-to-back launches, median of 20 replays, the method of the MiniMax-M3.1
MXFP8 fusion page's microbenchmark), the roofline of the dominant kernel, an
end-to-end number through pinned host buffers, and the CPU oracle as a
baseline. `--impl reference` times the CPU oracle on the same workload.

Run: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused norm/swiglu+quant µs/launch (M=8-192); HBM GB/s vs peak at M=8192"
M_PREFILL, H, I_PREFILL = 8192, 6144, 3072
I_DECODE = 768
DECODE_MS = (8, 16, 32, 64, 128, 192)
ROTATE = 3
WORKLOAD = ("prefill stress M=8192: add+Gemma-RMSNorm+MXFP8+bf16 copy+residual at H=6144, "
            "then OAI-SwiGLU+MXFP8 (fp32 source) at I=3072; bf16 N(0,1), 0.1% outliers x100, 1% zero 32-blocks")


def norm_bytes(M: int, Hd: int, residual=True, normed=True, fmt="mxfp8") -> int:
    """Algorithmic HBM bytes of one norm launch (weight counted once)."""
    per_row = 2 * Hd + Hd  # x read, E4M3 written
    per_row += {"mxfp8": Hd // 32, "block128": 4 * (Hd // 128), "per_token": 4}[fmt]
    if residual:
        per_row += 4 * Hd   # residual read + updated residual written
    if normed:
        per_row += 2 * Hd
    return M * per_row + 2 * Hd


def swiglu_bytes(M: int, I: int, fmt="mxfp8") -> int:
    per_row = 4 * I + I + {"mxfp8": I // 32, "block128": 4 * (I // 128), "per_token": 4}[fmt]
    return M * per_row


def step_bytes() -> int:
    return norm_bytes(M_PREFILL, H) + swiglu_bytes(M_PREFILL, I_PREFILL)


def _kernel_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "swiglu_fp8_activation_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _measured_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(kernel)
    if not entry or entry.get("source_sha") != _kernel_sha():
        return None
    return entry.get("bytes_per_launch")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


# --------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock, power and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=5)

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Max of a float over the ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ GPU workload

def _c_args(lib, dev_set, out, fmt=0):
    """Raw C-ABI argument tuples of one norm and one SwiGLU launch."""
    import ctypes as C

    import torch

    from swiglu_fp8_activation_gb300.binding import F_GEMMA_WEIGHT, F_QUANT_FROM_FP32
    p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    x, r, w, gu = dev_set
    norm = (fmt, F_GEMMA_WEIGHT, x.shape[0], x.shape[1], 1e-6, p(x), p(r), p(out["r_out"]), p(w), p(out["q"]),
            p(out["s"]), p(out["n"]), stream)
    swiglu = (fmt, 0, F_QUANT_FROM_FP32, gu.shape[0], gu.shape[1] // 2, 1.702, 1.0, 7.0, p(gu), p(out["q2"]),
              p(out["s2"]), stream)
    return norm, swiglu


def _call(fn, args):
    st = fn(*args)
    if st != 0:
        raise RuntimeError(f"launch failed with status {st}")


class Prefill:
    """Device-resident inputs (ROTATE sets) and outputs of the prefill step."""

    def __init__(self, dev):
        import torch

        from swiglu_fp8_activation_gb300 import inputs, library
        nc, sc = inputs.workloads()["cfg5_prefill"]
        t = inputs.make_norm(nc)
        gu = inputs.make_swiglu(sc)
        self.host = {"x": t["x"], "r": t["r"], "w": t["w"], "gu": gu}
        self.sets = []
        for i in range(ROTATE):
            self.sets.append(tuple(v.to(dev) for v in (t["x"], t["r"], t["w"], gu)))
        M = nc.M
        self.out = {"q": torch.empty(M, H, dtype=torch.uint8, device=dev),
                    "s": torch.empty(M, H // 32, dtype=torch.uint8, device=dev),
                    "n": torch.empty(M, H, dtype=torch.bfloat16, device=dev),
                    "r_out": torch.empty(M, H, dtype=torch.bfloat16, device=dev),
                    "q2": torch.empty(M, I_PREFILL, dtype=torch.uint8, device=dev),
                    "s2": torch.empty(M, I_PREFILL // 32, dtype=torch.uint8, device=dev)}
        self.lib = library()
        self.args = [_c_args(self.lib, s, self.out) for s in self.sets]

    def step(self, k, ev=None):
        na, sa = self.args[k % ROTATE]
        if ev is not None:
            ev[0].record()
        _call(self.lib.rmsnorm_add_quant, na)
        if ev is not None:
            ev[1].record()
        _call(self.lib.swiglu_quant, sa)
        if ev is not None:
            ev[2].record()


def time_prefill(pf, steps, warmup, world):
    """The timed region: `warmup` untimed steps, then exactly `steps` steps
    bracketed by a barrier and a device synchronisation on both sides, timed
    by one CUDA event pair around them. Nothing is recorded between the two
    kernels, so each launch may overlap the previous one's tail as it does in
    a serving loop (programmatic dependent launch). Returns the total ms."""
    import torch
    for k in range(warmup):
        pf.step(k)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record()
    for k in range(steps):
        pf.step(k)
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end)


def time_prefill_split(pf, steps):
    """The same steps again, each kernel between its own pair of CUDA events,
    for the per-kernel durations inside the step. An event recorded between
    two kernels keeps the second from starting before the first has ended,
    so these durations add up to more than the step above. Returns (total
    ms, mean norm ms, mean SwiGLU ms)."""
    import torch
    for k in range(3):
        pf.step(k)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for k in range(steps):
        pf.step(k, evs[k])
    end.record()
    torch.cuda.synchronize()
    norm_ms = [e[0].elapsed_time(e[1]) for e in evs]
    swiglu_ms = [e[1].elapsed_time(e[2]) for e in evs]
    return start.elapsed_time(end), statistics.mean(norm_ms), statistics.mean(swiglu_ms)


def time_alone(pf, which, steps):
    """One kernel of the prefill step launched `steps` times back to back
    (inputs rotated over the buffer sets, each larger than L2), timed with
    CUDA events around the loop: µs per launch."""
    import torch
    idx = 0 if which == "norm" else 1
    fn = pf.lib.rmsnorm_add_quant if which == "norm" else pf.lib.swiglu_quant
    for k in range(3):
        _call(fn, pf.args[k % ROTATE][idx])
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for k in range(steps):
        _call(fn, pf.args[k % ROTATE][idx])
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / steps


def host_us_per_call(dev, calls=2000):
    """Host time of one eager call of the raw C ABI at M=8 (norm + MXFP8 +
    bf16 copy, H=6144), through ctypes, while the GPU runs the launches;
    beside it the ctypes floor (a call of sgq_abi_version, which does
    nothing)."""
    import ctypes as C

    import torch

    from swiglu_fp8_activation_gb300 import inputs, library
    lib = library()
    case = inputs.norm_case_gemma_mx(8)
    t = inputs.make_norm(case)
    x, r, w = (t[k].to(dev) for k in ("x", "r", "w"))
    q = torch.empty(8, H, dtype=torch.uint8, device=dev)
    sc = torch.empty(8, H // 32, dtype=torch.uint8, device=dev)
    n = torch.empty(8, H, dtype=torch.bfloat16, device=dev)
    ro = torch.empty_like(n)
    ptr = lambda a: C.c_void_p(a.data_ptr())
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (0, 1, 8, H, 1e-6, ptr(x), ptr(r), ptr(ro), ptr(w), ptr(q), ptr(sc), ptr(n), stream)
    fn = lib.rmsnorm_add_quant
    for _ in range(50):
        _call(fn, args)
    torch.cuda.synchronize()
    best, floor = float("inf"), float("inf")
    for _ in range(5):
        t0 = time.perf_counter()
        for _ in range(calls):
            fn(*args)
        best = min(best, (time.perf_counter() - t0) / calls * 1e6)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(calls):
            lib.sgq_abi_version()
        floor = min(floor, (time.perf_counter() - t0) / calls * 1e6)
    return round(best, 3), round(floor, 3)


def graph_us_per_launch(fn, iters=200, reps=20):
    """µs per launch: a CUDA graph of `iters` back-to-back launches, 3 warm
    replays, median of `reps` timed replays."""
    import torch
    fn()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(iters):
            fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e) * 1000.0 / iters)
    return statistics.median(ts)


def decode_table(dev):
    """µs per launch at M = 8..192 for the two decode workloads (fused norm
    +MXFP8+bf16 copy at H=6144, with a separate residual output and with the
    residual updated in place; OAI SwiGLU+MXFP8 at I=768), each beside its
    unfused chain (norm to bf16, then a separate MXFP8 quant; SwiGLU to bf16,
    then a separate quant), both chains' launches in one graph, as the pages'
    decode table compares them."""
    import torch

    from swiglu_fp8_activation_gb300 import (inputs, quantize_fp8, rmsnorm_add, rmsnorm_add_quant, swiglu,
                                              swiglu_quant)
    out = {"norm_mxfp8_bf16copy_H6144": {}, "norm_mxfp8_bf16copy_H6144_inplace": {}, "norm_then_quant_H6144": {},
           "swiglu_oai_mxfp8_I768": {}, "swiglu_then_quant_I768": {}}
    for M in DECODE_MS:
        nc = inputs.norm_case_gemma_mx(M)
        t = inputs.make_norm(nc)
        x, r, w = (t[k].to(dev) for k in ("x", "r", "w"))
        q = torch.empty(M, H, dtype=torch.uint8, device=dev)
        s = torch.empty(M, H // 32, dtype=torch.uint8, device=dev)
        n = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
        ro = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
        fn = lambda: rmsnorm_add_quant(x, w, residual_in=r, residual_out=ro, q_out=q, scale_out=s, normed_out=n)
        out["norm_mxfp8_bf16copy_H6144"][str(M)] = round(graph_us_per_launch(fn), 3)
        ri = r.clone()   # the residual updated in place, launch after launch
        fni = lambda: rmsnorm_add_quant(x, w, residual_in=ri, residual_out=ri, q_out=q, scale_out=s, normed_out=n)
        out["norm_mxfp8_bf16copy_H6144_inplace"][str(M)] = round(graph_us_per_launch(fni), 3)

        def norm_chain():
            rmsnorm_add(x, w, residual_in=r, residual_out=ro, normed_out=n)
            quantize_fp8(n, q_out=q, scale_out=s)
        out["norm_then_quant_H6144"][str(M)] = round(graph_us_per_launch(norm_chain), 3)
        gu = inputs.make_swiglu(inputs.swiglu_case_oai_mx(M)).to(dev)
        q2 = torch.empty(M, I_DECODE, dtype=torch.uint8, device=dev)
        s2 = torch.empty(M, I_DECODE // 32, dtype=torch.uint8, device=dev)
        a2 = torch.empty(M, I_DECODE, dtype=torch.bfloat16, device=dev)
        fn2 = lambda: swiglu_quant(gu, q_out=q2, scale_out=s2)
        out["swiglu_oai_mxfp8_I768"][str(M)] = round(graph_us_per_launch(fn2), 3)

        def swiglu_chain():
            swiglu(gu, out=a2)
            quantize_fp8(a2, q_out=q2, scale_out=s2)
        out["swiglu_then_quant_I768"][str(M)] = round(graph_us_per_launch(swiglu_chain), 3)
    return out


L2_BYTES = 129 * 2 ** 20


def _input_sets(nbytes: int, M: int) -> int:
    """Input sets a measurement rotates over: one at decode sizes (inputs
    resident in L2, as the pages' microbenchmark), else enough that the sets
    together exceed 2.5 times the L2, so every launch reads its inputs from
    HBM."""
    return 1 if M < 1024 else max(3, -(-int(2.5 * L2_BYTES) // nbytes))


def other_configs(dev):
    """µs per launch (CUDA-graph replay, as above) of the Qwen3-like 1x128 and
    MLA-like per-token workloads. At M >= 1024 the graph's launches rotate
    over input sets larger than L2 together."""
    import torch

    from swiglu_fp8_activation_gb300 import inputs, rmsnorm_add_quant, swiglu_quant
    res = {}
    w = inputs.workloads()
    for case in w["cfg3_block128"] + w["cfg4_per_token"]:
        k = [0]
        if isinstance(case, inputs.NormCase):
            t = inputs.make_norm(case)
            n_sets = _input_sets(t["x"].numel() * 2, case.M)
            xs, wt = [t["x"].to(dev) for _ in range(n_sets)], t["w"].to(dev)
            q = torch.empty(case.M, case.H, dtype=torch.uint8, device=dev)
            shape = (case.M, 1) if case.fmt == "per_token" else (case.M, case.H // 128)
            s = torch.empty(shape, dtype=torch.float32, device=dev)

            def fn(c=case, xs=xs, wt=wt, q=q, s=s):
                x = xs[k[0] % len(xs)]
                k[0] += 1
                rmsnorm_add_quant(x, wt, fmt=c.fmt, eps=c.eps, gemma=c.gemma, quant_from_fp32=c.from_fp32,
                                  q_out=q, scale_out=s)
            key, nbytes = f"{case.name}_W{case.H}_M{case.M}", norm_bytes(case.M, case.H, False, False, case.fmt)
        else:
            g = inputs.make_swiglu(case)
            n_sets = _input_sets(g.numel() * 2, case.M)
            gus = [g.to(dev) for _ in range(n_sets)]
            q = torch.empty(case.M, case.I, dtype=torch.uint8, device=dev)
            s = torch.empty(case.M, case.I // 128, dtype=torch.float32, device=dev)

            def fn(c=case, gus=gus, q=q, s=s):
                gu = gus[k[0] % len(gus)]
                k[0] += 1
                swiglu_quant(gu, fmt=c.fmt, act=c.act, quant_from_fp32=c.from_fp32,
                             round_act_bf16=c.round_act_bf16, q_out=q, scale_out=s)
            key, nbytes = f"{case.name}_I{case.I}_M{case.M}", swiglu_bytes(case.M, case.I, case.fmt)
        us = graph_us_per_launch(fn, iters=max(100, 3 * n_sets), reps=10)
        res[key] = {"us": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
                    "inputs": "resident in L2" if n_sets == 1 else f"rotated over {n_sets} sets (> L2)"}
    return res


def wide_rows(dev):
    """µs per launch (graph replay, inputs rotated over sets larger than L2
    together) of rows wider than one CTA covers, at M = 4096: RMSNorm +
    per-token FP8 at W = 24576 (a cluster of two CTAs a row), add + Gemma
    RMSNorm + MXFP8 + bf16 copy at H = 24576 (a cluster of two), and
    SiLU-and-mul + 1x128 at I = 24576 (two column segments a row)."""
    import torch

    from swiglu_fp8_activation_gb300 import inputs, rmsnorm_add_quant, swiglu_quant
    res = {}
    M, W = 4096, 24576
    k = [0]
    t = inputs.norm_inputs(M, W, seed=24576, x_std=1.0, r_std=None, w_mean=1.0, w_std=0.1)
    n_sets = _input_sets(M * W * 2, M)
    xs, w = [t["x"].to(dev) for _ in range(n_sets)], t["w"].to(dev)
    q = torch.empty(M, W, dtype=torch.uint8, device=dev)
    s = torch.empty(M, 1, dtype=torch.float32, device=dev)

    def pt():
        rmsnorm_add_quant(xs[k[0] % n_sets], w, fmt="per_token", gemma=False, q_out=q, scale_out=s)
        k[0] += 1
    us = graph_us_per_launch(pt, iters=max(100, 3 * n_sets), reps=10)
    nb = norm_bytes(M, W, False, False, "per_token")
    res[f"rmsnorm_per_token_W{W}_M{M}"] = {"us": round(us, 3), "GBps": round(nb / us / 1e3, 1)}
    del xs
    t = inputs.norm_inputs(M, W, seed=24577, x_std=1.0, r_std=1.0, w_mean=0.0, w_std=0.1)
    n_sets = _input_sets(M * W * 4, M)
    xr = [(t["x"].to(dev), t["r"].to(dev)) for _ in range(n_sets)]
    w = t["w"].to(dev)
    ro, n = torch.empty(M, W, dtype=torch.bfloat16, device=dev), torch.empty(M, W, dtype=torch.bfloat16, device=dev)
    s = torch.empty(M, W // 32, dtype=torch.uint8, device=dev)

    def mx():
        x, r = xr[k[0] % n_sets]
        rmsnorm_add_quant(x, w, residual_in=r, residual_out=ro, q_out=q, scale_out=s, normed_out=n)
        k[0] += 1
    us = graph_us_per_launch(mx, iters=max(100, 3 * n_sets), reps=10)
    res[f"gemma_add_rmsnorm_mxfp8_H{W}_M{M}"] = {"us": round(us, 3), "GBps": round(norm_bytes(M, W) / us / 1e3, 1)}
    del xr, ro, n
    g = inputs.swiglu_inputs(M, W, seed=24578, std=1.0)
    n_sets = _input_sets(g.numel() * 2, M)
    gus = [g.to(dev) for _ in range(n_sets)]
    s = torch.empty(M, W // 128, dtype=torch.float32, device=dev)

    def silu():
        swiglu_quant(gus[k[0] % n_sets], fmt="block128", act="silu_mul", quant_from_fp32=False, round_act_bf16=True,
                     q_out=q, scale_out=s)
        k[0] += 1
    us = graph_us_per_launch(silu, iters=max(100, 3 * n_sets), reps=10)
    res[f"silu_mul_block128_I{W}_M{M}"] = {"us": round(us, 3), "GBps": round(swiglu_bytes(M, W, "block128") / us / 1e3, 1)}
    return res


def allreduce_norm(dev):
    """µs per launch (graph replay, as the decode table) of the tensor-parallel
    all-reduce folded into the fused norm, the ranks' partials in this GPU's
    memory (on a multi-GPU node they are peers' memory, read over NVLink):
    TP4 add + Gemma RMSNorm + MXFP8 + bf16 copy at H=6144, and TP8 RMSNorm +
    per-token FP8 at H=7168, at M = 1, 8, 64; beside each, the plain fused
    norm of the same rows (one input instead of the partials)."""
    import torch

    from swiglu_fp8_activation_gb300 import allreduce_rmsnorm_add_quant, inputs, rmsnorm_add_quant
    res = {}
    for name, n, Hd, fmt, gemma, normed, resid in (("tp4_gemma_norm_mxfp8_bf16copy_H6144", 4, 6144, "mxfp8", True,
                                                    True, True),
                                                   ("tp8_rmsnorm_per_token_H7168", 8, 7168, "per_token", False,
                                                    False, False)):
        row = {}
        for M in (1, 8, 64):
            parts = [inputs.norm_inputs(M, Hd, seed=k, x_std=1.0, r_std=None, w_mean=0.0, w_std=0.1)["x"].to(dev)
                     for k in range(n)]
            t = inputs.norm_inputs(M, Hd, seed=99, x_std=1.0, r_std=1.0, w_mean=0.0 if gemma else 1.0, w_std=0.1)
            w = t["w"].to(dev)
            r = t["r"].to(dev) if resid else None
            ro = torch.empty_like(r) if resid else None
            q = torch.empty(M, Hd, dtype=torch.uint8, device=dev)
            s = torch.empty(M, Hd // 32 if fmt == "mxfp8" else 1, dtype=torch.uint8 if fmt == "mxfp8" else torch.float32,
                            device=dev)
            nrm = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev) if normed else None
            fused = lambda: allreduce_rmsnorm_add_quant(parts, w, fmt=fmt, gemma=gemma, residual_in=r, residual_out=ro,
                                                        q_out=q, scale_out=s, normed_out=nrm)
            plain = lambda: rmsnorm_add_quant(parts[0], w, fmt=fmt, gemma=gemma, residual_in=r, residual_out=ro,
                                              q_out=q, scale_out=s, normed_out=nrm)
            row[str(M)] = {"allreduce_norm": round(graph_us_per_launch(fused, iters=100, reps=10), 3),
                           "norm_alone": round(graph_us_per_launch(plain, iters=100, reps=10), 3)}
        res[name] = row
    return res


def qkv_norm_configs(dev):
    """µs per launch (graph replay) of the q/kv latent norms of multi-head
    latent attention: q [M,1536] normed + per-token FP8, kv [M,512] normed to
    bf16, both read as column ranges of one [M,2112] projection output. One
    two-segment launch against two single-norm launches on copies of the
    same rows."""
    import torch

    from swiglu_fp8_activation_gb300 import rmsnorm_add_quant, rmsnorm_dual_quant
    res = {}
    Ha, Hb = 1536, 512
    for M in (1, 64, 4096):
        g = torch.Generator().manual_seed(M)
        buf = (torch.randn(M, Ha + Hb + 64, generator=g)).to(torch.bfloat16).to(dev)
        wa = (1 + 0.1 * torch.randn(Ha, generator=g)).to(torch.bfloat16).to(dev)
        wb = (1 + 0.1 * torch.randn(Hb, generator=g)).to(torch.bfloat16).to(dev)
        xa, xb = buf[:, :Ha], buf[:, Ha:Ha + Hb]
        fn = lambda: rmsnorm_dual_quant(xa, wa, xb, wb)
        xa_c, xb_c = xa.contiguous(), xb.contiguous()
        qa = torch.empty(M, Ha, dtype=torch.uint8, device=dev)
        sa = torch.empty(M, 1, dtype=torch.float32, device=dev)
        nb = torch.empty(M, Hb, dtype=torch.bfloat16, device=dev)
        qb = torch.empty(M, Hb, dtype=torch.uint8, device=dev)
        sb = torch.empty(M, 1, dtype=torch.float32, device=dev)

        def two():
            rmsnorm_add_quant(xa_c, wa, fmt="per_token", gemma=False, q_out=qa, scale_out=sa)
            rmsnorm_add_quant(xb_c, wb, fmt="per_token", gemma=False, q_out=qb, scale_out=sb, normed_out=nb)
        res[f"M{M}"] = {"dual_us": round(graph_us_per_launch(fn, iters=100, reps=10), 3),
                        "two_launches_us": round(graph_us_per_launch(two, iters=100, reps=10), 3)}
    return res


def time_e2e(pf, dev, steps, chunks=2):
    """The same step through the public API with host buffers. Every step
    copies x, r and gate_up from pinned host memory, runs both ops, and copies
    every output back to pinned host memory. The M rows are cut into `chunks`
    row blocks on three streams (H2D copy, compute, D2H copy) so that copies of
    one block overlap the kernels of its neighbours. Two blocks measured
    fastest on GB300 (1.88 ms per step against 2.07 ms for 8 and 5.9 ms for
    32, where issuing the copies becomes the cost; plain pinned copies of the
    same bytes in both directions at once take 1.74 ms). Returns (ms/step,
    H2D bytes, D2H bytes)."""
    import torch

    from swiglu_fp8_activation_gb300 import rmsnorm_add_quant, swiglu_quant
    hin = {k: pf.host[k].pin_memory() for k in ("x", "r", "gu")}
    x, r, w, gu = pf.sets[0]
    o = pf.out
    hout = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in o.items()}
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = sum(v.numel() * v.element_size() for v in hout.values())
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    M = x.shape[0]
    bounds = [(i * M // chunks, (i + 1) * M // chunks) for i in range(chunks)]
    dev_in = {"x": x, "r": r, "gu": gu}

    def one():
        done_in, done_comp = [], []
        for a, b in bounds:
            with torch.cuda.stream(s_in):
                for k, t in dev_in.items():
                    t[a:b].copy_(hin[k][a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
                done_in.append(e)
        for (a, b), e in zip(bounds, done_in):
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(e)
                rmsnorm_add_quant(x[a:b], w, residual_in=r[a:b], residual_out=o["r_out"][a:b], q_out=o["q"][a:b],
                                  scale_out=o["s"][a:b], normed_out=o["n"][a:b], stream=s_comp)
                swiglu_quant(gu[a:b], q_out=o["q2"][a:b], scale_out=o["s2"][a:b], stream=s_comp)
                e2 = torch.cuda.Event()
                e2.record(s_comp)
                done_comp.append(e2)
        for (a, b), e in zip(bounds, done_comp):
            with torch.cuda.stream(s_out):
                s_out.wait_event(e)
                for k, v in o.items():
                    hout[k][a:b].copy_(v[a:b], non_blocking=True)
        # the next step's copies into the device inputs wait for this step's kernels
        s_in.wait_stream(s_comp)
        s_comp.wait_stream(s_out)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for _ in range(steps):
        one()
    s_in.wait_stream(s_out)
    end.record(s_in)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, h2d, d2h


def cpu_oracle_gbps(budget_s: float, rows_per_chunk: int = 8, host=None):
    """The CPU oracle as it stands (single thread, no diagnostics) on prefill
    rows, norm then SwiGLU in turns, until `budget_s` seconds have passed.
    Returns (GB/s on the same algorithmic bytes, rows processed, seconds)."""
    import oracle
    from swiglu_fp8_activation_gb300 import inputs
    if host is None:
        nc, sc = inputs.workloads()["cfg5_prefill"]
        t = inputs.make_norm(nc)
        host = {"x": t["x"], "r": t["r"], "w": t["w"], "gu": inputs.make_swiglu(sc)}
    xb, rb, wb = (inputs.bf16_bits(host[k]) for k in ("x", "r", "w"))
    gub = inputs.bf16_bits(host["gu"])
    done_rows, nbytes = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s and done_rows < M_PREFILL:
        sl = slice(done_rows, done_rows + rows_per_chunk)
        oracle.rmsnorm_add_quant("mxfp8", xb[sl], rb[sl], wb, eps=1e-6, gemma=True, from_fp32=False,
                                 diagnostics=False)
        oracle.swiglu_quant("mxfp8", "swiglu_oai", gub[sl], from_fp32=True, diagnostics=False)
        n = xb[sl].shape[0]
        nbytes += norm_bytes(n, H) - 2 * H + swiglu_bytes(n, I_PREFILL)
        done_rows += n
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, done_rows, dt


def cpu_oracle_threads_gbps(budget_s: float, threads: int, rows_per_chunk: int = 8, host=None):
    """The same oracle on `threads` host threads at once, each taking its own
    row blocks (the C oracle runs outside the interpreter lock), for about
    `budget_s` seconds of wall time. Returns (GB/s, rows, seconds)."""
    import concurrent.futures as cf

    import oracle
    from swiglu_fp8_activation_gb300 import inputs
    if host is None:
        nc, sc = inputs.workloads()["cfg5_prefill"]
        t = inputs.make_norm(nc)
        host = {"x": t["x"], "r": t["r"], "w": t["w"], "gu": inputs.make_swiglu(sc)}
    xb, rb, wb = (inputs.bf16_bits(host[k]) for k in ("x", "r", "w"))
    gub = inputs.bf16_bits(host["gu"])
    oracle.lib()
    t0 = time.perf_counter()

    def worker(k):
        rows = nbytes = 0
        start = k * rows_per_chunk
        while time.perf_counter() - t0 < budget_s and start < M_PREFILL:
            sl = slice(start, start + rows_per_chunk)
            oracle.rmsnorm_add_quant("mxfp8", xb[sl], rb[sl], wb, eps=1e-6, gemma=True, from_fp32=False,
                                     diagnostics=False)
            oracle.swiglu_quant("mxfp8", "swiglu_oai", gub[sl], from_fp32=True, diagnostics=False)
            n = xb[sl].shape[0]
            nbytes += norm_bytes(n, H) - 2 * H + swiglu_bytes(n, I_PREFILL)
            rows += n
            start += threads * rows_per_chunk
        return rows, nbytes

    with cf.ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(worker, range(threads)))
    dt = time.perf_counter() - t0
    return sum(b for _, b in res) / dt / 1e9, sum(r for r, _ in res), dt


# ---------------------------------------------------------------- arms

def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step runs the oracle on a
    bounded sample of the same workload (16 rows of the norm, 16 of SwiGLU)."""
    if rank != 0:
        return
    import oracle
    from swiglu_fp8_activation_gb300 import inputs
    oracle.lib()
    nc, sc = inputs.workloads()["cfg5_prefill"]
    t = inputs.make_norm(nc)
    host = {"x": t["x"], "r": t["r"], "w": t["w"], "gu": inputs.make_swiglu(sc)}
    rows = 16
    xb, rb, wb = (inputs.bf16_bits(host[k]) for k in ("x", "r", "w"))
    gub = inputs.bf16_bits(host["gu"])

    def step(k):
        sl = slice((k * rows) % M_PREFILL, (k * rows) % M_PREFILL + rows)
        oracle.rmsnorm_add_quant("mxfp8", xb[sl], rb[sl], wb, eps=1e-6, gemma=True, from_fp32=False,
                                 diagnostics=False)
        oracle.swiglu_quant("mxfp8", "swiglu_oai", gub[sl], from_fp32=True, diagnostics=False)

    for k in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(args.warmup + k)
    dt = time.perf_counter() - t0
    nbytes = args.steps * (norm_bytes(rows, H) + swiglu_bytes(rows, I_PREFILL))
    gbps = nbytes / dt / 1e9
    sample = f"{rows} norm rows + {rows} SwiGLU rows of the M=8192 workload per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(gbps, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_rows_per_step": rows},
            "cpu_baseline": {"value": round(gbps, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbps, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _gpu_id():
    """nvidia-smi's id of the current CUDA device (its UUID), if nvidia-smi knows it."""
    try:
        import torch
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        gid = u if u.startswith("GPU-") else f"GPU-{u}"
        r = subprocess.run(["nvidia-smi", "-i", gid, "--query-gpu=index", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=30)
        return gid if r.returncode == 0 else None
    except Exception:
        return None


def run_ours(args, world, rank, local):
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import oracle
    oracle.lib()   # build the CPU oracle before any timing
    pf = Prefill(dev)
    peak, peak_kind = _peaks()
    with ClockSampler(_gpu_id()) as clocks:
        total_ms = time_prefill(pf, args.steps, args.warmup, world)
        split_ms, norm_ms, swiglu_ms = time_prefill_split(pf, args.steps)
        decode = decode_table(dev) if rank == 0 and not args.quick else None
        others = other_configs(dev) if rank == 0 and not args.quick else None
        qkv = qkv_norm_configs(dev) if rank == 0 and not args.quick else None
        wide = wide_rows(dev) if rank == 0 and not args.quick else None
        arn = allreduce_norm(dev) if rank == 0 and not args.quick else None
    total_ms = max_over_ranks(total_ms, world)
    alone_steps = max(args.steps, 200)
    norm_alone_us = time_alone(pf, "norm", alone_steps)
    swiglu_alone_us = time_alone(pf, "swiglu", alone_steps)
    host_us, ctypes_us = host_us_per_call(dev) if rank == 0 and not args.quick else (None, None)
    e2e_ms, h2d, d2h = time_e2e(pf, dev, args.e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, world)
    if rank != 0:
        barrier(world)
        return
    sb = step_bytes()
    ms_step = total_ms / args.steps
    value = world * sb / (ms_step * 1e-3) / 1e9
    nb = norm_bytes(M_PREFILL, H)
    norm_gbs = nb / (norm_ms * 1e-3) / 1e9
    swiglu_gbs = swiglu_bytes(M_PREFILL, I_PREFILL) / (swiglu_ms * 1e-3) / 1e9
    cpu_gbs, cpu_rows, cpu_s = cpu_oracle_gbps(args.cpu_budget, host=pf.host)
    ncores = os.cpu_count() or 1
    cpu_all, cpu_all_rows, cpu_all_s = cpu_oracle_threads_gbps(min(2.0, args.cpu_budget), ncores, host=pf.host)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_PREFILL, "H": H, "I": I_PREFILL, "format": "mxfp8",
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"inputs larger than L2, rotated over {ROTATE} buffer sets",
                   "bytes_per_step": sb},
        "roofline": {"bound": "hbm", "kernel": "norm_quant_kernel (add+Gemma RMSNorm+MXFP8+bf16 copy)",
                     "achieved": round(norm_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(norm_gbs / peak, 4), "peak_kind": peak_kind,
                     "traffic": _measured_traffic("norm_mxfp8_H6144_M8192"), "algorithmic_bytes": nb,
                     "timed": f"the norm's mean duration over {args.steps} steps with an event pair around each kernel"},
        "step_frac": round(value / world / peak, 4),
        "kernels": {"norm_us": round(norm_ms * 1e3, 2), "norm_GBps": round(norm_gbs, 1),
                    "swiglu_us": round(swiglu_ms * 1e3, 2), "swiglu_GBps": round(swiglu_gbs, 1),
                    "swiglu_frac": round(swiglu_gbs / peak, 4),
                    "evented_step_us": round(split_ms / args.steps * 1e3, 2),
                    "note": "norm_us / swiglu_us: each kernel between its own event pair, in a second pass of the "
                            "same steps (the events keep each kernel from overlapping its neighbour's tail)",
                    "alone": {"launches": alone_steps,
                              "norm_us": round(norm_alone_us, 2),
                              "norm_frac": round(nb / (norm_alone_us * 1e-6) / 1e9 / peak, 4),
                              "swiglu_us": round(swiglu_alone_us, 2),
                              "swiglu_frac": round(swiglu_bytes(M_PREFILL, I_PREFILL) / (swiglu_alone_us * 1e-6)
                                                   / 1e9 / peak, 4)},
                    # SwiGLU's added cost inside the step: the step's time less the norm's time back to
                    # back (each norm launch there also writes back its predecessor's dirty lines, as the
                    # SwiGLU kernel does for the norm inside the step)
                    "in_step_marginal": {
                        "swiglu_us": round(ms_step * 1e3 - norm_alone_us, 2),
                        "swiglu_frac": round(swiglu_bytes(M_PREFILL, I_PREFILL)
                                             / max((ms_step * 1e3 - norm_alone_us) * 1e-6, 1e-12) / 1e9 / peak, 4),
                        "note": "step time (no events) minus the norm's back-to-back time, same run"}},
        "host_us_per_eager_call_M8": {"rmsnorm_add_quant": host_us, "ctypes_floor": ctypes_us},
        "decode_us_per_launch": decode,
        "other_configs": others,
        "qkv_latent_norm_us": qkv,
        "wide_rows_us": wide,
        "allreduce_norm_us": arn,
        "e2e": {"value": round(sb / (e2e_ms * 1e-3) / 1e9 * world, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 3),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "cpu_baseline": {"value": round(cpu_gbs, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{cpu_rows} rows of each op of the M=8192 workload in {cpu_s:.1f} s",
                         "arch": platform.machine()},
        "cpu_baseline_all_cores": {"value": round(cpu_all, 5), "unit": "GB/s", "cores": ncores, "kind": "oracle",
                                   "sample": f"{cpu_all_rows} rows of each op in {cpu_all_s:.1f} s on {ncores} threads",
                                   "arch": platform.machine()},
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    barrier(world)


def run_profile(args):
    """One kernel only (for ncu): `--warmup` untimed then `--steps` timed
    launches. norm / swiglu: the M=8192 prefill workload (inputs > L2,
    rotated). pertoken: RMSNorm + per-token FP8 at W=7168, M=4096 (three
    rotating input sets, 176 MB together); pertoken512 the same at W=512
    (the persistent kernel). silu128: SiLU-and-mul + 1x128
    (bf16 roundings) at I=12288, M=2048 (three sets, 302 MB together);
    silu128_m256 the same at M=256 and norm128_m256 RMSNorm + 1x128 (fp32
    source) at W=4096, M=256 (the Qwen3-like workload's largest M).
    norm8: the decode norm (add + Gemma RMSNorm + MXFP8 + bf16 copy, separate
    residual output) at M=8, H=6144, inputs resident in L2; norm8_inplace:
    the same with the residual updated in place (whole rows, one CTA each);
    norm192 / norm192_inplace: the same at M=192."""
    import torch
    dev = torch.device("cuda", 0)
    if args.profile in ("silu128", "silu128_m256"):
        from swiglu_fp8_activation_gb300 import inputs, library
        import ctypes as C
        M, I = (2048 if args.profile == "silu128" else 256), 12288
        gu = inputs.swiglu_inputs(M, I, seed=2, std=1.0)
        sets = [gu.to(dev) for _ in range(ROTATE)]
        q = torch.empty(M, I, dtype=torch.uint8, device=dev)
        sc = torch.empty(M, I // 128, dtype=torch.float32, device=dev)
        lib = library()
        stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        arglist = [(1, 1, 4, M, I, 1.702, 1.0, 7.0, C.c_void_p(g.data_ptr()), C.c_void_p(q.data_ptr()),
                    C.c_void_p(sc.data_ptr()), stream) for g in sets]
        fn = lib.swiglu_quant
        nbytes = swiglu_bytes(M, I, "block128")
        get = lambda k: arglist[k % ROTATE]
    elif args.profile in ("norm8", "norm8_inplace", "norm192", "norm192_inplace"):
        from swiglu_fp8_activation_gb300 import inputs, library
        import ctypes as C
        case = inputs.norm_case_gemma_mx(192 if args.profile.startswith("norm192") else 8)
        t = inputs.make_norm(case)
        x, r, w = (t[k].to(dev) for k in ("x", "r", "w"))
        q = torch.empty(case.M, case.H, dtype=torch.uint8, device=dev)
        sc = torch.empty(case.M, case.H // 32, dtype=torch.uint8, device=dev)
        nrm = torch.empty(case.M, case.H, dtype=torch.bfloat16, device=dev)
        ro = r if args.profile.endswith("_inplace") else torch.empty_like(nrm)
        lib = library()
        stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        ptr = lambda a: C.c_void_p(a.data_ptr())
        args1 = (0, 1, case.M, case.H, case.eps, ptr(x), ptr(r), ptr(ro), ptr(w), ptr(q), ptr(sc), ptr(nrm), stream)
        fn = lib.rmsnorm_add_quant
        nbytes = norm_bytes(case.M, case.H)
        get = lambda k: args1
    elif args.profile in ("pertoken", "pertoken512", "norm128_m256"):
        from swiglu_fp8_activation_gb300 import inputs, library
        pt = args.profile.startswith("pertoken")
        W = 512 if args.profile == "pertoken512" else 7168
        case = inputs.norm_case_per_token(4096, W) if pt else inputs.norm_case_block128(256)
        t = inputs.make_norm(case)
        sets = [(t["x"].to(dev), t["w"].to(dev)) for _ in range(ROTATE)]
        q = torch.empty(case.M, case.H, dtype=torch.uint8, device=dev)
        sc = torch.empty(case.M, 1 if pt else case.H // 128, dtype=torch.float32, device=dev)
        import ctypes as C
        lib = library()
        stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        flags = 0 if pt else 2                      # 1x128 quantised from the fp32 normed value
        arglist = [(2 if pt else 1, flags, case.M, case.H, case.eps, C.c_void_p(x.data_ptr()), None, None,
                    C.c_void_p(w.data_ptr()), C.c_void_p(q.data_ptr()), C.c_void_p(sc.data_ptr()), None, stream)
                   for x, w in sets]
        fn, pick = lib.rmsnorm_add_quant, None
        nbytes = norm_bytes(case.M, case.H, False, False, case.fmt)
        get = lambda k: arglist[k % ROTATE]
    else:
        pf = Prefill(dev)
        fn = pf.lib.rmsnorm_add_quant if args.profile == "norm" else pf.lib.swiglu_quant
        pick = 0 if args.profile == "norm" else 1
        nbytes = norm_bytes(M_PREFILL, H) if args.profile == "norm" else swiglu_bytes(M_PREFILL, I_PREFILL)
        get = lambda k: pf.args[k % ROTATE][pick]
    for k in range(args.warmup):
        _call(fn, get(k))
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for k in range(args.steps):
        _call(fn, get(k))
    e.record()
    torch.cuda.synchronize()
    us = s.elapsed_time(e) * 1e3 / args.steps
    print(json.dumps({"profile": args.profile, "us_per_launch": round(us, 2),
                      "GBps": round(nbytes / us / 1e3, 1), "launches": args.warmup + args.steps}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of CPU oracle time")
    ap.add_argument("--quick", action="store_true", help="skip the decode and other-config tables")
    ap.add_argument("--profile", choices=("norm", "swiglu", "pertoken", "pertoken512", "silu128", "silu128_m256", "norm128_m256",
                                          "norm8", "norm8_inplace", "norm192", "norm192_inplace"),
                    help="time one kernel only (for ncu)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
