#!/usr/bin/env python3
"""Benchmark of the SRFT KV-cache hot path on GB300.

One step = one pass of the whole path over the packed-cache decode workload
(B=16 sequences, 32 query heads, 8 kv heads, d=128, 131072 cached tokens):
  1. srft_kv_quantize   : encode the whole fp16 K/V cache (2 x 16.8 M head
                          vectors) to int4 codes + fp32 group-16 scales;
  2. srft_kv_dequantize : decode it back to fp16;
  3. q4kv_decode_attention : one decode step of attention for all 512 query
                          rows, reading the packed cache directly;
  4. srft_kv_quantize   : append one new token per (sequence, kv head).
`value` = KV head vectors pushed through the step per second (all ranks).
Inputs are synthetic (seeded N(0,1) fp16), created on the device before the
timed region; they are 8.6 GB, far larger than the 129 MB L2, so no flush is
needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs the same workload on its own GPU (weak scaling,
no data exchange); rank 0 prints one JSON line.

Profiling cases: python bench.py --kernel quantize|dequantize|attention [--steps K] [--warmup W]
launches only that kernel on a cut-down decode workload (quantize/dequantize:
B=2, the full 131072 tokens x 8 kv heads, 4.2 M vectors, about 1.6 GB held;
attention: B=4, T=32768, a 201 MB packed cache) so that ncu captures stay
small; it prints one JSON line with the median event time per launch.
--kernel gemma_quantize|gemma_dequantize does the same for the d = 256 codec
on the full Gemma-3-1B-shaped cache (0.21 M vectors, 150 MB), and
--kernel d192_quantize|d192_dequantize (and d256_...) for the d = 192 (256)
codec on the decode cache shape at that d cut to B=2 (4.2 M vectors, about
2.2 GB (2.9 GB) held); d80_, d96_, d192_ and d256_ cases of quantize,
dequantize and attention run the same cuts at that head dimension;
long_attention runs attention on B=4 at the full T=131072 with 8 splits (512
chunks a split, so the per-split work weighs as little as on the full
decode workload; an 805 MB packed cache).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV vectors quantized/s and q4 decode-attn HBM GB/s (fraction of GB300 peak)"
WORKLOAD = "packed-cache decode attention B=16 Hq=32 Hkv=8 d=128 T=131072, int4/int4 group 16"
FALLBACK_HBM = 6800.0
# algorithmic bytes per unit
QUANT_BYTES_PER_VEC = 128 * 2 + 64 + 32      # read fp16 row, write int4 codes + 8 fp32 scales
DEQ_BYTES_PER_VEC = QUANT_BYTES_PER_VEC
ATTN_BYTES_PER_TOKEN_HEAD = 2 * (64 + 32)    # K and V: codes + scales per (b, t, kv head)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--kernel", default=None,
                    choices=("quantize", "dequantize", "attention", "gemma_quantize", "gemma_dequantize",
                             "d80_quantize", "d80_dequantize", "d80_attention", "d96_quantize", "d96_dequantize",
                             "d96_attention", "d192_quantize", "d192_dequantize", "d192_attention", "d256_attention",
                             "long_attention",
                             "d256_quantize", "d256_dequantize"),
                    help="profiling case: launch only this kernel on a small workload")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM, "fallback"


# the sources each timed kernel is built from: a recorded ncu traffic figure
# counts only while these are unchanged
KERNEL_SOURCES = {  # (api.cu encodes the tensor maps, whose L2 promotion affects the traffic)
    "srft_quantize_tc_kernel": ("codec_tc.cu", "codec_tc_common.cuh", "codec_impl.cuh", "tcgen05.cuh",
                                "srft_math.cuh", "ptx.cuh", "api.cu"),
    "srft_dequantize_tc_kernel": ("codec_tc.cu", "codec_tc_common.cuh", "codec_impl.cuh", "tcgen05.cuh",
                                  "srft_math.cuh", "ptx.cuh", "api.cu"),
    "q4kv_attn_split_kernel": ("attention.cu", "ptx.cuh", "srft_math.cuh", "api.cu"),
}


def kernel_source_sha(kernel: str = "srft_quantize_tc_kernel") -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "int8_kv_cache_srft_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` on the bench workload from the committed ncu record, if it was taken
    on the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    ent = j.get(kernel)
    if not ent or ent.get("source_sha") != kernel_source_sha(kernel):
        return None
    return float(ent["dram_bytes_per_launch"])


def max_over_ranks(ms: float, device=None) -> float:
    """The slowest rank's time: an all-reduce (MAX) over the default process group when one is initialised
    (NCCL on the GPUs, or any backend for the given device), else ms itself."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, units_per_rank: int, ms_per_step: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes units_per_rank per step."""
    return world * units_per_rank / (ms_per_step * 1e-3)


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples; stop() keeps the samples whose timestamps fall inside the
    timed region (the sampler starts earlier, since nvidia-smi takes a moment to print its first line)."""

    FIELDS = ("timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks.mem", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    @staticmethod
    def _when(stamp: str):
        import datetime

        try:  # local time of this machine, as time.time() sees it
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, t_begin: float, t_end: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            r = dict(zip(self.FIELDS, parts))
            try:
                r["sm"], r["max"] = float(r["clocks.sm"]), float(r["clocks.max.sm"])
            except ValueError:
                continue
            r["t"] = self._when(r["timestamp"])
            rows.append(r)
        inside = [r for r in rows if r["t"] is not None and t_begin <= r["t"] <= t_end]
        use = inside if inside else rows

        def med(key):
            vals = []
            for r in use:
                try:
                    vals.append(float(r[key]))
                except ValueError:
                    pass
            return statistics.median(vals) if vals else None

        reasons = sorted({n for r in use for n in self.REASONS
                          if r["clocks_event_reasons." + n].lower().startswith("active")})
        return {"sm_mhz": med("sm"), "sm_max_mhz": max(r["max"] for r in use) if use else None,
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "whole sampler run (no sample inside the timed region)",
                "mem_mhz": med("clocks.mem"), "power_w": med("power.draw")}


# ---------------------------------------------------------------------------
# CPU side: the fp64 oracle on a bounded sample of the same workload
# ---------------------------------------------------------------------------
def host_cores() -> dict:
    """Host cores this process may run on, and the thread count of the BLAS numpy calls (queried from the loaded
    OpenBLAS when threadpoolctl is absent)."""
    info = {"affinity_cores": len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count(),
            "cpu_count": os.cpu_count(), "blas_threads": None, "blas": None}
    try:
        from threadpoolctl import threadpool_info

        pools = [p for p in threadpool_info() if p.get("user_api") == "blas"]
        if pools:
            info["blas_threads"] = pools[0].get("num_threads")
            info["blas"] = pools[0].get("internal_api")
            return info
    except ImportError:
        pass
    import ctypes

    import numpy  # noqa: F401  (loads numpy's BLAS)

    try:
        with open("/proc/self/maps") as f:
            libs = sorted({ln.split()[-1] for ln in f if "openblas" in ln.lower() and ln.strip().endswith(".so")
                           or "openblas" in ln.lower() and ".so" in ln.split()[-1]})
    except OSError:
        libs = []
    for path in libs:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("openblas_get_num_threads64_", "scipy_openblas_get_num_threads64_", "openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                info["blas_threads"] = int(fn())
                info["blas"] = os.path.basename(path)
                return info
    return info


class _CpuClock:
    """Wall and process CPU time of a region: cpu/wall is the number of cores the region kept busy."""

    def __enter__(self):
        self.w0, self.c0 = time.perf_counter(), time.process_time()
        return self

    def __exit__(self, *exc):
        self.wall = time.perf_counter() - self.w0
        self.cpu = time.process_time() - self.c0
        self.busy_cores = self.cpu / self.wall if self.wall > 0 else None


def oracle_sample(seconds: float):
    """Time the oracle's quantize -> dequantize -> attention on slices of the decode workload (one sequence, one
    kv head, 4 query heads, 1024 tokens per slice) until about `seconds` of wall time has been spent."""
    import numpy as np
    from oracle import srft_oracle as O

    rng = np.random.default_rng(5)
    d, T, rep = 128, 1024, 4
    vecs, slices = 0, 0
    with _CpuClock() as clk:
        while True:
            k = rng.standard_normal((1, T, 1, d)).astype(np.float16).astype(np.float64)
            v = rng.standard_normal((1, T, 1, d)).astype(np.float16).astype(np.float64)
            q = rng.standard_normal((1, rep, d)).astype(np.float16).astype(np.float64)
            ek = O.srft_kv_quantize(k, None, 4, 16, 5)
            ev = O.srft_kv_quantize(v, None, 4, 16, 5)
            O.srft_kv_dequantize(ek["codes"], ek["scales"], None, 4, 16, 5)
            O.srft_kv_dequantize(ev["codes"], ev["scales"], None, 4, 16, 5)
            O.packed_decode_attention(q, {"bits": 4, "codes": ek["codes"], "scales": ek["scales"], "lam": None,
                                          "group": 16},
                                      {"bits": 4, "codes": ev["codes"], "scales": ev["scales"], "lam": None,
                                       "group": 16}, 5)
            vecs += 2 * T
            slices += 1
            if time.perf_counter() - clk.w0 >= seconds:
                break
    el = clk.wall
    hc = host_cores()
    return {"value": vecs / el, "unit": "KV vectors/s", "cores": hc["affinity_cores"], "kind": "oracle",
            "busy_cores": clk.busy_cores, "blas_threads": hc["blas_threads"], "blas": hc["blas"],
            "sample": f"{slices} slices of 1 sequence x 1 kv head x 1024 tokens x d=128 (K and V quantised, "
                      f"dequantised and attended by 4 query heads), {el:.1f} s; numpy fp64"}


def oracle_per_config(seconds_each: float):
    """The oracle on bounded samples of each workload, one figure per (workload, direction), plus a "fast CPU"
    line: the same fp64 arithmetic with the d x d SRFT matrix R formed once and applied as a matrix product
    (still O(d^2) a vector, no FFT).  Each sample is a whole number of (layer, token range) slices of the
    workload's own seeded input, grown until about `seconds_each` of wall time."""
    import numpy as np
    import torch
    from oracle import srft_oracle as O
    from int8_kv_cache_srft_gb300 import inputs as I

    out = {}

    def run(key, w, direction, fast):
        d, G, seed = w.d, w.group, w.sign_seed
        R = O.srft_matrix(d, seed) if fast else None
        toks = min(w.tokens, 512)
        n_vec, n_slices, mse_num, mse_den, wall, cpu = 0, 0, 0.0, 0.0, 0.0, 0.0
        while wall < seconds_each and n_vec < w.vectors_per_side:
            # one slice: 1 layer x toks tokens x all kv heads of the workload's distribution (inputs generated
            # outside the timed region)
            ws = w.resized(n_outer=1, tokens=toks, data_seed=w.data_seed * 1000 + n_slices)
            x = I.kv_side(ws, "k").to(torch.float64).numpy()
            lam = I.lam_table(ws, "k")
            lam = None if lam is None else lam[:, None].to(torch.float64).numpy()
            with _CpuClock() as clk:
                if fast:
                    z = x @ R.T
                    z = z if lam is None else z * lam
                    qv, sc, _ = O.quantize_groups(z, 4, G)
                    if direction == "dequantize":
                        zh = np.repeat(sc, G, axis=-1) * qv
                        xh = (zh if lam is None else zh / lam) @ R
                else:
                    enc = O.srft_kv_quantize(x, lam, 4, G, seed)
                    if direction == "dequantize":
                        xh = O.srft_kv_dequantize(enc["codes"], enc["scales"], lam, 4, G, seed)
            wall += clk.wall
            cpu += clk.cpu
            if direction == "dequantize":
                mse_num += float(((xh - x) ** 2).sum())
                mse_den += float((x ** 2).sum())
            n_vec += x.shape[1] * x.shape[2]
            n_slices += 1
        ent = {"vectors_per_s": n_vec / wall, "vectors": n_vec, "of_workload": n_vec / w.vectors_per_side,
               "seconds": wall, "busy_cores": cpu / wall if wall > 0 else None,
               "sample": f"{n_slices} slices of 1 layer x {toks} tokens x {w.kv_heads} kv heads (K side), d={d}"}
        if direction == "dequantize":
            ent["relative_mse"] = mse_num / mse_den
            ent["note"] = "quantize of the sample included (the dequantize input is the oracle's own codes)"
        out[key] = ent

    for name, w in (("tiny", I.TINY), ("gemma_d256", I.GEMMA), ("qwen_d128_lambda", I.QWEN)):
        for fast in (False, True):
            run(f"{name}_quantize" + ("_fast" if fast else ""), w, "quantize", fast)
    for fast in (False, True):
        run("gemma_d256_dequantize" + ("_fast" if fast else ""), I.GEMMA, "dequantize", fast)
    return out


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    per_step = []
    for _ in range(args.warmup):
        oracle_sample(0.0)
    for _ in range(args.steps):
        r = oracle_sample(max(0.5, args.cpu_seconds / max(args.steps, 1)))
        per_step.append(r["value"])
    val = statistics.median(per_step)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "KV vectors/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": "oracle slices (see cpu_baseline)"},
            "cpu_baseline": {"value": val, "unit": "KV vectors/s", "cores": r["cores"], "kind": "oracle",
                             "busy_cores": r["busy_cores"], "blas_threads": r["blas_threads"],
                             "sample": r["sample"]},
            "e2e": {"value": val, "unit": "KV vectors/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------
def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import int8_kv_cache_srft_gb300 as K
    from int8_kv_cache_srft_gb300 import inputs as I

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    K.library()
    w = I.DECODE
    B, Hkv, d, T, Hq, G = w.n_outer, w.kv_heads, w.d, w.tokens, w.q_heads, w.group
    t_cap = T + 64
    seed = w.sign_seed
    wd = w.resized(data_seed=w.data_seed + 100 * rank)
    xk, xv = I.kv_side(wd, "k", device=dev), I.kv_side(wd, "v", device=dev)
    q = I.query(wd, device=dev)
    sk, sv = K.alloc_side(B, t_cap, Hkv, d, 4, G, device=dev), K.alloc_side(B, t_cap, Hkv, d, 4, G, device=dev)
    sk.x, sv.x = xk, xv
    dk, dv = torch.empty_like(xk), torch.empty_like(xv)
    deq_k, deq_v = K.Side(sk.codes, sk.scales, 4, x=dk), K.Side(sv.codes, sv.scales, 4, x=dv)
    g = torch.Generator(device=dev).manual_seed(99 + rank)
    nk = torch.randn((B, 1, Hkv, d), generator=g, device=dev).half()
    nv = torch.randn((B, 1, Hkv, d), generator=g, device=dev).half()
    app_k, app_v = K.Side(sk.codes, sk.scales, 4, x=nk), K.Side(sv.codes, sv.scales, 4, x=nv)
    seq = torch.full((B,), T, dtype=torch.int32, device=dev)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, t_cap, 0), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    n_vec = 2 * B * T * Hkv
    LAUNCHES = 6

    ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for k in ("quant", "deq", "attn", "append")}
    times = {k: [] for k in ev}

    def step(timed_parts: bool):
        if timed_parts:
            ev["quant"][0].record(stream)
        K.srft_kv_quantize(sk, sv, B, T, Hkv, d, G, t_cap, 0, seed, stream)
        if timed_parts:
            ev["quant"][1].record(stream)
            ev["deq"][0].record(stream)
        K.srft_kv_dequantize(deq_k, deq_v, B, T, Hkv, d, G, t_cap, 0, seed, stream)
        if timed_parts:
            ev["deq"][1].record(stream)
            ev["attn"][0].record(stream)
        K.q4kv_decode_attention(q, out, sk, sv, B, Hq, Hkv, d, G, t_cap, seq, 0.0, seed, 0, ws, stream)
        if timed_parts:
            ev["attn"][1].record(stream)
            ev["append"][0].record(stream)
        K.srft_kv_quantize(app_k, app_v, B, 1, Hkv, d, G, t_cap, T, seed, stream)
        if timed_parts:
            ev["append"][1].record(stream)

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step(False)
    torch.cuda.synchronize()

    # per-kernel durations (events on the launching stream), outside the main timed loop
    for _ in range(10):
        step(True)
        torch.cuda.synchronize()
        for k, (a, b) in ev.items():
            times[k].append(a.elapsed_time(b))

    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step(False)
    e1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    clk = clocks.stop(t_begin, t_end)
    barrier()
    ms_total = e0.elapsed_time(e1)
    ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    value = job_value(world, n_vec, ms_step)

    # variants of the cache format on the same workload and kernels (outside the timed step): the Hadamard
    # rotation, and fp16 / e8m0 scale planes; each timed as the median of 10 launches with CUDA events on the
    # launching stream.  Algorithmic bytes follow the plane sizes (scales of 4, 2 or 1 bytes).
    def time_launch(fn, reps=10):
        ts = []
        for _ in range(reps + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts[2:])

    variants = {}
    for name, tr, sf in (("srht", "srht", "fp32"), ("fp16_scales", "srft", "fp16"), ("e8m0_scales", "srft", "e8m0")):
        sb = {"fp32": 4, "fp16": 2, "e8m0": 1}[sf]
        vec_bytes = 2 * d + d // 2 + (d // G) * sb
        tok_bytes = 2 * (d // 2 + (d // G) * sb)
        vk = K.alloc_side(B, t_cap, Hkv, d, 4, G, device=dev, transform=tr, scale_format=sf)
        vv = K.alloc_side(B, t_cap, Hkv, d, 4, G, device=dev, transform=tr, scale_format=sf)
        vk.x, vv.x = xk, xv
        qv = time_launch(lambda: K.srft_kv_quantize(vk, vv, B, T, Hkv, d, G, t_cap, 0, seed, stream))
        dqk = K.Side(vk.codes, vk.scales, 4, x=dk, transform=tr, scale_format=sf)
        dqv = K.Side(vv.codes, vv.scales, 4, x=dv, transform=tr, scale_format=sf)
        dv_ms = time_launch(lambda: K.srft_kv_dequantize(dqk, dqv, B, T, Hkv, d, G, t_cap, 0, seed, stream))
        av = time_launch(lambda: K.q4kv_decode_attention(q, out, vk, vv, B, Hq, Hkv, d, G, t_cap, seq, 0.0, seed, 0,
                                                         ws, stream))
        variants[name] = {"transform": tr, "scales": sf, "quant_ms": qv, "deq_ms": dv_ms, "attn_ms": av,
                          "quant_gbs": n_vec * vec_bytes / (qv * 1e-3) / 1e9,
                          "deq_gbs": n_vec * vec_bytes / (dv_ms * 1e-3) / 1e9,
                          "attn_gbs": B * T * Hkv * tok_bytes / (av * 1e-3) / 1e9,
                          "attn_bytes_per_token_head": tok_bytes}
        del vk, vv, dqk, dqv

    # other head dimensions on the same cache shape: d = 96 (the first 96 coordinates of the inputs), d = 80, 192
    # and 256 (the decode workload's generator at that d), all through the tensor-core codec, int4/int4,
    # group 16, fp32 scales; attention also on the raw fp16 cache of the same inputs
    def nonpow2_variant(dn, xkn, xvn, qn):
        vk = K.alloc_side(B, t_cap, Hkv, dn, 4, G, device=dev)
        vv = K.alloc_side(B, t_cap, Hkv, dn, 4, G, device=dev)
        vk.x, vv.x = xkn, xvn
        qv = time_launch(lambda: K.srft_kv_quantize(vk, vv, B, T, Hkv, dn, G, t_cap, 0, seed, stream))
        okn, ovn = torch.empty_like(xkn), torch.empty_like(xvn)
        dqk, dqv = K.Side(vk.codes, vk.scales, 4, x=okn), K.Side(vv.codes, vv.scales, 4, x=ovn)
        dv_ms = time_launch(lambda: K.srft_kv_dequantize(dqk, dqv, B, T, Hkv, dn, G, t_cap, 0, seed, stream))
        outn = torch.empty((B, Hq, dn), dtype=torch.float32, device=dev)
        wsn = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, dn, t_cap, 0), dtype=torch.uint8,
                          device=dev)
        av = time_launch(lambda: K.q4kv_decode_attention(qn, outn, vk, vv, B, Hq, Hkv, dn, G, t_cap, seq, 0.0, seed,
                                                         0, wsn, stream))
        del okn, ovn, dqk, dqv, vk, vv
        rkn = K.Side(xkn.permute(0, 2, 1, 3).contiguous(), None, 16)
        rvn = K.Side(xvn.permute(0, 2, 1, 3).contiguous(), None, 16)
        wsr = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, dn, T, 0), dtype=torch.uint8, device=dev)
        fn = time_launch(lambda: K.q4kv_decode_attention(qn, outn, rkn, rvn, B, Hq, Hkv, dn, G, T, seq, 0.0, seed,
                                                         0, wsr, stream))
        del rkn, rvn
        vecn = 2 * dn + dn // 2 + (dn // G) * 4
        tokn = 2 * (dn // 2 + (dn // G) * 4)
        return {"head_dim": dn, "transform": "srft", "scales": "fp32", "quant_ms": qv, "deq_ms": dv_ms,
                "attn_ms": av, "quant_gbs": n_vec * vecn / (qv * 1e-3) / 1e9,
                "deq_gbs": n_vec * vecn / (dv_ms * 1e-3) / 1e9,
                "attn_gbs": B * T * Hkv * tokn / (av * 1e-3) / 1e9, "attn_bytes_per_token_head": tokn,
                "fp16_cache_ms": fn, "attn_speedup_vs_fp16_cache": fn / av}

    variants["d96"] = nonpow2_variant(96, xk[..., :96].contiguous(), xv[..., :96].contiguous(),
                                      q[..., :96].contiguous())
    torch.cuda.empty_cache()
    # d = 80: the decode workload's generator at that d (int4 rows of 40 bytes: the attention reads them as rows
    # of token pairs)
    w80 = wd.resized(d=80)
    variants["d80"] = nonpow2_variant(80, I.kv_side(w80, "k", device=dev), I.kv_side(w80, "v", device=dev),
                                      I.query(w80, device=dev))
    torch.cuda.empty_cache()
    w192 = wd.resized(d=192)
    variants["d192"] = nonpow2_variant(192, I.kv_side(w192, "k", device=dev), I.kv_side(w192, "v", device=dev),
                                       I.query(w192, device=dev))
    torch.cuda.empty_cache()
    # the same cache shape at d = 256 (33.5 M vectors, 704 B each: 23.6 GB through each codec launch)
    w256 = wd.resized(d=256)
    variants["d256"] = nonpow2_variant(256, I.kv_side(w256, "k", device=dev), I.kv_side(w256, "v", device=dev),
                                       I.query(w256, device=dev))
    torch.cuda.empty_cache()

    other = other_workloads(K, I, torch, dev, stream, time_launch) if rank == 0 else None

    # fp16-cache comparator: the same attention kernel on the raw fp16 cache (head-major like the packed planes)
    raw_k = K.Side(xk.permute(0, 2, 1, 3).contiguous(), None, 16)
    raw_v = K.Side(xv.permute(0, 2, 1, 3).contiguous(), None, 16)
    ws16 = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, 0), dtype=torch.uint8, device=dev)
    t16 = []
    for i in range(13):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        K.q4kv_decode_attention(q, out, raw_k, raw_v, B, Hq, Hkv, d, G, T, seq, 0.0, seed, 0, ws16, stream)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            t16.append(a.elapsed_time(b))

    # end to end through the public API from pinned host memory: every step copies its inputs (K, V, q) host ->
    # device, runs the step and reads the attention output back, all on one stream.  The host link carries
    # about 211 GB/s with the GPU otherwise idle but drops to about 23 GB/s while a kernel saturates HBM with
    # reads, so copies overlapped with the step (a second stream and a second set of input buffers) made a step
    # take 85 ms instead of 46: they stay serialised.
    e2e = None
    if args.e2e_steps > 0:
        hk = xk.cpu().pin_memory()
        hv = xv.cpu().pin_memory()
        hq = q.cpu().pin_memory()
        hout = torch.empty_like(out, device="cpu").pin_memory()
        h2d = hk.numel() * 2 + hv.numel() * 2 + hq.numel() * 2
        d2h = hout.numel() * 4
        # one untimed step first, as for every other timed loop: the first copies out of freshly pinned
        # buffers run slower than the link's steady rate
        xk.copy_(hk, non_blocking=True)
        xv.copy_(hv, non_blocking=True)
        q.copy_(hq, non_blocking=True)
        step(False)
        hout.copy_(out, non_blocking=True)
        barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.e2e_steps):
            xk.copy_(hk, non_blocking=True)
            xv.copy_(hv, non_blocking=True)
            q.copy_(hq, non_blocking=True)
            step(False)
            hout.copy_(out, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(a.elapsed_time(b) / args.e2e_steps, dev)
        # the same copies alone (no kernels): the host link's rate, which bounds the end-to-end figure
        a.record(stream)
        for _ in range(args.e2e_steps):
            xk.copy_(hk, non_blocking=True)
            xv.copy_(hv, non_blocking=True)
            q.copy_(hq, non_blocking=True)
            hout.copy_(out, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        ms_copy = a.elapsed_time(b) / args.e2e_steps
        e2e = {"value": job_value(world, n_vec, ms_e2e), "unit": "KV vectors/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e, "copy_only_ms_per_step": ms_copy,
               "host_link_gbs_copy_only": (h2d + d2h) / (ms_copy * 1e-3) / 1e9,
               "bound": "host link: the step's copies alone take copy_only_ms_per_step of ms_per_step"}

    if rank != 0:
        return
    med = {k: statistics.median(v) for k, v in times.items()}
    peak, peak_kind = peaks()
    quant_bytes = n_vec * QUANT_BYTES_PER_VEC
    attn_bytes = B * T * Hkv * ATTN_BYTES_PER_TOKEN_HEAD
    achieved = quant_bytes / (med["quant"] * 1e-3) / 1e9
    attn_gbs = attn_bytes / (med["attn"] * 1e-3) / 1e9
    # one roofline entry per HBM-bound kernel of the step (algorithmic bytes per launch / median event time);
    # the line's "roofline" is the entry of the longest one
    rooflines = {}
    for part, kern, nbytes in (("quant", "srft_quantize_tc_kernel", quant_bytes),
                               ("deq", "srft_dequantize_tc_kernel", n_vec * DEQ_BYTES_PER_VEC),
                               ("attn", "q4kv_attn_split_kernel", attn_bytes)):
        gbs = nbytes / (med[part] * 1e-3) / 1e9
        tr = recorded_traffic(kern)
        rooflines[kern] = {"bound": "hbm", "kernel": kern, "ms": med[part], "achieved": gbs, "peak": peak,
                           "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak, "traffic": tr,
                           "traffic_over_algorithmic": None if tr is None else tr / nbytes,
                           "algorithmic_bytes_per_launch": nbytes}
    dominant = max(rooflines.values(), key=lambda r: r["ms"])
    fp16_ms = statistics.median(t16)
    for vname in variants:  # against the d = 128 fp16 cache unless the variant timed its own
        variants[vname].setdefault("attn_speedup_vs_fp16_cache", fp16_ms / variants[vname]["attn_ms"])
        # each kernel of the variant against the same measured HBM peak (algorithmic bytes / event time)
        for kk in ("quant", "deq", "attn"):
            variants[vname][kk + "_frac"] = variants[vname][kk + "_gbs"] / peak
    cpu = None
    if not args.no_cpu:
        cpu = oracle_sample(args.cpu_seconds)
        cpu["per_workload"] = oracle_per_config(args.cpu_seconds / 8)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "KV vectors/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "q_heads": Hq, "kv_heads": Hkv, "head_dim": d, "context": T,
                   "bits_k": 4, "bits_v": 4, "group": G, "scales": "fp32", "vectors_per_step": n_vec,
                   "step": "quantize cache + dequantize cache + decode attention + 1-token append",
                   "l2": "inputs 8.6 GB >> 129 MB L2, no flush needed"},
        "roofline": dominant,
        "rooflines": rooflines,
        "kernels_ms": med,
        "quantize": {"vectors_per_s": n_vec / (med["quant"] * 1e-3), "gbs": achieved, "frac": achieved / peak},
        "dequantize": {"vectors_per_s": n_vec / (med["deq"] * 1e-3),
                       "gbs": n_vec * DEQ_BYTES_PER_VEC / (med["deq"] * 1e-3) / 1e9,
                       "frac": n_vec * DEQ_BYTES_PER_VEC / (med["deq"] * 1e-3) / 1e9 / peak},
        "attention": {"int4_ms": med["attn"], "hbm_gbs": attn_gbs, "frac": attn_gbs / peak,
                      "frac_of_nominal_8000": attn_gbs / 8000.0, "decode_tokens_per_s": B / (med["attn"] * 1e-3),
                      "kv_tokens_per_s": B * T / (med["attn"] * 1e-3), "fp16_cache_ms": fp16_ms,
                      "fp16_cache_gbs": 2 * B * T * Hkv * d * 2 / (fp16_ms * 1e-3) / 1e9,
                      "int4_speedup_vs_fp16_cache": fp16_ms / med["attn"],
                      "algorithmic_bytes_per_launch": attn_bytes,
                      "traffic": recorded_traffic("q4kv_attn_split_kernel")},
        "append_us": med["append"] * 1e3,
        "variants": variants,
        "other_workloads": other,
        "gpu_launches": LAUNCHES * args.steps,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "kernel_source_sha": {k: kernel_source_sha(k) for k in KERNEL_SOURCES},
    }
    print(json.dumps(line), flush=True)


def other_workloads(K, I, torch, dev, stream, time_launch):
    """The codec workloads besides the decode cache, each launch timed alone (median of 10, CUDA events on the
    launching stream): the Gemma-3-1B-shaped cache (d = 256, 0.21 M vectors, 150 MB: L2 flushed before every
    launch by writing 256 MB), the Qwen2.5-1.5B-shaped cache with per-channel lambda (3.67 M vectors, 1.29 GB)
    and the K8V4 one-token append onto a prebuilt 7B-like cache (K int8 / V int4, 256 + 256 vectors a step)."""
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn, l2_flush):
        def run():
            fn()
        if not l2_flush:
            return time_launch(run)
        ts = []
        for _ in range(12):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts[2:])

    for key, w, l2_flush in (("gemma_d256", I.GEMMA, True), ("qwen_d128_lambda", I.QWEN, False)):
        n, T, H, d, G, seed = w.n_outer, w.tokens, w.kv_heads, w.d, w.group, w.sign_seed
        xk, xv = I.kv_side(w, "k", device=dev), I.kv_side(w, "v", device=dev)
        lk, lv = I.lam_table(w, "k", device=dev), I.lam_table(w, "v", device=dev)
        sk, sv = K.alloc_side(n, T, H, d, 4, G, device=dev), K.alloc_side(n, T, H, d, 4, G, device=dev)
        sk.x, sv.x, sk.lam, sv.lam = xk, xv, lk, lv
        qms = timed(lambda: K.srft_kv_quantize(sk, sv, n, T, H, d, G, T, 0, seed, stream), l2_flush)
        ok, ov = torch.empty_like(xk), torch.empty_like(xv)
        dk, dv = K.Side(sk.codes, sk.scales, 4, x=ok, lam=lk), K.Side(sv.codes, sv.scales, 4, x=ov, lam=lv)
        dms = timed(lambda: K.srft_kv_dequantize(dk, dv, n, T, H, d, G, T, 0, seed, stream), l2_flush)
        vec = 2 * n * T * H
        vb = 2 * d + d // 2 + 4 * (d // G)
        rel = [float(((o.float() - x.float()) ** 2).sum() / (x.float() ** 2).sum()) for o, x in ((ok, xk), (ov, xv))]
        out[key] = {"workload": w.name, "vectors": vec, "bytes_per_vector": vb,
                    "quant_ms": qms, "quant_vectors_per_s": vec / (qms * 1e-3), "quant_gbs": vec * vb / (qms * 1e-3) / 1e9,
                    "deq_ms": dms, "deq_gbs": vec * vb / (dms * 1e-3) / 1e9,
                    "relative_mse_k_v": rel, "l2_flushed": l2_flush}
        del xk, xv, sk, sv, ok, ov, dk, dv

    w = I.K8V4
    n, T, H, d, G, seed, t_cap = w.n_outer, w.tokens, w.kv_heads, w.d, w.group, w.sign_seed, w.t_cap
    xk, xv = I.kv_side(w, "k", device=dev), I.kv_side(w, "v", device=dev)
    sk = K.alloc_side(n, t_cap, H, d, w.bits_k, G, device=dev)
    sv = K.alloc_side(n, t_cap, H, d, w.bits_v, G, device=dev)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, n, T, H, d, G, t_cap, 0, seed, stream)  # the prebuilt cache
    del xk, xv
    g = torch.Generator(device=dev).manual_seed(404)
    nk = torch.randn((n, 1, H, d), generator=g, device=dev).half()
    nv = torch.randn((n, 1, H, d), generator=g, device=dev).half()
    ak = K.Side(sk.codes, sk.scales, w.bits_k, x=nk)
    av = K.Side(sv.codes, sv.scales, w.bits_v, x=nv)
    ts = []
    for step in range(102):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        K.srft_kv_quantize(ak, av, n, 1, H, d, G, t_cap, T + step % (t_cap - T), seed, stream)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    # the same append captured once in a CUDA graph and replayed: the GPU-side latency without the host's
    # per-call work (argument checks, tensor-map encoding, launch)
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        K.srft_kv_quantize(ak, av, n, 1, H, d, G, t_cap, T, seed, cap)
    torch.cuda.synchronize()
    tg = []
    for _ in range(102):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        tg.append(a.elapsed_time(b))
    del graph
    vb_k, vb_v = 2 * d + d * w.bits_k // 8 + 4 * (d // G), 2 * d + d * w.bits_v // 8 + 4 * (d // G)
    out["k8v4_append"] = {"workload": w.name, "vectors_per_step": 2 * n * H,
                          "bytes_per_step": n * H * (vb_k + vb_v), "append_us_median": statistics.median(ts[2:]) * 1e3,
                          "append_us_min": min(ts[2:]) * 1e3,
                          "append_us_graph_replay_median": statistics.median(tg[2:]) * 1e3}
    del sk, sv, flush
    torch.cuda.empty_cache()
    return out


def run_case(args):
    """One kernel of the path on a cut-down decode workload, for ncu captures."""
    import torch
    import int8_kv_cache_srft_gb300 as K
    from int8_kv_cache_srft_gb300 import inputs as I

    torch.cuda.set_device(0)
    K.library()
    attn = args.kernel.endswith("attention")
    kind = args.kernel.split("_")[-1]
    if args.kernel.startswith("gemma_"):
        w = I.GEMMA
    elif args.kernel == "long_attention":  # long splits: 4 x 131072 tokens, 8 splits per (sequence, kv head)
        w = I.DECODE.resized(n_outer=4)
    elif args.kernel[0] == "d" and args.kernel[1].isdigit():  # d80_, d96_, d192_, d256_ cases
        dk = int(args.kernel[1:].split("_")[0])
        w = I.DECODE.resized(n_outer=4, tokens=32768, d=dk) if attn else I.DECODE.resized(n_outer=2, d=dk)
    else:
        w = I.DECODE.resized(n_outer=4, tokens=32768) if attn else I.DECODE.resized(n_outer=2)
    B, Hkv, d, T, Hq, G, seed = w.n_outer, w.kv_heads, w.d, w.tokens, w.q_heads, w.group, w.sign_seed
    xk, xv = I.kv_side(w, "k", device="cuda"), I.kv_side(w, "v", device="cuda")
    sk, sv = K.alloc_side(B, T, Hkv, d, 4, G), K.alloc_side(B, T, Hkv, d, 4, G)
    sk.x, sv.x = xk, xv
    K.srft_kv_quantize(sk, sv, B, T, Hkv, d, G, T, 0, seed)
    if kind == "quantize":
        def launch():
            K.srft_kv_quantize(sk, sv, B, T, Hkv, d, G, T, 0, seed)
    elif kind == "dequantize":
        dk, dv = torch.empty_like(xk), torch.empty_like(xv)
        deq_k, deq_v = K.Side(sk.codes, sk.scales, 4, x=dk), K.Side(sv.codes, sv.scales, 4, x=dv)

        def launch():
            K.srft_kv_dequantize(deq_k, deq_v, B, T, Hkv, d, G, T, 0, seed)
    else:
        del xk, xv
        sk.x = sv.x = None
        q = I.query(w, device="cuda")
        out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
        ns = 8 if args.kernel == "long_attention" else 0
        ws = torch.empty(K.q4kv_decode_attention_workspace_size(B, Hq, Hkv, d, T, ns), dtype=torch.uint8,
                         device="cuda")

        def launch():
            K.q4kv_decode_attention(q, out, sk, sv, B, Hq, Hkv, d, G, T, None, 0.0, seed, ns, ws)
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    assert K.srftkv_device_fault() == 0
    print(json.dumps({"profile_case": args.kernel, "B": B, "T": T, "kv_heads": Hkv, "d": d, "bits": 4, "group": G,
                      "launches": args.steps, "median_ms": statistics.median(ts)}), flush=True)


def main():
    args = parse()
    if args.kernel is not None:
        run_case(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
