#!/usr/bin/env python
"""Benchmark of the blockwise-scaled FP8 grouped GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1] [--impl ours|reference]

One step is one grouped GEMM over the workload (default: config 1, the grouped MoE
blockwise FP8 problem with 8 experts, 4096 token rows by uniform routing, N=4096,
K=7168).  Inputs are seeded synthetic data generated on the host and copied to HBM
before the timed region.  W untimed warm-up steps are followed by exactly K timed steps,
each bracketed by CUDA events on the launching stream; L2 is flushed (a 512 MiB write)
between steps, outside the events.  Rank 0 prints one JSON line.

With --gpus N > 1 (launched by torchrun) every rank runs an independent replica of the
workload on its own GPU (weak scaling; the GEMM has no exchange step), and the step time
is the max over ranks.

--impl reference times the CPU oracle (the plain C++ statement of the method) on a
bounded sample of the same workload, on this machine's host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped blockwise-FP8 GEMM TFLOP/s and % of GB300 FP8 tensor peak (1 GPU)"
FP8_PER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor throughput ratio (4.5 / 2.25 PFLOP/s)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The sources each workload's kernel is built from: a committed ncu summary is used for
# `traffic` only while these are byte-identical to the ones it was captured on.
_COMMON_SOURCES = ("ptx.cuh", "sched.cuh", "common.cuh", "tmem_plan.cuh")
KERNEL_SOURCES = {
    "blockwise": _COMMON_SOURCES + ("bsfp8_grouped.cu",),
    "mx_swap": _COMMON_SOURCES + ("bsmxfp8_grouped.cu",),
    "mx_pair": _COMMON_SOURCES + ("bsmxfp8_pair.cu",),
}
WORKLOAD_KERNEL = {"config0": "blockwise", "config1": "blockwise", "config2": "blockwise",
                   "config3": "blockwise", "config4": "mx_swap", "config5": "mx_pair",
                   "fp4:mxfp8xmxfp4": "mx_swap", "fp4:mxfp4xmxfp4": "mx_swap",
                   "fp4:nvfp4xnvfp4": "mx_swap"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# host helpers
# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def strip_comments(src: str) -> str:
    """C/C++ source without comments and blank lines (string literals kept whole), so that
    the kernel hash changes with the code and not with its commentary."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = ("".join(out)).splitlines()
    return "\n".join(ln.rstrip() for ln in lines if ln.strip())


def kernel_hash(workload_key: str = "config1", sources=None) -> str:
    """First 12 hex digits of the SHA-256 over the sources of this workload's kernel, comments
    removed (sources: optional {file name: text} to hash instead of the files on disk)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_fp8_persistent_gb300", "csrc")
    for name in KERNEL_SOURCES[WORKLOAD_KERNEL[workload_key]]:
        if sources is not None:
            text = sources.get(name)
        else:
            p = os.path.join(csrc, name)
            text = open(p, encoding="utf-8").read() if os.path.exists(p) else None
        if text is not None:
            h.update(name.encode() + b"\0" + strip_comments(text).encode())
    return h.hexdigest()[:12]


def traffic_from_profiles(workload_key: str):
    """DRAM bytes per launch from the committed ncu summary of this workload, if it was
    captured on the current kernel sources (else None)."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None, None
    want = kernel_hash(workload_key)
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".txt"):
            continue
        text = open(os.path.join(pdir, name)).read()
        key = f"workload_key: {workload_key}\n"
        if key not in text:
            continue
        # the workload's own section: from its key to the next workload's key
        sect = text[text.index(key) + len(key):].split("workload_key:")[0]
        m_hash = re.search(r"kernel_sources_sha256_12: ([0-9a-f]+)", text)
        m_bytes = re.search(r"dram_bytes_per_launch: ([0-9.eE+]+)", sect)
        if m_hash and m_bytes and m_hash.group(1) == want:
            return float(m_bytes.group(1)), name
    return None, None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        busy = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] if power else []
        return {"sm_mhz": statistics.median(busy or sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# distributed (replicas only: barrier + max of step time)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def aggregate(dist, local_ms: float, local_flops: float):
    """(max step ms over ranks, total flops over ranks)."""
    if dist is None:
        return local_ms, local_flops
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    f = torch.tensor([local_flops], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(f, op=dist.ReduceOp.SUM)
    return float(t.item()), float(f.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle timing (bounded sample)
# ---------------------------------------------------------------------------
def oracle_rows_for(p, seconds: float):
    import oracle
    dt1, _, _ = oracle.timed_rows(p, 8)
    per_row = max(dt1 / 8, 1e-6)
    return int(max(1, min(p.M_total, seconds / per_row)))


def oracle_sample(p, rows: int):
    import oracle
    dt, flops, th = oracle.timed_rows(p, rows)
    return dt, flops, th


def sample_parity(got_bits, ref_bits, T) -> dict:
    """The GPU's C against the oracle on the rows the CPU baseline computed, element by
    element, with the tests' acceptance bound: |C - ref| <= 2 ulp_bf16(ref) + 1e-6 T, where
    ulp_bf16(x) = 2^(max(floor(log2|x|), -126) - 7) and T is the sum of |products| (both
    from the oracle)."""
    import numpy as np
    to_f64 = lambda b: (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(  # noqa: E731
        np.float32).astype(np.float64)
    got, ref = to_f64(got_bits), to_f64(ref_bits)
    a = np.abs(ref)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126), -126)
    bound = 2.0 * np.ldexp(1.0, (e - 7).astype(np.int64)) + 1e-6 * np.asarray(T, np.float64)
    err = np.abs(got - ref)
    return {"elements": int(err.size), "outside_bound": int((~(err <= bound)).sum()),
            "max_err_over_bound": float(np.max(err / bound)) if err.size else 0.0,
            "bit_identical": int((np.asarray(got_bits, np.uint16)
                                  == np.asarray(ref_bits, np.uint16)).sum())}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def workload_descr(cfg: int, p) -> dict:
    import gen
    return {"workload": f"config {cfg}: {gen.CONFIG_NAMES[cfg]}", "experts": p.E,
            "M_total": p.M_total, "N": p.N, "K": p.K, "mode": p.mode,
            "expert_rows": [int(c) for c in p.counts][:16] + (["..."] if p.E > 16 else []),
            "seed": cfg, "l2": "flushed between steps (512 MiB write outside the timed events)",
            "inputs": "seeded synthetic, generated on the host, resident in HBM before timing"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import gen
    p = gen.config_problem(args.config)
    budget = args.ref_budget  # seconds of oracle work for the whole reference run
    rows = oracle_rows_for(p, budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(p, rows)
    times, flops, th = [], 0.0, 1
    for _ in range(args.steps):
        dt, fl, th = oracle_sample(p, rows)
        times.append(dt)
        flops = fl
    ms = 1e3 * statistics.mean(times)
    value = flops / (ms * 1e-3) / 1e12
    sample = (f"{rows} of {p.M_total} rows x all {p.N} columns (K={p.K}) of config {args.config} "
              f"per step; oracle threads {th}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_descr(args.config, p),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_secondary(cfg, args, flush, stream, peaks, peak_src):
    """Time another workload (the other blockwise configs 0, 2, 3, the MXFP8 decode config 4,
    or the dense MXFP8 config 5) with the same protocol: warm-up, then args.steps launches,
    each bracketed by CUDA events, L2 flushed between them.  Config 0 is a launch-latency
    case: its roofline fraction says how far a 0.4 MB problem is from both roofs."""
    import numpy as np
    import torch
    import gen
    import block_scaled_fp8_persistent_gb300 as bsfp8
    dev = flush.device
    p = gen.config_problem(cfg)
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(dev)
         for k in ("A", "B", "a_scales", "b_scales", "offsets")}
    C = torch.empty((p.M_total, p.N), dtype=torch.bfloat16, device=dev)

    def step():
        fn = bsfp8.bsmxfp8_grouped_gemm if p.mode == "mx" else bsfp8.bsfp8_grouped_gemm
        fn(d["A"], d["B"], d["a_scales"], d["b_scales"], d["offsets"], C, p.M_total, p.N, p.K, p.E,
           stream=stream)

    for _ in range(args.warmup):
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    err = bsfp8.bsfp8_get_device_error(stream)
    gbs = p.bytes() / (ms * 1e-3) / 1e9
    tflops = p.flops() / (ms * 1e-3) / 1e12
    traffic, prof_file = traffic_from_profiles(f"config{cfg}")
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    if p.flops() / (fp8_peak * 1e12) >= p.bytes() / (peaks["hbm_gbs"] * 1e9):
        roof = {"bound": "tensor", "achieved": tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": tflops / fp8_peak,
                "peak_source": f"{peak_src} bf16 burst x {FP8_PER_BF16} (nominal fp8/bf16 ratio)"}
    else:
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peak_src} copy bandwidth"}
    roof.update({"traffic": traffic, "algorithmic_bytes": p.bytes()})
    out = {"workload": f"config {cfg}: {gen.CONFIG_NAMES[cfg]}", "M_total": p.M_total,
           "experts": p.E, "N": p.N, "K": p.K, "ms_per_step": ms, "value": tflops,
           "unit": "TFLOP/s", "roofline": roof, "device_error": err, "gpu_launches": args.steps}
    if p.mode == "blockwise":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        out["tile_plan"] = bsfp8.bsfp8_blockwise_plan(p.M_total, p.N, p.E, sms)
    if p.mode == "mx" and cfg == 4:
        # the same decode GEMM on weight scales packed once beforehand (not timed)
        packed = torch.empty_like(d["b_scales"])
        bsfp8.bsmxfp8_pack_b_scales(d["b_scales"], packed, p.E, p.N, p.K, stream=stream)

        def step_packed():
            bsfp8.bsmxfp8_grouped_gemm_prepacked(d["A"], d["B"], d["a_scales"], packed,
                                                 d["offsets"], C, p.M_total, p.N, p.K, p.E,
                                                 stream=stream)

        for _ in range(args.warmup):
            step_packed()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step_packed()
            ends[i].record(stream)
        torch.cuda.synchronize()
        ms_p = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
        gbs_p = p.bytes() / (ms_p * 1e-3) / 1e9
        out["prepacked_b_scales"] = {
            "entry_point": "bsmxfp8_grouped_gemm_prepacked", "ms_per_step": ms_p,
            "achieved_gbs": gbs_p, "frac": gbs_p / peaks["hbm_gbs"],
            "device_error": bsfp8.bsfp8_get_device_error(stream)}
        del packed
    if prof_file:
        out["roofline"]["traffic_source"] = f"profiles/{prof_file}"
    del d, C
    torch.cuda.empty_cache()
    return out


def time_mx_skewed(args, flush, stream, peaks, peak_src):
    """MXFP8 on config 2's routing and shape (64 experts, 16384 token rows by Zipf(1.2),
    N=2048, K=7168): the library's own kernel choice and each forced form (CTA-pair tiles for
    every expert, swap-AB tiles for every expert, and the split by expert size), same
    protocol: the library's choice against each form on skewed routing."""
    import os
    import numpy as np
    import torch
    import gen
    import block_scaled_fp8_persistent_gb300 as bsfp8
    dev = flush.device
    counts = gen.config_counts(2)
    N, K = gen.CONFIG_SHAPES[2]
    p = gen.mx_problem(counts, N, K, seed=2)
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(dev)
         for k in ("A", "B", "a_scales", "b_scales", "offsets")}
    C = torch.empty((p.M_total, N), dtype=torch.bfloat16, device=dev)
    out = {"workload": "MXFP8 on config 2's routing: E=64 M_total=16384 (Zipf 1.2) N=2048 K=7168",
           "experts_with_256_rows_or_more": int(sum(int(c) >= 256 for c in counts)),
           "algorithmic_bytes": p.bytes(), "forms": {}}
    saved = os.environ.get("BSFP8_MX_KERNEL")
    try:
        for form in ("plan", "pair", "swap", "split"):
            if form == "plan":
                os.environ.pop("BSFP8_MX_KERNEL", None)
            else:
                os.environ["BSFP8_MX_KERNEL"] = form

            def step():
                bsfp8.bsmxfp8_grouped_gemm(d["A"], d["B"], d["a_scales"], d["b_scales"],
                                           d["offsets"], C, p.M_total, N, K, p.E, stream=stream)

            for _ in range(args.warmup):
                step()
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            torch.cuda.synchronize()
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize()
            ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
            gbs = p.bytes() / (ms * 1e-3) / 1e9
            out["forms"][form] = {"ms_per_step": ms, "TFLOP/s": p.flops() / (ms * 1e-3) / 1e12,
                                  "achieved_gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
                                  "device_error": bsfp8.bsfp8_get_device_error(stream)}
    finally:
        if saved is None:
            os.environ.pop("BSFP8_MX_KERNEL", None)
        else:
            os.environ["BSFP8_MX_KERNEL"] = saved
    out["hbm_peak_source"] = f"{peak_src} copy bandwidth"
    del d, C
    torch.cuda.empty_cache()
    return out


FP4_PAIRS = (("mxfp8", "mxfp4"), ("mxfp4", "mxfp4"), ("nvfp4", "nvfp4"))


def time_fp4_formats(args, flush, stream, peaks, ref_ms):
    """The decode workload's shape (config 4's routing, N=4096, K=7168) with fp4 operands,
    the format pairs of the block-scaled example (fp4 weights stream half the bytes of e4m3),
    through bsmx_grouped_gemm with the same protocol.  Inputs: random e2m1 codes and scales
    as random_quantized_tensor draws them; mxfp8 tokens as the decode workload draws them."""
    import numpy as np
    import torch
    import gen
    import block_scaled_fp8_persistent_gb300 as bsfp8
    dev = flush.device
    counts = gen.config_counts(4)
    N, K = gen.CONFIG_SHAPES[4]
    out = {"workload": "config 4's routing and shape (E=128 x U{1..32} rows, N=4096, K=7168) "
                       "with fp4 operands", "pairs": {}}
    for af, bf in FP4_PAIRS:
        p = gen.fmt_problem(counts, N, K, seed=4, a_fmt=af, b_fmt=bf, a_recipe="quantized")
        d = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(dev)
             for k in ("A", "B", "a_scales", "b_scales", "offsets")}
        C = torch.empty((p.M_total, N), dtype=torch.bfloat16, device=dev)

        def step():
            bsfp8.bsmx_grouped_gemm(af, bf, d["A"], d["B"], d["a_scales"], d["b_scales"],
                                    d["offsets"], C, p.M_total, N, K, p.E, p.num_experts,
                                    stream=stream)

        for _ in range(args.warmup):
            step()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
        gbs = p.bytes() / (ms * 1e-3) / 1e9
        traffic, prof_file = traffic_from_profiles(f"fp4:{af}x{bf}")
        kinds = os.environ.get("BSFP8_FP4_MMA") != "convert"
        out["pairs"][f"{af} x {bf}"] = {
            "mma": ({"nvfp4": "kind::mxf4nvf4 scale_vec::4X", "mxfp4": "kind::mxf4",
                     "mxfp8": "kind::mxf8f6f4, e2m1 weights loaded padded"}[af]
                    if kinds else "packed fp4 tiles converted on chip"),
            "ms_per_step": ms, "TFLOP/s": p.flops() / (ms * 1e-3) / 1e12,
            "algorithmic_bytes": p.bytes(), "achieved_gbs": gbs,
            "hbm_frac": gbs / peaks["hbm_gbs"], "traffic": traffic,
            "traffic_source": f"profiles/{prof_file}" if prof_file else None,
            "time_vs_mxfp8_decode": (ms / ref_ms) if ref_ms else None,
            "device_error": bsfp8.bsfp8_get_device_error(stream), "gpu_launches": args.steps}
        del d, C
        torch.cuda.empty_cache()
    return out


FP4_PER_BF16 = 6.0  # nominal dense fp4 / bf16 tensor throughput ratio (13.5 / 2.25 PFLOP/s)


def time_fp4_dense(args, flush, stream, peaks):
    """The fp4 format pairs on a dense prefill-sized problem (one expert, M = N = K = 8192, the
    block-scaled example's benchmark shape), through bsmx_grouped_gemm: compute-bound, so
    against the tensor peak of the MMA kind (fp4 kinds twice the fp8 rate; mxfp8 x mxfp4 runs
    kind::mxf8f6f4 at the fp8 rate)."""
    import numpy as np
    import torch
    import gen
    import block_scaled_fp8_persistent_gb300 as bsfp8
    dev = flush.device
    M = N = K = 8192
    out = {"workload": "dense fp4, one expert, M=N=K=8192 (prefill-sized; the plan's CTA-pair "
                       "256x256 tiles on the fp4 kinds)", "pairs": {}}
    for af, bf in FP4_PAIRS:
        p = gen.fmt_problem([M], N, K, seed=5, a_fmt=af, b_fmt=bf)
        d = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).to(dev)
             for k in ("A", "B", "a_scales", "b_scales", "offsets")}
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

        def step():
            bsfp8.bsmx_grouped_gemm(af, bf, d["A"], d["B"], d["a_scales"], d["b_scales"],
                                    d["offsets"], C, M, N, K, 1, 1, stream=stream)

        for _ in range(args.warmup):
            step()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
        tflops = p.flops() / (ms * 1e-3) / 1e12
        ratio = FP8_PER_BF16 if af == "mxfp8" else FP4_PER_BF16
        peak = peaks["bf16_tflops"] * ratio
        out["pairs"][f"{af} x {bf}"] = {
            "ms_per_step": ms, "TFLOP/s": tflops, "peak_tflops": peak,
            "peak_source": f"measured bf16 burst x {ratio} (nominal ratio of the MMA kind)",
            "frac": tflops / peak,
            "device_error": bsfp8.bsfp8_get_device_error(stream), "gpu_launches": args.steps}
        del d, C
        torch.cuda.empty_cache()
    return out


def time_expert_ids(p, d, C, args, flush, stream):
    """The same workload routed through the expert indirection (group g multiplies expert
    perm[g] of the same B, perm a seeded permutation) with the same protocol."""
    import numpy as np
    import torch
    import block_scaled_fp8_persistent_gb300 as bsfp8
    perm = np.random.default_rng(p.E).permutation(p.E).astype(np.int32)
    ids = torch.from_numpy(perm).to(flush.device)
    fn = bsfp8.bsfp8_grouped_gemm_ids if p.mode == "blockwise" else bsfp8.bsmxfp8_grouped_gemm_ids

    def step():
        fn(d["A"], d["B"], d["a_scales"], d["b_scales"], d["offsets"], ids, C, p.M_total, p.N,
           p.K, p.E, p.E, stream=stream)

    for _ in range(args.warmup):
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    return {"workload": "the main workload with group g on expert perm[g] (seeded permutation)",
            "entry_point": fn.__name__, "expert_ids": perm.tolist(), "ms_per_step": ms,
            "value": p.flops() / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "device_error": bsfp8.bsfp8_get_device_error(stream), "gpu_launches": args.steps}


def run_ours(args):
    import numpy as np
    import torch
    import gen
    import block_scaled_fp8_persistent_gb300 as bsfp8
    from block_scaled_fp8_persistent_gb300 import build as libbuild

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (GB300)")
    torch.cuda.set_device(local)
    dist = dist_init(world, "nccl")
    if rank == 0:
        libbuild.build()
    barrier(dist)
    bsfp8.load_library()

    cfg = args.config
    t0 = time.time()
    fmt = tuple(args.fmt.split(":")) if args.fmt else None
    if fmt is not None:
        # fp4 operands on this workload's routing and shape (bsmx_grouped_gemm), for ncu
        if not args.profile:
            raise SystemExit("--fmt is for --profile runs only")
        N = args.n_override or gen.CONFIG_SHAPES[cfg][0]
        p = gen.fmt_problem(gen.config_counts(cfg), N, gen.CONFIG_SHAPES[cfg][1], seed=cfg,
                            a_fmt=fmt[0], b_fmt=fmt[1], a_recipe="quantized")
    elif args.n_override:
        # profiling-sized copy of a workload: same routing, K and kernel, fewer columns
        if not args.profile:
            raise SystemExit("--n-override is for --profile runs only")
        counts = gen.config_counts(cfg)
        make = gen.mx_problem if cfg in (4, 5) else gen.blockwise_problem
        p = make(counts, args.n_override, gen.CONFIG_SHAPES[cfg][1], seed=cfg)
    else:
        p = gen.config_problem(cfg)
    log(f"[bench] rank {rank}: generated config {cfg} in {time.time() - t0:.1f}s "
        f"(M_total={p.M_total}, E={p.E})")
    dev = torch.device("cuda", local)
    host = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).pin_memory()
            for k in ("A", "B", "a_scales", "b_scales", "offsets")}
    d = {k: v.to(dev) for k, v in host.items()}
    C = torch.empty((p.M_total, p.N), dtype=torch.bfloat16, device=dev)
    C_host = torch.empty((p.M_total, p.N), dtype=torch.bfloat16).pin_memory()
    fn = bsfp8.bsfp8_grouped_gemm if p.mode == "blockwise" else bsfp8.bsmxfp8_grouped_gemm
    stream = torch.cuda.current_stream(dev)

    def step():
        if fmt is not None:
            bsfp8.bsmx_grouped_gemm(fmt[0], fmt[1], d["A"], d["B"], d["a_scales"],
                                    d["b_scales"], d["offsets"], C, p.M_total, p.N, p.K, p.E,
                                    p.num_experts, stream=stream)
            return
        fn(d["A"], d["B"], d["a_scales"], d["b_scales"], d["offsets"], C, p.M_total, p.N, p.K,
           p.E, stream=stream)

    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(local)
    if not args.profile:
        sampler.start()
        time.sleep(0.3)
    # warm-up only: a longer run of launches before the timed steps (a soak) holds the clock
    # at the power cap afterwards, and the peak the result is compared with is a burst figure
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if bsfp8.bsfp8_get_device_error(stream) != 0:
        raise SystemExit("device error word set during warm-up")

    # ---- timed region: exactly K steps ----
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    wall0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    wall1 = time.time()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    local_ms = statistics.mean(step_ms)
    dev_err = bsfp8.bsfp8_get_device_error(stream)
    if args.profile:
        if rank == 0:
            print(json.dumps({"profile_run": True, "config": cfg, "step_ms": step_ms,
                              "device_error": dev_err}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return 0

    # ---- end to end through the public call with host buffers ----
    # Every step copies its inputs from pinned host memory and reads its C back; the copies
    # of step i+1 overlap the GEMM and the read-back of step i (two device buffer sets, an
    # upload stream, the GEMM stream and a read-back stream, ordered by events).  Two
    # readings of "the step's inputs": every operand of the GEMM (the headline e2e), and the
    # token side only (A, its scales, the routing offsets) with the expert weights and their
    # scales resident on the device as model parameters (uploaded once, before timing).
    d2h = C.numel() * C.element_size()

    def e2e_run(per_step):
        bufs = [d, {k: (torch.empty_like(v) if k in per_step else v) for k, v in d.items()}]
        outs = [C, torch.empty_like(C)]
        hosts_c = [C_host, torch.empty_like(C_host).pin_memory()]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        loaded = [ev() for _ in range(args.steps)]
        done = [ev() for _ in range(args.steps)]
        read = [ev() for _ in range(args.steps)]
        e2e_start = torch.cuda.Event(enable_timing=True)
        e2e_end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e2e_start.record(up)
        for i in range(args.steps):
            b, o = bufs[i % 2], outs[i % 2]
            if i >= 2:
                up.wait_event(done[i - 2])       # step i-2's GEMM has read this buffer set
            with torch.cuda.stream(up):
                for k in per_step:
                    b[k].copy_(host[k], non_blocking=True)
            loaded[i].record(up)
            stream.wait_event(loaded[i])
            if i >= 2:
                stream.wait_event(read[i - 2])   # step i-2's C has been read back
            fn(b["A"], b["B"], b["a_scales"], b["b_scales"], b["offsets"], o, p.M_total, p.N,
               p.K, p.E, stream=stream)
            done[i].record(stream)
            down.wait_event(done[i])
            with torch.cuda.stream(down):
                hosts_c[i % 2].copy_(o, non_blocking=True)
            read[i].record(down)
        up.wait_stream(down)
        e2e_end.record(up)
        torch.cuda.synchronize()
        ms = e2e_start.elapsed_time(e2e_end) / args.steps
        h2d_bytes = sum(host[k].numel() * host[k].element_size() for k in per_step)
        del bufs, outs
        return ms, h2d_bytes

    e2e_ms_local, h2d = e2e_run(("A", "B", "a_scales", "b_scales", "offsets"))
    e2e_tok_ms_local, h2d_tok = e2e_run(("A", "a_scales", "offsets"))

    flops = p.flops()
    max_ms, total_flops = aggregate(dist, local_ms, flops)
    e2e_ms, _ = aggregate(dist, e2e_ms_local, flops)
    e2e_tok_ms, _ = aggregate(dist, e2e_tok_ms_local, flops)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    value = total_flops / (max_ms * 1e-3) / 1e12
    achieved = flops / (local_ms * 1e-3) / 1e12
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    tensor_bound = p.flops() / (fp8_peak * 1e12) >= p.bytes() / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:
        peak = fp8_peak
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "peak_source": f"{peak_src} bf16 burst {peaks['bf16_tflops']} TFLOP/s x {FP8_PER_BF16} "
                               f"(nominal fp8/bf16 ratio)"}
    else:
        gbs = p.bytes() / (local_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peak_src} copy bandwidth"}
    key = f"config{cfg}"
    traffic, prof_file = traffic_from_profiles(key)
    roof["traffic"] = traffic
    roof["algorithmic_bytes"] = p.bytes()
    roof["algorithmic_flops"] = flops
    if prof_file:
        roof["traffic_source"] = f"profiles/{prof_file}"

    # The timings after the main one each report a failure in their own entry of the line
    # instead of losing the main result (a CUDA error that breaks the context still ends
    # the run: those calls raise again below).
    def guarded(fn, *a):
        try:
            return fn(*a)
        except Exception as exc:  # noqa: BLE001 -- reported in the JSON line
            log(f"[bench] {fn.__name__} failed: {exc!r}")
            return {"error": repr(exc)}

    # ---- the same workload through the expert indirection (group -> expert ids) ----
    routed = None if args.no_secondary else guarded(time_expert_ids, p, d, C, args, flush,
                                                    stream)

    # ---- the second mode of the path: the MXFP8 decode workload, timed the same way ----
    secondary = extra = None
    others = {}
    if not args.no_secondary:
        for c in (3, 2, 0):
            if c != cfg:
                others[f"config{c}"] = guarded(time_secondary, c, args, flush, stream, peaks,
                                               peak_src)
    if not args.no_secondary and cfg != 4:
        secondary = guarded(time_secondary, 4, args, flush, stream, peaks, peak_src)
    if not args.no_secondary and cfg not in (4, 5):
        extra = guarded(time_secondary, 5, args, flush, stream, peaks, peak_src)
    fp4 = None
    if not args.no_secondary:
        ref_ms = secondary.get("ms_per_step") if secondary else None
        fp4 = guarded(time_fp4_formats, args, flush, stream, peaks, ref_ms)
    mx_skewed = None if args.no_secondary else guarded(time_mx_skewed, args, flush, stream,
                                                       peaks, peak_src)
    fp4_dense = None if args.no_secondary else guarded(time_fp4_dense, args, flush, stream,
                                                       peaks)

    clocks = sampler.stop()  # sampled from before the warm-up through the timings above

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        rows = oracle_rows_for(p, args.cpu_seconds)
        dt, fl, th, (rsel, ref, T) = oracle.timed_rows(p, rows, keep=True)
        # the same rows of the GPU's C (the last end-to-end step's read-back of this workload)
        got = C_host.view(torch.int16).numpy().view(np.uint16)[rsel]
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
               "sample": f"{rows} of {p.M_total} rows x all {p.N} columns (K={p.K}), {dt:.1f} s",
               "parity_of_sample": sample_parity(got, ref, T)}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": workload_descr(cfg, p),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": total_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipeline": "inputs of step i+1 uploaded while step i computes and reads back",
                "weights_resident": {
                    "value": total_flops / (e2e_tok_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": e2e_tok_ms, "h2d_bytes_per_step": h2d_tok,
                    "d2h_bytes_per_step": d2h,
                    "reading": "expert weights and their scales uploaded once before timing; "
                               "each step uploads A, its scales and the offsets"}},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms), "max": max(step_ms)},
        "wall_s_timed_region": wall1 - wall0,
        "device_error": dev_err,
        "kernel_sources_sha256_12": kernel_hash(f"config{cfg}"),
    }
    if others:
        line["blockwise_configs"] = others
    if routed is not None:
        line["expert_ids_variant"] = routed
    if secondary is not None:
        line["secondary"] = secondary
    if extra is not None:
        line["extra"] = extra
    if fp4 is not None:
        line["fp4_formats"] = fp4
    if mx_skewed is not None:
        line["mx_skewed_routing"] = mx_skewed
    if fp4_dense is not None:
        line["fp4_dense"] = fp4_dense
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=1, choices=[0, 1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=150.0,
                    help="--impl reference: seconds of oracle work across all steps")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the MXFP8 decode workload that is timed after the main one")
    ap.add_argument("--n-override", type=int, default=0,
                    help="with --profile: run the workload with this many columns N")
    ap.add_argument("--fmt", default="",
                    help="with --profile: operand formats a:b (e.g. mxfp8:mxfp4, nvfp4:nvfp4) "
                         "on the workload's routing and shape")
    ap.add_argument("--profile", action="store_true",
                    help="only warm-up + timed steps (for ncu): no soak, e2e, clocks or CPU baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
