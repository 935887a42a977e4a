#!/usr/bin/env python3
"""Benchmark of the NVFP4 batched decode GEMV on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload headline|attn_qkv|o_proj|fused_qkv|mid_m|decode_step|ffn_verify|moe_decode]
                    [--n TOKENS] [--tiling one_pass|greedy_321] [--variant auto|fp4|tc|mma|simt|generic]
    python bench.py --policy-sweep            # tile-policy table: variant x tiling x n, us/call
    python bench.py --profile-case attn_qkv:1,16 [--reps 1]   # a few launches for ncu
    python bench.py --profile-case headline   # one launch of every headline call (ncu traffic)
    python bench.py --profile-quantize bf16   # the device quantizer, for ncu

Prints ONE JSON line (rank 0).  A step is one pass of the hot path over one
batch of every headline configuration: attention qkv (N=14336, K=5120) at
n = 1, 2, 3, 4, 8 and 16 decode tokens, output projection (N=5120, K=6144)
at n = 8 with 1 % x20 outlier activations, and the fused projection
(N=16384, K=5120) at n = 16 -- eight calls, each on its own rotated weight
copy (16 copies per shape, so every call streams its weights from HBM, not
from the 129 MB L2).  `value` is the whole-job algorithmic HBM throughput
(packed weights + scales + activations, GB/s) of the step; `per_call` gives
every configuration's us/call, GB/s, fraction of the measured HBM peak, ncu
DRAM traffic and, for qkv, the ratio to n = 1.  Steps are replayed from CUDA
graphs and timed with CUDA events on the launching stream.  After timing,
sampled outputs of the last timed step are checked against the CPU oracle
(exit status 1 on a mismatch).

`--impl reference` times the CPU oracle (oracle/, test infrastructure) on the
host cores on a bounded sample of the same workload, in the same metric.
With torchrun (--gpus N > 1) every rank runs an independent replica (the
GEMV has no exchange step); rank 0 prints the max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import multiprocessing as mp
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "NVFP4 batched GEMV µs/call & HBM GB/s (frac of GB300 peak), n=1–16"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
COPIES = 16
L2_BYTES = 129 * 2 ** 20
TOL = 1e-2

SHAPES = {"attn_qkv": (14336, 5120), "o_proj": (5120, 6144), "fused_qkv": (16384, 5120),
          # dense SwiGLU verify FFN, hidden 5120, intermediate 17408: gate/up rows interleaved, then down
          "ffn_gu": (2 * 17408, 5120), "ffn_down": (5120, 17408),
          # one routed expert of an MoE layer (hidden 2048, expert intermediate 768): gate/up, down
          "moe_gu": (2 * 768, 2048), "moe_down": (2048, 768)}
OUTLIER = {"attn_qkv": 0.0, "o_proj": 0.01, "fused_qkv": 0.0, "ffn_gu": 0.0, "ffn_down": 0.0, "moe_gu": 0.0,
           "moe_down": 0.0}
HEADLINE = [("attn_qkv", n) for n in (1, 2, 3, 4, 8, 16)] + [("o_proj", 8), ("fused_qkv", 16)]
MOE_EXPERTS, MOE_TOPK = 128, 8
KERNEL_NAMES = {"fp4": "gemv_fp4_kernel (+ fp4_xprep_kernel)", "tc": "gemv_tc_kernel (+ tc_reduce_kernel)",
                "mma": "gemv_stream_kernel<mma>", "simt": "gemv_stream_kernel<simt>",
                "generic": "gemv_generic_kernel", "moe": "moe_mma_kernel (gate/up + down)"}


def workload_calls(name: str, n_sweep: int):
    if name == "headline":
        return list(HEADLINE)
    if name == "attn_qkv":
        return [("attn_qkv", n) for n in (1, 2, 3, 4)]
    if name == "o_proj":
        return [("o_proj", 8)]
    if name == "fused_qkv":
        return [("fused_qkv", 16)]
    if name == "mid_m":  # verify / prefill widths: one call of n tokens (n = 17..64)
        return [("attn_qkv", n_sweep)]
    if name == "decode_step":
        return [(s, n_sweep) for _ in range(16) for s in ("attn_qkv", "o_proj")]
    if name == "ffn_verify":
        return [("ffn_gu", n_sweep), ("ffn_down", n_sweep)]
    if name == "moe_decode":  # for the CPU sample: one expert's gate/up and down per assignment
        return [("moe_gu", 1), ("moe_down", 1)]
    raise SystemExit(f"unknown workload {name}")


def workload_desc(name: str, n: int) -> str:
    return {
        "headline": "every headline call once per step: attention qkv N=14336 K=5120 at n=1,2,3,4,8,16; "
                    "output projection N=5120 K=6144 at n=8 (activations with 1% x20 outliers); "
                    "fused projection N=16384 K=5120 at n=16",
        "attn_qkv": "attention qkv projection N=14336 K=5120, n=1,2,3,4 (one call each per step)",
        "o_proj": "output projection N=5120 K=6144, n=8, activations with 1% x20 outliers",
        "fused_qkv": "fused projection N=16384 K=5120, n=16",
        "mid_m": f"attention qkv projection N=14336 K=5120, n={n} (mid-M: one read of W per 32 tokens)",
        "decode_step": f"decode step: 16 x (qkv N=14336 K=5120, o_proj N=5120 K=6144), n={n}",
        "ffn_verify": f"dense SwiGLU verify FFN D=5120 F=17408 (gate/up GEMV with fused SwiGLU, then down), n={n}",
        "moe_decode": f"MoE decode, {MOE_EXPERTS} experts D=2048 F=768, top-{MOE_TOPK} of n={n} tokens: "
                      f"grouped read-once gate/up (+SwiGLU) then down",
    }[name]


def call_bytes(shape: str, n: int) -> int:
    """Algorithmic HBM bytes of one call as the headline metric counts them:
    W (K/2 per row) + scales (K/16 per row) + activations (2nK).  The bf16
    outputs (2nN, under 1.2 % of the total at n = 16) are not counted."""
    N, K = SHAPES[shape]
    return N * K // 2 + N * K // 16 + 2 * n * K


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------- ncu DRAM traffic
# variant -> (committed summary, sources its counters depend on)
TRAFFIC_FILES = {
    "fp4": ("traffic_gemv_fp4_headline.md", ("gemv_fp4.cu", "ptx.cuh", "tcgen05.cuh", "internal.h")),
}


def source_hash(names) -> str:
    """sha256 of the named kernel sources' code: comments and blank lines
    removed, so that a comment edit keeps the recorded counters valid."""
    csrc = os.path.join(ROOT, "nvfp4_weight_quantized_gemv_gb300", "csrc")
    h = hashlib.sha256()
    for name in names:
        text = open(os.path.join(csrc, name), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode("utf-8"))
    return h.hexdigest()


def traffic_table(variant: str):
    """{(shape, n): DRAM read+write bytes of one call} from the committed ncu
    summary of the variant's kernels, or {} when there is none or the kernel
    sources changed since its counters were taken."""
    if variant not in TRAFFIC_FILES:
        return {}
    fname, sources = TRAFFIC_FILES[variant]
    try:
        text = open(os.path.join(ROOT, "profiles", fname)).read()
    except OSError:
        return {}
    m = re.search(r"sources_sha256:\s*([0-9a-f]{64})", text)
    if not m or m.group(1) != source_hash(sources):
        return {}
    return {(s, int(n)): int(b) for s, n, b in re.findall(r"traffic_([a-z_]+)_n(\d+):\s*([0-9]+)", text)}


def synth_bf16_weights(torch, N, K, seed, dev):
    """Seeded N(0, 0.02) weights as a bf16 device tensor (host draw, one copy in)."""
    bits = synth.to_bf16_bits(synth.weights_f32(N, K, seed))
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)


# ------------------------------------------------------------ replicas
def max_over_ranks(torch, dist, value, device):
    """The slowest rank's time (all ranks receive it); `value` itself on one process."""
    if dist is None:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, step_bytes, ms_per_step):
    """Whole-job throughput: every rank moved step_bytes per step in the slowest rank's time."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"nvfp4_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]), hw=parts[5],
                                 hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower() in ("active", "1", "yes"):
                    reasons.add(name)
        # samples under load: power above the idle floor
        p_max = max(r["power"] for r in rows)
        loaded = [r for r in rows if r["power"] >= 0.5 * p_max] or rows
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded)}


# ------------------------------------------------------------ CPU oracle
_ORACLE_TASKS = None


def _oracle_init(spec, cores):
    """Pool initializer: draw and quantize (with the oracle) every sampled call's
    rows once per worker, so that the timed maps send only task indices."""
    global _ORACLE_TASKS
    import oracle
    tasks = []
    for N, K, n, outlier, rows, wseed in spec:
        packed, scale, g = oracle.quantize(synth.weights_f32(rows, K, wseed))
        x = synth.activations_bf16(n, K, 1, outlier)
        per = -(-rows // cores)
        for r0 in range(0, rows, per):
            tasks.append((packed[r0:r0 + per].copy(), scale[r0:r0 + per].copy(), g, x))
    _ORACLE_TASKS = tasks


def _oracle_run(task):
    """Task (i, rows): the first `rows` rows of sampled chunk i."""
    import oracle
    i, rows = task
    packed, scale, g, x = _ORACLE_TASKS[i]
    oracle.gemv_rows(packed[:rows], scale[:rows], g, x)
    return i


def cpu_oracle_sample(calls, rows_per_core: int, cores: int, repeats: int = 3, warmup: int = 1,
                      step_budget_s=None):
    """Time the CPU oracle on a bounded sample of one step of the workload.

    For every call of the step, up to `rows_per_core * cores` output rows (all
    of the call's tokens) are computed by the fp64 oracle, split over `cores`
    spawned processes that hold the sampled inputs already.  `warmup` untimed
    passes, then `repeats` timed ones.  With `step_budget_s`, the timed passes
    compute only as many rows of each chunk as the last warm-up pass says fit
    in that budget.  Returns (GB/s of the sampled algorithmic bytes at the
    median wall time, median wall seconds, all wall seconds, description)."""
    import oracle
    oracle.build()
    spec = []
    for ci, (shape, n) in enumerate(calls):
        N, K = SHAPES[shape]
        spec.append((N, K, n, OUTLIER[shape], min(N, rows_per_core * cores), 1000 + ci))
    chunks = []  # (call index, rows of the chunk)
    for ci, (N, K, n, _, rows, _) in enumerate(spec):
        per = -(-rows // cores)
        chunks += [(ci, min(per, rows - r0)) for r0 in range(0, rows, per)]

    def step_bytes(cap):
        nb = 0
        for ci, (N, K, n, _, _, _) in enumerate(spec):
            r = sum(min(cap, c) for cj, c in chunks if cj == ci)
            nb += r * (K // 2 + K // 16) + 2 * n * K
        return nb

    ctx = mp.get_context("spawn")
    walls = []
    full = max(c for _, c in chunks)
    with ctx.Pool(cores, initializer=_oracle_init, initargs=(spec, cores)) as pool:
        cap = full
        for w in range(max(1, warmup)):  # untimed; the first also waits for every initializer
            t0 = time.perf_counter()
            pool.map(_oracle_run, [(i, cap) for i in range(len(chunks))], chunksize=1)
            t_warm = time.perf_counter() - t0
            if w < 2 and step_budget_s is not None:  # the first two full passes size the sample
                cap_next = max(1, min(full, int(full * step_budget_s / max(t_warm, 1e-6))))
                cap = full if w == 0 else cap_next
                if w == 0 and warmup == 1:
                    cap = cap_next
        tasks = [(i, cap) for i in range(len(chunks))]
        for _ in range(repeats):
            t0 = time.perf_counter()
            pool.map(_oracle_run, tasks, chunksize=1)
            walls.append(time.perf_counter() - t0)
    wall = statistics.median(walls)
    rows_step = sum(min(cap, c) for _, c in chunks) // max(1, len(calls))
    names = ", ".join(f"{s} n={n}" for s, n in calls[:8]) + ("..." if len(calls) > 8 else "")
    sample = (f"{rows_step} output rows (all tokens) of each of the {len(calls)} calls of one step "
              f"({names}); fp64 oracle over {cores} spawned processes holding the inputs; median of {repeats} "
              f"timed repeats after {max(1, warmup)} untimed; GB/s of the sampled rows' weight+scale+activation "
              f"bytes")
    return step_bytes(cap) / wall / 1e9, wall, walls, sample


# --------------------------------------------------- oracle check of outputs
def sample_points(n, N, count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = np.concatenate([[0, 1, 127, 128, N - 129, N - 128, N - 1], rng.integers(0, N, count)])
    return rng.integers(0, n, rows.shape[0]), rows


def check_outputs(torch, checks):
    """Compare sampled outputs of the last timed step with the CPU oracle.

    checks: list of (label, packed, scale, g, x_bits, shift, y_device): the
    call's weights are the host matrix with rows rolled by `shift` (copy c of
    a shape), so output row r is the oracle's row (r - shift) mod N."""
    import oracle
    oracle.build()
    total, worst = 0, 0.0
    failed = []
    for label, packed, scale, g, x, shift, y in checks:
        n, N = y.shape
        toks, rows = sample_points(n, N, 64, 7 + total)
        ref, _ = oracle.gemv_points(packed, scale, g, x, toks, (rows - shift) % N)
        got = y.view(torch.int16).cpu().view(torch.bfloat16).double().numpy()[toks, rows]
        ratio = np.abs(got - ref) / (TOL * (np.abs(ref) + 1.0))
        worst = max(worst, float(np.nanmax(ratio)) if np.all(np.isfinite(got)) else float("inf"))
        if not np.all(ratio <= 1.0):
            failed.append(label)
        total += rows.shape[0]
    return {"points": total, "calls": len(checks), "worst_err_over_tol": round(worst, 4),
            "tolerance": "|y - y_oracle| <= 1e-2 (|y_oracle| + 1)", "ok": not failed, "failed": failed}


# ----------------------------------------------------------------- MoE decode
def run_moe(args, torch, nv, rank, world, local_rank, wl_desc, cores):
    """One MoE layer's expert FFN for n decode tokens: grouped gate/up with fused
    SwiGLU over the routed assignments, then grouped down; each active expert is
    read once per step.  `value` = GB/s of the active experts' weights + X."""
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream()
    E, k, n = MOE_EXPERTS, MOE_TOPK, args.n
    (Ngu, D), (Dd, F) = SHAPES["moe_gu"], SHAPES["moe_down"]

    # expert weights: one host draw per matrix kind, quantized by the library's
    # host quantizer, E copies with rows rolled (distinct per expert)
    def stack(N, K, seed):
        packed, scale, g = nv.nvfp4_quantize_ref(synth.weights_f32(N, K, seed))
        wp0, ws0 = torch.from_numpy(packed).to(dev), torch.from_numpy(scale).to(dev)
        wp = torch.stack([torch.roll(wp0, shifts=e * 37, dims=0) for e in range(E)]).contiguous()
        ws = torch.stack([torch.roll(ws0, shifts=e * 37, dims=0) for e in range(E)]).contiguous()
        return wp, ws, torch.full((E,), g, dtype=torch.float32, device=dev)
    gu, down = stack(Ngu, D, 300), stack(Dd, F, 301)
    # R seeded routings (distinct experts per token, sorted by expert), rotated per step
    R = 8
    rng = np.random.Generator(np.random.PCG64(7))
    routes, active = [], []
    for _ in range(R):
        choice = np.stack([rng.choice(E, size=k, replace=False) for _ in range(n)])  # [n][k]
        pairs = sorted((int(e), t) for t in range(n) for e in choice[t])
        off = np.zeros(E + 1, dtype=np.int32)
        for e, _ in pairs:
            off[e + 1] += 1
        off = np.cumsum(off).astype(np.int32)
        tok = np.array([t for _, t in pairs], dtype=np.int32)
        routes.append((torch.from_numpy(off).to(dev), torch.from_numpy(tok).to(dev)))
        active.append(int((np.diff(off) > 0).sum()))
    A = n * k
    ident = torch.arange(A, dtype=torch.int32, device=dev)
    x_host = torch.from_numpy(synth.activations_bf16(n, D, 1).view(np.int16)).view(torch.bfloat16).pin_memory()
    x = x_host.to(dev)
    h = torch.empty((A, F), dtype=torch.bfloat16, device=dev)
    y = torch.empty((A, D), dtype=torch.bfloat16, device=dev)
    y_host = torch.empty((A, D), dtype=torch.bfloat16).pin_memory()
    exp_bytes = Ngu * D // 2 + Ngu * D // 16 + Dd * F // 2 + Dd * F // 16
    step_bytes = [a * exp_bytes + 2 * n * D for a in active]  # active experts read once + X

    def step(i, st):
        off, tok = routes[i % R]
        nv.nvfp4_moe_gemv_grouped(gu[0], gu[1], gu[2], x, off, tok, y=h, swiglu=True, stream=st)
        # down: h rows are already one per assignment, grouped by expert
        nv.nvfp4_moe_gemv_grouped(down[0], down[1], down[2], h, off, ident, y=y, stream=st)

    with torch.cuda.stream(stream):
        step(0, stream)
    stream.synchronize()
    graphs = []
    for i in range(R):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            step(i, stream)
        graphs.append(gph)
    cycle = torch.cuda.CUDAGraph()  # the R routings' steps chained in one graph launch
    with torch.cuda.graph(cycle, stream=stream):
        for i in range(R):
            step(i, stream)

    def replay_steps(k):
        for _ in range(k // R):
            cycle.replay()
        for j in range(k % R):
            graphs[j].replay()

    with torch.cuda.stream(stream):
        replay_steps(-(-args.warmup // R) * R)
    stream.synchronize()
    if nv.nvfp4_device_error(stream) != 0:
        raise SystemExit("device error during warm-up")
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        replay_steps(args.steps)
        ev1.record(stream)
    ev1.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(torch, dist, ms, dev)
    if nv.nvfp4_device_error(stream) != 0:
        raise SystemExit("device error during the timed region")
    ms_per_step = ms / args.steps
    # the timed steps' own bytes: whole cycles of the R routings, then the first steps % R
    timed_bytes = (args.steps // R) * sum(step_bytes) + sum(step_bytes[:args.steps % R])
    mean_bytes = timed_bytes / args.steps
    value = whole_job_gbs(world, mean_bytes, ms_per_step)
    # end to end: X in from pinned host memory, Y out, every step
    e2e_steps = max(20, min(2000, args.steps // 10))
    with torch.cuda.stream(stream):
        for i in range(3):
            x.copy_(x_host, non_blocking=True)
            step(i, stream)
            y_host.copy_(y, non_blocking=True)
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(e2e_steps):
            x.copy_(x_host, non_blocking=True)
            step(i, stream)
            y_host.copy_(y, non_blocking=True)
        b.record(stream)
    b.synchronize()
    e2e_ms = max_over_ranks(torch, dist, a.elapsed_time(b) / e2e_steps, dev)
    hbm_peak, peak_kind = peaks()
    achieved = mean_bytes / (ms_per_step * 1e-3) / 1e9
    if dist is not None:
        dist.barrier()
        if rank != 0:
            dist.destroy_process_group()
            return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        gbs, wall, walls, sample = cpu_oracle_sample(workload_calls("moe_decode", n), args.cpu_rows, cores)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
               "repeat_walls_s": [round(w, 3) for w in walls]}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16*f16+f32 (nvfp4 weights, bf16 activations)",
        "data": "synthetic (seeded PCG64: expert W~N(0,0.02) quantized to NVFP4, X~N(0,1) bf16, random top-k routing)",
        "config": {"workload": wl_desc, "experts": E, "top_k": k, "tokens": n, "assignments": A,
                   "active_experts_mean": round(sum(active) / R, 2), "routings_rotated": R,
                   "per_token_bytes_if_not_grouped": A * exp_bytes,
                   "l2": "active expert weights per step above L2; routings rotated", "parallelism": f"replicas x{world}"},
        "per_call": {f"moe_step_n{n}": {"us_per_call": round(ms_per_step * 1e3, 3), "GB_s": round(achieved, 1),
                                        "frac_of_measured_hbm": round(achieved / hbm_peak, 4)}},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": None,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": KERNEL_NAMES["moe"], "algorithmic_bytes_per_step": round(mean_bytes),
                     "traffic_note": "null: no ncu counters of the current expert kernel in this run's summaries"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * mean_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": y_host.numel() * 2,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# -------------------------------------------------------------- helpers
VARIANT_ARG = {"auto": 0, "mma": 1, "simt": 2, "generic": 3, "tc": 4, "fp4": 5}


def launches_of(plan_info):
    """Kernel launches of one call under its plan."""
    v, passes = plan_info["variant"], plan_info["passes"]
    if v == "fp4":
        return 2 * passes                               # activation prep + GEMV per pass
    if v == "tc":
        wide = max(plan_info["tile_tokens"]) > 16
        return passes * (3 if wide else 2)              # (X conversion +) GEMV + split-row reduction
    return passes


def make_weights(torch, nv, dev, shape, seed, copies):
    """One host draw of the shape, quantized by the library's host quantizer,
    then `copies` device copies with the rows rolled by 97 * c (copy c)."""
    N, K = SHAPES[shape]
    packed, scale, g = nv.nvfp4_quantize_ref(synth.weights_f32(N, K, seed))
    wp0 = torch.from_numpy(packed).to(dev)
    ws0 = torch.from_numpy(scale).to(dev)
    out = [(torch.roll(wp0, shifts=c * 97, dims=0).contiguous(), torch.roll(ws0, shifts=c * 97, dims=0).contiguous(),
            torch.tensor([g], dtype=torch.float32, device=dev)) for c in range(copies)]
    return out, (packed, scale, g)


def time_graph(torch, stream, enqueue, reps, calls_per_replay):
    """us per call of a captured sequence of calls, replayed `reps` times."""
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=stream):
        enqueue()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g1.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g1.replay()
        b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) * 1e3 / (reps * calls_per_replay)


# -------------------------------------------------------------- ncu cases
def profile_case(args):
    """A few eager calls for ncu: `shape:n1,n2,...` (one weight copy of the
    shape, --reps calls per n, synchronized) or `headline` (each headline call
    once on its own shape's weights)."""
    import torch
    import nvfp4_weight_quantized_gemv_gb300 as nv
    nv.build()
    dev = torch.device("cuda", 0)
    if args.profile_case == "headline":
        cases = list(HEADLINE)
    else:
        shape, ns = args.profile_case.split(":")
        cases = [(shape, int(v)) for v in ns.split(",")]
    weights = {}
    for si, s in enumerate(sorted({s for s, _ in cases})):
        weights[s] = make_weights(torch, nv, dev, s, 100 + si, 1)[0][0]
    variant, tiling = VARIANT_ARG[args.variant], 1 if args.tiling == "one_pass" else 2
    for s, n in cases:
        N, K = SHAPES[s]
        x = torch.from_numpy(synth.activations_bf16(n, K, 1, OUTLIER[s]).view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty((n, N), dtype=torch.bfloat16, device=dev)
        wp, ws, gs = weights[s]
        times = []
        for _ in range(args.reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            nv.nvfp4_gemv_batched_ex(wp, ws, gs, x, y, variant=variant, tiling=tiling)
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
        plan = nv.nvfp4_gemv_plan(n, N, K, variant=variant, tiling=tiling)
        print(f"{s} N={N} K={K} n={n} variant={plan['variant']}: {np.mean(times):.2f} us/call "
              f"(mean of {args.reps}, eager, synchronized)")
    if nv.nvfp4_device_error() != 0:
        raise SystemExit("device error")


def profile_quantize(args):
    import torch
    import nvfp4_weight_quantized_gemv_gb300 as nv
    nv.build()
    N, K = SHAPES["attn_qkv"]
    w32 = synth.weights_f32(N, K, 100)
    if args.profile_quantize == "bf16":
        w = torch.from_numpy(synth.to_bf16_bits(w32).view(np.int16)).cuda().view(torch.bfloat16)
    else:
        w = torch.from_numpy(w32).cuda()
    times = []
    for _ in range(args.reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        nv.nvfp4_quantize(w)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    print(f"quantize {args.profile_quantize} N={N} K={K}: {np.mean(times):.2f} us/call (mean of {args.reps})")
    if nv.nvfp4_device_error() != 0:
        raise SystemExit("device error")


# ------------------------------------------------------------ policy sweep
def policy_sweep(args):
    """us/call of every (variant, tiling) the policy layer chooses between, for
    the decode-step shapes at n = 1, 4, 8, 16: each timed over 16 rotated
    weight copies from a CUDA graph.  One JSON line per case, then a summary
    line with AUTO's choices."""
    import torch
    import nvfp4_weight_quantized_gemv_gb300 as nv
    nv.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream()
    hbm_peak, _ = peaks()
    arms = [("fp4", "one_pass"), ("fp4", "greedy_321"), ("tc", "one_pass"), ("tc", "greedy_321"),
            ("mma", "one_pass"), ("simt", "one_pass"), ("mma", "greedy_321")]
    shapes = args.sweep_shapes.split(",")
    ns = [int(v) for v in args.sweep_ns.split(",")]
    rows = []
    for si, s in enumerate(shapes):
        N, K = SHAPES[s]
        copies, _ = make_weights(torch, nv, dev, s, 100 + si, COPIES)
        for n in ns:
            x = torch.from_numpy(synth.activations_bf16(n, K, 1, OUTLIER[s]).view(np.int16)).to(dev).view(
                torch.bfloat16)
            y = torch.empty((n, N), dtype=torch.bfloat16, device=dev)
            for variant, tiling in arms:
                v, t = VARIANT_ARG[variant], 1 if tiling == "one_pass" else 2
                plan = nv.nvfp4_gemv_plan(n, N, K, variant=v, tiling=t)

                def enqueue():
                    for wp, ws, gs in copies:
                        nv.nvfp4_gemv_batched_ex(wp, ws, gs, x, y, stream=stream, variant=v, tiling=t)
                with torch.cuda.stream(stream):
                    enqueue()
                stream.synchronize()
                us = time_graph(torch, stream, enqueue, args.sweep_reps, len(copies))
                gbs = call_bytes(s, n) / (us * 1e-6) / 1e9
                row = {"shape": s, "N": N, "K": K, "n": n, "variant": variant, "tiling": tiling,
                       "passes": plan["passes"], "us_per_call": round(us, 3), "GB_s": round(gbs, 1),
                       "frac_of_measured_hbm": round(gbs / hbm_peak, 4)}
                rows.append(row)
                print(json.dumps(row), flush=True)
            auto = nv.nvfp4_gemv_plan(n, N, K)
            best = min((r for r in rows if r["shape"] == s and r["n"] == n), key=lambda r: r["us_per_call"])
            print(json.dumps({"shape": s, "n": n, "auto": [auto["variant"], auto["tiling"]],
                              "fastest": [best["variant"], best["tiling"]], "fastest_us": best["us_per_call"]}),
                  flush=True)
        del copies
        torch.cuda.empty_cache()
    if nv.nvfp4_device_error(stream) != 0:
        raise SystemExit("device error during the sweep")


# ------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="headline",
                    choices=["headline", "attn_qkv", "o_proj", "fused_qkv", "mid_m", "decode_step", "ffn_verify",
                             "moe_decode"])
    ap.add_argument("--n", type=int, default=8,
                    help="tokens per call for --workload mid_m / decode_step / ffn_verify / moe_decode")
    ap.add_argument("--tiling", default="one_pass", choices=["one_pass", "greedy_321"])
    ap.add_argument("--variant", default="auto", choices=list(VARIANT_ARG))
    ap.add_argument("--cpu-rows", type=int, default=96, help="oracle sample rows per host core and call")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", default=None, help="'shape:n1,n2' or 'headline': eager calls for ncu")
    ap.add_argument("--profile-quantize", default=None, choices=["bf16", "fp32"])
    ap.add_argument("--reps", type=int, default=1, help="calls per n for --profile-case / --profile-quantize")
    ap.add_argument("--policy-sweep", action="store_true")
    ap.add_argument("--sweep-shapes", default="attn_qkv,o_proj")
    ap.add_argument("--sweep-ns", default="1,4,8,16")
    ap.add_argument("--sweep-reps", type=int, default=100)
    args = ap.parse_args()
    if args.profile_case:
        return profile_case(args)
    if args.profile_quantize:
        return profile_quantize(args)
    if args.policy_sweep:
        return policy_sweep(args)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    calls = workload_calls(args.workload, args.n)
    step_bytes = sum(call_bytes(s, n) for s, n in calls)
    cores = os.cpu_count() or 1
    wl_desc = workload_desc(args.workload, args.n)
    is_ffn = args.workload == "ffn_verify"
    # the CPU sample: one qkv and one o_proj call of the decode step
    cpu_calls = calls[:2] if args.workload == "decode_step" else calls

    # ---------------------------------------------------- reference arm
    if args.impl == "reference":
        if rank != 0:
            return
        # exactly --warmup untimed and --steps timed steps, each a bounded
        # sample of the step (rows per chunk sized from the last warm-up step
        # so that the timed steps take about half a minute in all)
        budget = min(0.3, max(0.002, 30.0 / max(1, args.steps)))
        gbs, wall, walls, sample = cpu_oracle_sample(cpu_calls, args.cpu_rows, cores, repeats=args.steps,
                                                     warmup=args.warmup, step_budget_s=budget)
        line = {"metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded PCG64: W~N(0,0.02) quantized to NVFP4, X~N(0,1) bf16)",
                "config": {"workload": wl_desc, "tiling": "per token (each output computed on its own)",
                           "sample_per_step": sample},
                "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                 "sample": sample,
                                 "step_walls_s": {"min": round(min(walls), 4), "median": round(wall, 4),
                                                  "max": round(max(walls), 4)}},
                "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line), flush=True)
        return

    # ------------------------------------------------------------ our arm
    import torch
    import nvfp4_weight_quantized_gemv_gb300 as nv

    nv.build()
    if args.workload == "moe_decode":
        return run_moe(args, torch, nv, rank, world, local_rank, wl_desc, cores)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream()
    variant = VARIANT_ARG[args.variant]
    tiling = nv.TILING_ONE_PASS if args.tiling == "one_pass" else nv.TILING_GREEDY_321

    # weights: COPIES rotated device copies per shape (4 for the 150 MB FFN matrices)
    shapes_used = sorted({s for s, _ in calls})
    weights, host_w = {}, {}
    for si, s in enumerate(shapes_used):
        weights[s], host_w[s] = make_weights(torch, nv, dev, s, 100 + si, 4 if is_ffn else COPIES)
    # every distinct call's X and Y live in one pinned host buffer and one device
    # buffer each (views per call), so that an end-to-end step moves its inputs
    # in with one copy and its outputs out with one
    keys = list(dict.fromkeys(calls))
    x_host_all = torch.empty(sum(n * SHAPES[s][1] for s, n in keys), dtype=torch.bfloat16).pin_memory()
    y_host_all = torch.empty(sum(n * SHAPES[s][0] for s, n in keys), dtype=torch.bfloat16).pin_memory()
    x_dev_all = torch.empty_like(x_host_all, device=dev)
    y_dev_all = torch.empty_like(y_host_all, device=dev)
    xs, ys, xs_host, ys_host, x_bits = {}, {}, {}, {}, {}
    xo = yo = 0
    for s, n in keys:
        N, K = SHAPES[s]
        x_bits[(s, n)] = synth.activations_bf16(n, K, 1, OUTLIER[s])
        xs_host[(s, n)] = x_host_all[xo:xo + n * K].view(n, K)
        xs_host[(s, n)].copy_(torch.from_numpy(x_bits[(s, n)].view(np.int16)).view(torch.bfloat16).view(n, K))
        xs[(s, n)] = x_dev_all[xo:xo + n * K].view(n, K)
        ys_host[(s, n)] = y_host_all[yo:yo + n * N].view(n, N)
        ys[(s, n)] = y_dev_all[yo:yo + n * N].view(n, N)
        xo += n * K
        yo += n * N
    x_dev_all.copy_(x_host_all)

    # Phase p of the step cycle uses, for the j-th call of shape s in the step,
    # weight copy (p * calls_of[s] + j) mod copies: consecutive phases never
    # share a copy, and a copy comes back only after more than L2's bytes.
    calls_of = {s: sum(1 for c, _ in calls if c == s) for s in shapes_used}
    ncopies = min(len(w) for w in weights.values())
    phases = max(1, ncopies // max(calls_of.values()))

    def copy_index(s, j, p):
        return (p * calls_of[s] + j) % len(weights[s])

    h_ffn = torch.empty((args.n, SHAPES["ffn_down"][1]), dtype=torch.bfloat16, device=dev) if is_ffn else None

    def ffn_call(c, x, y, st):
        nv.nvfp4_ffn_swiglu(weights["ffn_gu"][c], weights["ffn_down"][c], x, h=h_ffn, y=y, stream=st)

    def enqueue_step(st, p):
        if is_ffn:
            ffn_call(p % len(weights["ffn_gu"]), xs[calls[0]], ys[calls[1]], st)
            return
        seen = {s: 0 for s in shapes_used}
        for s, n in calls:
            wp, ws, gs = weights[s][copy_index(s, seen[s], p)]
            seen[s] += 1
            nv.nvfp4_gemv_batched_ex(wp, ws, gs, xs[(s, n)], ys[(s, n)], stream=st, variant=variant, tiling=tiling)

    # The end-to-end leg calls the C ABI entry point itself (nvfp4_gemv_batched,
    # the call a C or C++ user makes) with the pointers marshalled once.
    abi = nv.lib()
    abi_args = []
    for p in range(phases):
        seen = {s: 0 for s in shapes_used}
        step_args = []
        for s, n in calls:
            wp, ws, gs = weights[s][copy_index(s, seen[s], p)]
            seen[s] += 1
            N, K = SHAPES[s]
            step_args.append((wp.data_ptr(), ws.data_ptr(), gs.data_ptr(), xs[(s, n)].data_ptr(),
                              ys[(s, n)].data_ptr(), n, N, K, ctypes.c_void_p(stream.cuda_stream)))
        abi_args.append(step_args)

    # warm the library (workspace for this stream, descriptors) outside capture
    with torch.cuda.stream(stream):
        enqueue_step(stream, 0)
    stream.synchronize()
    graphs = []
    for p in range(phases):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            enqueue_step(stream, p)
        graphs.append(gph)
    # all phases in one graph, as a served decode step captures all its layers:
    # consecutive steps then chain inside one graph launch
    cycle = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cycle, stream=stream):
        for p in range(phases):
            enqueue_step(stream, p)

    def replay_steps(k):
        # exactly k steps: whole cycles, then the first k % phases phases
        for _ in range(k // phases):
            cycle.replay()
        for j in range(k % phases):
            graphs[j].replay()

    if is_ffn:
        plans = [nv.nvfp4_gemv_plan(args.n, *SHAPES["ffn_gu"]), nv.nvfp4_gemv_plan(args.n, *SHAPES["ffn_down"])]
    else:
        plans = [nv.nvfp4_gemv_plan(n, *SHAPES[s], variant=variant, tiling=tiling) for s, n in calls]
    launches_per_step = sum(launches_of(pl) for pl in plans)
    main_variant = plans[0]["variant"]

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # warm-up (whole cycles, so the timed region starts at phase 0 on fresh weight copies)
    with torch.cuda.stream(stream):
        replay_steps(-(-args.warmup // phases) * phases)
    stream.synchronize()
    if nv.nvfp4_device_error(stream) != 0:
        raise SystemExit("device error during warm-up")

    # clocks are sampled over the timed steps and the per-call timings after them
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        replay_steps(args.steps)
        ev1.record(stream)
    ev1.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(torch, dist, ms, dev)
    ms_per_step = ms / args.steps
    value = whole_job_gbs(world, step_bytes, ms_per_step)
    if nv.nvfp4_device_error(stream) != 0:
        raise SystemExit("device error during the timed region")

    # the last timed step's outputs against the oracle (sampled points per call)
    check = None
    if not is_ffn and rank == 0:
        last_p = (args.steps - 1) % phases
        seen = {s: 0 for s in shapes_used}
        items, done = [], set()
        for s, n in calls:
            c = copy_index(s, seen[s], last_p)
            seen[s] += 1
            if (s, n) in done:      # a repeated call (decode step): its buffer holds the last one
                items = [it for it in items if it[0] != f"{s}_n{n}"]
            done.add((s, n))
            packed, scale, g = host_w[s]
            items.append((f"{s}_n{n}", packed, scale, g, x_bits[(s, n)], c * 97, ys[(s, n)]))
        check = check_outputs(torch, items)

    # per-call breakdown: each distinct call alone, over the shape's weight copies
    per_call = {}
    hbm_peak, peak_kind = peaks()
    traffic = traffic_table(main_variant) if variant in (0, 5) and tiling == nv.TILING_ONE_PASS else {}
    if is_ffn:  # the FFN is one library call: time it alone over its weight copies
        n = args.n

        def enqueue_ffn():
            for c in range(len(weights["ffn_gu"])):
                ffn_call(c, xs[calls[0]], ys[calls[1]], stream)
        us = time_graph(torch, stream, enqueue_ffn, 200, len(weights["ffn_gu"]))
        per_call[f"ffn_n{n}"] = {"us_per_call": round(us, 3), "GB_s": round(step_bytes / (us * 1e-6) / 1e9, 1),
                                 "launches": launches_per_step}
    for ci, (s, n) in enumerate([] if is_ffn else dict.fromkeys(calls)):
        def enqueue_one(s=s, n=n):
            for wp, ws, gs in weights[s]:
                nv.nvfp4_gemv_batched_ex(wp, ws, gs, xs[(s, n)], ys[(s, n)], stream=stream, variant=variant,
                                         tiling=tiling)
        reps = max(20, min(400, 40000 // len(weights[s])))
        us = time_graph(torch, stream, enqueue_one, reps, len(weights[s]))
        nbytes = call_bytes(s, n)
        gbs = nbytes / (us * 1e-6) / 1e9
        pl = nv.nvfp4_gemv_plan(n, *SHAPES[s], variant=variant, tiling=tiling)
        tr = traffic.get((s, n))
        per_call[f"{s}_n{n}"] = {
            "us_per_call": round(us, 3), "GB_s": round(gbs, 1), "algorithmic_bytes": nbytes,
            "traffic": tr, "traffic_over_algorithmic": round(tr / nbytes, 4) if tr else None,
            "variant": pl["variant"], "passes": pl["passes"], "launches": launches_of(pl)}
    for v in per_call.values():
        v["frac_of_measured_hbm"] = round(v["GB_s"] / hbm_peak, 4)
        v["frac_of_8TBs"] = round(v["GB_s"] / NOMINAL_HBM_GBS, 4)
    if "attn_qkv_n1" in per_call:
        base = per_call["attn_qkv_n1"]["us_per_call"]
        for key, v in per_call.items():
            if key.startswith("attn_qkv_"):
                v["ratio_to_n1"] = round(v["us_per_call"] / base, 3)
    clk = clocks.stop()
    if nv.nvfp4_device_error(stream) != 0:
        raise SystemExit("device error during the per-call timings")

    # device requantization of bf16 weights to NVFP4 (amax pass + block pass),
    # two weight copies alternating so that no call finds its input in L2
    quant = None
    if args.workload in ("headline", "attn_qkv", "fused_qkv"):
        N, K = SHAPES["attn_qkv"]
        wq = [synth_bf16_weights(torch, N, K, 200 + c, dev) for c in range(2)]
        qp = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
        qs = torch.empty((N, K // 16), dtype=torch.uint8, device=dev)
        qg = torch.empty(1, dtype=torch.float32, device=dev)
        reps = 40
        with torch.cuda.stream(stream):
            for c in range(4):
                nv._quantize_into(wq[c % 2], qp, qs, qg, stream)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for c in range(reps):
                nv._quantize_into(wq[c % 2], qp, qs, qg, stream)
            b.record(stream)
        b.synchronize()
        if nv.nvfp4_device_error(stream) != 0:
            raise SystemExit("device error in the quantizer")
        us = a.elapsed_time(b) * 1e3 / reps
        qbytes = N * K * 2 + N * K // 2 + N * K // 16  # read W once, write codes and scales
        quant = {"shape": f"N={N} K={K} bf16 -> nvfp4", "us_per_call": round(us, 2),
                 "algorithmic_bytes": qbytes, "GB_s": round(qbytes / (us * 1e-6) / 1e9, 1),
                 "frac_of_measured_hbm": round(qbytes / (us * 1e-6) / 1e9 / hbm_peak, 4),
                 "launches_per_call": 3, "note": "two passes over W by design (amax, then blocks)"}
        del wq

    # end to end through the C ABI with host buffers: every step copies the
    # activations in from pinned host memory, makes the C-ABI calls
    # (nvfp4_gemv_batched, un-captured) and copies the outputs back out
    e2e_steps = max(20, min(2000, args.steps // 10))
    if is_ffn:  # x goes in, y comes out (h stays on the device)
        h2d, d2h = xs_host[calls[0]].numel() * 2, ys_host[calls[1]].numel() * 2
    else:       # every distinct call's X in with one copy, every Y out with one
        h2d, d2h = x_host_all.numel() * 2, y_host_all.numel() * 2

    def e2e_step(i):
        if is_ffn:
            xs[calls[0]].copy_(xs_host[calls[0]], non_blocking=True)
            ffn_call(i % len(weights["ffn_gu"]), xs[calls[0]], ys[calls[1]], stream)
            ys_host[calls[1]].copy_(ys[calls[1]], non_blocking=True)
            return
        x_dev_all.copy_(x_host_all, non_blocking=True)
        for args in abi_args[i % phases]:
            st_ = abi.nvfp4_gemv_batched(*args)
            if st_ != nv.NVFP4_OK:
                raise SystemExit(f"nvfp4_gemv_batched: {nv.nvfp4_last_error()}")
        y_host_all.copy_(y_dev_all, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
        stream.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_host = time.perf_counter()
        a.record(stream)
        for i in range(e2e_steps):
            e2e_step(i)
        b.record(stream)
        host_s = time.perf_counter() - t_host
    b.synchronize()
    e2e_ms = a.elapsed_time(b) / e2e_steps
    e2e_ms = max_over_ranks(torch, dist, e2e_ms, dev)
    e2e_value = whole_job_gbs(world, step_bytes, e2e_ms)
    host_us_per_call = host_s * 1e6 / (e2e_steps * len(calls))

    achieved = step_bytes / (ms_per_step * 1e-3) / 1e9  # per GPU: algorithmic bytes per step / step time
    step_traffic = None
    if traffic and all((s, n) in traffic for s, n in calls):
        step_traffic = sum(traffic[(s, n)] for s, n in calls)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": step_traffic,
                "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "frac_of_8TBs": round(achieved / NOMINAL_HBM_GBS, 4),
                "kernel": KERNEL_NAMES.get(main_variant, main_variant),
                "algorithmic_bytes_per_step": step_bytes,
                "timing": "CUDA events around the timed steps on the launching stream (all of a step's launches)",
                "traffic_note": ("ncu dram read+write bytes of one cold launch of each call, summed over the step "
                                 f"(profiles/{TRAFFIC_FILES[main_variant][0]})" if step_traffic else
                                 "null: no ncu counters of the current kernel sources for every call of this step")}

    if dist is not None:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        gbs, wall, walls, sample = cpu_oracle_sample(cpu_calls, args.cpu_rows, cores)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
               "repeat_walls_s": [round(w, 3) for w in walls]}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e2m1 x e2m1 (block-scaled MMA) + f32: nvfp4 weights, bf16 activations as 8 NVFP4 terms"
                  if main_variant == "fp4" else "f16*f16+f32 (nvfp4 weights, bf16 activations)"),
        "data": "synthetic (seeded PCG64: W~N(0,0.02) quantized to NVFP4, X~N(0,1) bf16)",
        "config": {"workload": wl_desc, "tiling": args.tiling, "variant": main_variant,
                   "weight_copies": ncopies, "graph_phases": phases,
                   "l2": "inputs larger than L2: weight copies rotated, no copy reused within a step or the next",
                   "grid": plans[0]["num_ctas"], "stages": plans[0]["stages"], "parallelism": f"replicas x{world}"},
        "per_call": per_call,
        "oracle_check": check,
        "quantize": quant,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "host_us_per_call": round(host_us_per_call, 2),
                "how": "per step: one H2D copy of every call's X from pinned memory, the C-ABI calls "
                       "nvfp4_gemv_batched (un-captured, default options), one D2H copy of every Y; CUDA events on "
                       "the stream; host_us_per_call = host time to enqueue a call"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    if check is not None and not check["ok"]:
        sys.stderr.write(f"oracle check failed for {check['failed']}\n")
        raise SystemExit(1)


if __name__ == "__main__":
    main()
