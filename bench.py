#!/usr/bin/env python3
"""Benchmark of the NVFP4 batched decode GEMV on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload attn_qkv|o_proj|fused_qkv|mid_m|decode_step|ffn_verify|moe_decode] [--tiling one_pass|greedy_321]

Prints ONE JSON line (rank 0).  A step is one pass of the hot path over one
batch: for the default workload (attention qkv projection, N=14336, K=5120)
that is four calls, n = 1, 2, 3 and 4 decode tokens, each on its own weight
copy.  Sixteen rotated weight copies (661 MB) keep the working set above the
129 MB L2, so every call streams its weights from HBM.  `value` is the
whole-job algorithmic HBM throughput (packed weights + scales + activations,
GB/s); per-n µs/call are reported beside it.  Steps are replayed from CUDA
graphs and timed with CUDA events on the launching stream.

`--impl reference` times the CPU oracle (oracle/, test infrastructure) on the
host cores on a bounded sample of the same workload, in the same metric.
With torchrun (--gpus N > 1) every rank runs an independent replica (the
GEMV has no exchange step); rank 0 prints the max-over-ranks timing.
"""
from __future__ import annotations

import argparse
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

# workload -> list of (shape name, n) calls per step
SHAPES = {"attn_qkv": (14336, 5120), "o_proj": (5120, 6144), "fused_qkv": (16384, 5120),
          # dense SwiGLU verify FFN, hidden 5120, intermediate 17408: gate/up rows interleaved, then down
          "ffn_gu": (2 * 17408, 5120), "ffn_down": (5120, 17408),
          # one routed expert of an MoE layer (hidden 2048, expert intermediate 768): gate/up, down
          "moe_gu": (2 * 768, 2048), "moe_down": (2048, 768)}
OUTLIER = {"attn_qkv": 0.0, "o_proj": 0.01, "fused_qkv": 0.0, "ffn_gu": 0.0, "ffn_down": 0.0, "moe_gu": 0.0,
           "moe_down": 0.0}
MOE_EXPERTS, MOE_TOPK = 128, 8


def workload_calls(name: str, n_sweep: int):
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


def call_bytes(shape: str, n: int) -> int:
    """Algorithmic HBM bytes of one call: W (K/2 per row) + scales (K/16 per row) + X (2nK)."""
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


# variant -> (kernel source, committed ncu summary, kernel name)
KERNELS = {
    "tc": ("gemv_tc.cu", "gemv_tc_attn_qkv.md", "gemv_tc_kernel"),
    "moe": ("moe_mma.cu", "moe_mma_moe_decode.md", "moe_mma_kernel"),
    "mma": ("gemv_stream.cu", "gemv_stream_mma_attn_qkv.md", "gemv_stream_kernel<mma>"),
    "simt": ("gemv_stream.cu", "gemv_stream_simt_attn_qkv.md", "gemv_stream_kernel<simt>"),
    "generic": ("gemv_generic.cu", "gemv_generic_attn_qkv.md", "gemv_generic_kernel"),
}


def kernel_traffic(variant):
    """Per-launch DRAM bytes of the variant's kernel from the committed ncu summary,
    if the kernel source is unchanged since those counters were taken."""
    src_name, prof_name, _ = KERNELS[variant]
    csrc = os.path.join(ROOT, "nvfp4_weight_quantized_gemv_gb300", "csrc")
    prof = os.path.join(ROOT, "profiles", prof_name)
    try:
        text = open(prof).read()
        # every source hash the summary records must match the current file
        checks = {"source_sha256": src_name, "ptx_sha256": "ptx.cuh", "tcgen05_sha256": "tcgen05.cuh"}
        for key, name in checks.items():
            m = re.search(key + r":\s*([0-9a-f]{64})", text)
            if key == "source_sha256" and not m:
                return None, None
            if m and m.group(1) != hashlib.sha256(open(os.path.join(csrc, name), "rb").read()).hexdigest():
                return None, None
    except OSError:
        return None, None
    m_tr = re.search(r"dram_bytes_per_(?:launch|step)_n(\d+):\s*([0-9]+)", text)
    if not m_tr:
        return None, None
    return int(m_tr.group(2)), int(m_tr.group(1))


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
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), hw=parts[5], hwt=parts[6], swt=parts[7],
                                 pcap=parts[8]))
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
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------ CPU oracle
def _oracle_task(args):
    packed, scale, g, x = args
    import oracle
    oracle.gemv_rows(packed, scale, g, x)
    return packed.shape[0]


def cpu_oracle_sample(calls, rows_per_core: int, cores: int, steps: int = 1):
    """Time the CPU oracle on a bounded sample of one step of the workload.

    For every call of the step, `rows_per_core * cores` output rows (all of the
    call's tokens) are computed by the fp64 oracle, split over `cores` spawned
    processes.  Inputs are drawn and quantized (by the oracle) in this process
    before timing.  Returns (GB/s of the sampled algorithmic bytes, wall seconds
    per step, description)."""
    import oracle
    oracle.build()
    tasks, nbytes = [], 0
    for ci, (shape, n) in enumerate(calls):
        N, K = SHAPES[shape]
        rows = min(N, rows_per_core * cores)
        packed, scale, g = oracle.quantize(synth.weights_f32(rows, K, 1000 + ci))
        x = synth.activations_bf16(n, K, 1, OUTLIER[shape])
        per = -(-rows // cores)
        for r0 in range(0, rows, per):
            r1 = min(rows, r0 + per)
            tasks.append((packed[r0:r1].copy(), scale[r0:r1].copy(), g, x))
        nbytes += rows * (K // 2 + K // 16) + 2 * n * K
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        pool.map(_oracle_task, [(t[0][:1], t[1][:1], t[2], t[3]) for t in tasks[:cores]])  # warm workers
        t0 = time.perf_counter()
        for _ in range(steps):
            pool.map(_oracle_task, tasks, chunksize=1)
        wall = (time.perf_counter() - t0) / steps
    sample = (f"{rows_per_core * cores} output rows (all tokens) of each of the {len(calls)} calls of one step "
              f"({', '.join(f'{s} n={n}' for s, n in calls[:4])}{'...' if len(calls) > 4 else ''}); fp64 oracle "
              f"over {cores} spawned processes; GB/s of the sampled rows' weight+scale+activation bytes")
    return nbytes / wall / 1e9, wall, sample


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
    mean_bytes = sum(step_bytes) / R

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
            x.copy_(x_host, non_blocking=True); step(i, stream); y_host.copy_(y, non_blocking=True)
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
        gbs, wall, sample = cpu_oracle_sample(workload_calls("moe_decode", n), args.cpu_rows, cores)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    # ncu DRAM bytes of one step (both launches) from the committed summary, for n = 16 only
    moe_traffic, moe_traffic_note = None, "null: no ncu counters for this kernel source and n"
    tr, tr_n = kernel_traffic("moe")
    if tr is not None and tr_n == n:
        moe_traffic = tr
        moe_traffic_note = (f"ncu dram read+write bytes of one captured step (gate/up + down) at n={n}; "
                            "steps differ in their active experts")
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
                     "frac": round(achieved / hbm_peak, 4), "traffic": moe_traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": "moe_mma_kernel (gate/up + down)", "algorithmic_bytes_per_step": round(mean_bytes),
                     "traffic_note": moe_traffic_note},
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


# ------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="attn_qkv",
                    choices=["attn_qkv", "o_proj", "fused_qkv", "mid_m", "decode_step", "ffn_verify", "moe_decode"])
    ap.add_argument("--n", type=int, default=8,
                    help="tokens per call for --workload mid_m / decode_step / ffn_verify / moe_decode")
    ap.add_argument("--tiling", default="one_pass", choices=["one_pass", "greedy_321"])
    ap.add_argument("--variant", default="auto", choices=["auto", "mma", "simt", "generic"])
    ap.add_argument("--cpu-rows", type=int, default=96, help="oracle sample rows per host core and call")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    calls = workload_calls(args.workload, args.n)
    step_bytes = sum(call_bytes(s, n) for s, n in calls)
    cores = os.cpu_count() or 1
    wl_desc = {
        "attn_qkv": "attention qkv projection N=14336 K=5120, n=1,2,3,4 (one call each per step)",
        "o_proj": "output projection N=5120 K=6144, n=8, activations with 1% x20 outliers",
        "fused_qkv": "fused projection N=16384 K=5120, n=16",
        "mid_m": f"attention qkv projection N=14336 K=5120, n={args.n} (mid-M: one read of W per 32 tokens)",
        "decode_step": f"decode step: 16 x (qkv N=14336 K=5120, o_proj N=5120 K=6144), n={args.n}",
        "ffn_verify": f"dense SwiGLU verify FFN D=5120 F=17408 (gate/up GEMV with fused SwiGLU, then down), "
                      f"n={args.n}",
        "moe_decode": f"MoE decode, {MOE_EXPERTS} experts D=2048 F=768, top-{MOE_TOPK} of n={args.n} tokens: "
                      f"grouped read-once gate/up (+SwiGLU) then down",
    }[args.workload]
    is_ffn = args.workload == "ffn_verify"

    # ---------------------------------------------------- reference arm
    if args.impl == "reference":
        if rank != 0:
            return
        # each step is a bounded sample (cpu_rows rows per core of every call);
        # the run is capped at 5 timed steps so it ends within a few minutes
        steps_run = max(1, min(args.steps, 5))
        cpu_oracle_sample(calls, max(1, args.cpu_rows // 8), cores, steps=1)  # warm-up sample
        gbs, wall, sample = cpu_oracle_sample(calls, args.cpu_rows, cores, steps=steps_run)
        line = {"metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
                "steps": steps_run, "warmup": 1, "ms_per_step": round(wall * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded PCG64: W~N(0,0.02) quantized to NVFP4, X~N(0,1) bf16)",
                "config": {"workload": wl_desc, "tiling": "per token (each output computed on its own)",
                           "sample_per_step": sample},
                "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                 "sample": sample},
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
    variant = {"auto": nv.VARIANT_AUTO, "mma": nv.VARIANT_MMA, "simt": nv.VARIANT_SIMT,
               "generic": nv.VARIANT_GENERIC}[args.variant]
    tiling = nv.TILING_ONE_PASS if args.tiling == "one_pass" else nv.TILING_GREEDY_321

    # weights: one host draw per shape, quantized by the library's host
    # quantizer, then COPIES distinct device copies (rows rolled per copy)
    shapes_used = sorted({s for s, _ in calls})
    weights = {}
    for si, s in enumerate(shapes_used):
        N, K = SHAPES[s]
        packed, scale, g = nv.nvfp4_quantize_ref(synth.weights_f32(N, K, 100 + si))
        wp0 = torch.from_numpy(packed).to(dev)
        ws0 = torch.from_numpy(scale).to(dev)
        ncopies = 4 if is_ffn else COPIES  # ffn: 4 x 150 MB of weights, well above L2
        copies = []
        for c in range(ncopies):
            copies.append((torch.roll(wp0, shifts=c * 97, dims=0).contiguous(),
                           torch.roll(ws0, shifts=c * 97, dims=0).contiguous(),
                           torch.tensor([g], dtype=torch.float32, device=dev)))
        weights[s] = copies
        del wp0, ws0
    # every distinct call's X and Y live in one pinned host buffer and one device
    # buffer each (views per call), so that an end-to-end step moves its inputs
    # in with one copy and its outputs out with one
    keys = list(dict.fromkeys(calls))
    x_len = {(s, n): n * SHAPES[s][1] for s, n in keys}
    y_len = {(s, n): n * SHAPES[s][0] for s, n in keys}
    x_host_all = torch.empty(sum(x_len.values()), dtype=torch.bfloat16).pin_memory()
    y_host_all = torch.empty(sum(y_len.values()), dtype=torch.bfloat16).pin_memory()
    x_dev_all = torch.empty_like(x_host_all, device=dev)
    y_dev_all = torch.empty_like(y_host_all, device=dev)
    xs, ys, xs_host, ys_host = {}, {}, {}, {}
    xo = yo = 0
    for s, n in keys:
        N, K = SHAPES[s]
        xh = synth.activations_bf16(n, K, 1, OUTLIER[s])
        xs_host[(s, n)] = x_host_all[xo:xo + n * K].view(n, K)
        xs_host[(s, n)].copy_(torch.from_numpy(xh.view(np.int16)).view(torch.bfloat16).view(n, K))
        xs[(s, n)] = x_dev_all[xo:xo + n * K].view(n, K)
        ys_host[(s, n)] = y_host_all[yo:yo + n * N].view(n, N)
        ys[(s, n)] = y_dev_all[yo:yo + n * N].view(n, N)
        xo += n * K
        yo += n * N
    x_dev_all.copy_(x_host_all)

    # Step p (p = 0..P-1) uses weight copies rotating so that consecutive
    # calls never reuse a copy within 16 calls of each other.
    counters = {s: 0 for s in shapes_used}

    h_ffn = torch.empty((args.n, SHAPES["ffn_down"][1]), dtype=torch.bfloat16, device=dev) if is_ffn else None

    def ffn_call(c, x, y, st):
        nv.nvfp4_ffn_swiglu(weights["ffn_gu"][c], weights["ffn_down"][c], x, h=h_ffn, y=y, stream=st)

    def enqueue_step(st):
        if is_ffn:
            c = counters["ffn_gu"] % len(weights["ffn_gu"])
            counters["ffn_gu"] += 1
            ffn_call(c, xs[calls[0]], ys[calls[1]], st)
            return
        for s, n in calls:
            wp, ws, gs = weights[s][counters[s] % len(weights[s])]
            counters[s] += 1
            nv.nvfp4_gemv_batched_ex(wp, ws, gs, xs[(s, n)], ys[(s, n)], stream=st, variant=variant, tiling=tiling)

    # warm the library (workspace for this stream, descriptors) outside capture
    with torch.cuda.stream(stream):
        enqueue_step(stream)
    stream.synchronize()
    per_step_calls = len(calls)
    phases = max(1, min(16, max(len(w) for w in weights.values()) // max(1, per_step_calls)))
    graphs = []
    for _ in range(phases):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            enqueue_step(stream)
        graphs.append(gph)
    # all phases in one graph, as a served decode step captures all its layers:
    # consecutive steps then chain inside one graph launch
    cycle = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cycle, stream=stream):
        for _ in range(phases):
            enqueue_step(stream)

    def replay_steps(k):
        # exactly k steps: whole cycles, then the first k % phases phases
        for _ in range(k // phases):
            cycle.replay()
        for j in range(k % phases):
            graphs[j].replay()

    plan = nv.nvfp4_gemv_plan(calls[-1][1], *SHAPES[calls[-1][0]], variant=variant, tiling=tiling)
    def launches(plan_info):
        # tcgen05 path: GEMV and split-row reduction per pass, plus the X
        # conversion when a pass stages 32 tokens (n > 16)
        if plan_info["variant"] != "tc":
            return plan_info["passes"]
        wide = max(plan_info["tile_tokens"]) > 16
        return plan_info["passes"] * (3 if wide else 2)

    launches_per_step = sum(launches(nv.nvfp4_gemv_plan(n, *SHAPES[s], variant=variant, tiling=tiling))
                            for s, n in calls)

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
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(torch, dist, ms, dev)
    ms_per_step = ms / args.steps
    value = whole_job_gbs(world, step_bytes, ms_per_step)
    if nv.nvfp4_device_error(stream) != 0:
        raise SystemExit("device error during the timed region")

    # per-call breakdown (each call shape timed alone, back-to-back graph replays)
    per_call = {}
    if is_ffn:  # the FFN is one library call: time it alone over its weight copies
        n = args.n
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            for c in range(len(weights["ffn_gu"])):
                ffn_call(c, xs[calls[0]], ys[calls[1]], stream)
        reps = 200
        with torch.cuda.stream(stream):
            for _ in range(3):
                g1.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g1.replay()
            b.record(stream)
        b.synchronize()
        us = a.elapsed_time(b) * 1e3 / (reps * len(weights["ffn_gu"]))
        per_call[f"ffn_n{n}"] = {"us_per_call": round(us, 3), "GB_s": round(step_bytes / (us * 1e-6) / 1e9, 1)}
    for s, n in ([] if is_ffn else dict.fromkeys(calls)):
        key = f"{s}_n{n}"
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            for c in range(len(weights[s])):
                wp, ws, gs = weights[s][c]
                nv.nvfp4_gemv_batched_ex(wp, ws, gs, xs[(s, n)], ys[(s, n)], stream=stream, variant=variant,
                                         tiling=tiling)
        reps = max(20, min(400, 40000 // len(weights[s])))
        with torch.cuda.stream(stream):
            for _ in range(3):
                g1.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g1.replay()
            b.record(stream)
        b.synchronize()
        us = a.elapsed_time(b) * 1e3 / (reps * len(weights[s]))
        gbs = call_bytes(s, n) / (us * 1e-6) / 1e9
        per_call[key] = {"us_per_call": round(us, 3), "GB_s": round(gbs, 1)}
    hbm_peak, peak_kind = peaks()
    for v in per_call.values():
        v["frac_of_measured_hbm"] = round(v["GB_s"] / hbm_peak, 4)
        v["frac_of_8TBs"] = round(v["GB_s"] / NOMINAL_HBM_GBS, 4)
    if args.workload == "attn_qkv":
        base = per_call["attn_qkv_n1"]["us_per_call"]
        for v in per_call.values():
            v["ratio_to_n1"] = round(v["us_per_call"] / base, 3)

    # device requantization of bf16 weights to NVFP4 (amax pass + block pass),
    # two weight copies alternating so that no call finds its input in L2
    quant = None
    if args.workload in ("attn_qkv", "fused_qkv"):
        N, K = SHAPES[calls[0][0]]
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
        hbm_peak_q, _ = peaks()
        quant = {"shape": f"N={N} K={K} bf16 -> nvfp4", "us_per_call": round(us, 2),
                 "algorithmic_bytes": qbytes, "GB_s": round(qbytes / (us * 1e-6) / 1e9, 1),
                 "frac_of_measured_hbm": round(qbytes / (us * 1e-6) / 1e9 / hbm_peak_q, 4),
                 "launches_per_call": 3, "note": "two passes over W by design (amax, then blocks)"}
        del wq

    # end to end through the public API with host buffers: every step copies
    # the activations in from pinned host memory and the outputs back out
    e2e_steps = max(20, min(2000, args.steps // 20))
    if is_ffn:  # x goes in, y comes out (h stays on the device)
        h2d, d2h = xs_host[calls[0]].numel() * 2, ys_host[calls[1]].numel() * 2
    else:       # every distinct call's X in with one copy, every Y out with one
        h2d, d2h = x_host_all.numel() * 2, y_host_all.numel() * 2

    def e2e_step():
        if is_ffn:
            c = counters["ffn_gu"] % len(weights["ffn_gu"])
            counters["ffn_gu"] += 1
            xs[calls[0]].copy_(xs_host[calls[0]], non_blocking=True)
            ffn_call(c, xs[calls[0]], ys[calls[1]], stream)
            ys_host[calls[1]].copy_(ys[calls[1]], non_blocking=True)
            return
        x_dev_all.copy_(x_host_all, non_blocking=True)
        for s, n in calls:
            wp, ws, gs = weights[s][counters[s] % len(weights[s])]
            counters[s] += 1
            nv.nvfp4_gemv_batched(wp, ws, gs, xs[(s, n)], ys[(s, n)], stream=stream)
        y_host_all.copy_(y_dev_all, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        stream.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
    b.synchronize()
    e2e_ms = a.elapsed_time(b) / e2e_steps
    e2e_ms = max_over_ranks(torch, dist, e2e_ms, dev)
    e2e_value = whole_job_gbs(world, step_bytes, e2e_ms)

    # the recorded counters are of the attention qkv shape (N=14336, K=5120): other shapes report none
    qkv_only = args.workload == "attn_qkv"
    traffic, traffic_n = kernel_traffic(plan["variant"]) if qkv_only else (None, None)
    achieved = step_bytes / (ms_per_step * 1e-3) / 1e9  # per GPU: algorithmic bytes per launch / launch time
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "frac_of_8TBs": round(achieved / NOMINAL_HBM_GBS, 4),
                "kernel": KERNELS[plan["variant"]][2],
                "algorithmic_bytes_per_step": step_bytes,
                "traffic_note": (f"ncu dram read+write bytes per launch at n={traffic_n} (attention qkv shape)"
                                 if traffic else
                                 "null: the recorded ncu counters cover the attention qkv shape only" if not qkv_only
                                 else "null: no ncu counters for the current kernel source")}

    if dist is not None:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        gbs, wall, sample = cpu_oracle_sample(calls if args.workload != "decode_step" else calls[:2],
                                              args.cpu_rows, cores)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16*f16+f32 (nvfp4 weights, bf16 activations)",
        "data": "synthetic (seeded PCG64: W~N(0,0.02) quantized to NVFP4, X~N(0,1) bf16)",
        "config": {"workload": wl_desc, "tiling": args.tiling, "variant": plan["variant"],
                   "weight_copies": len(weights[calls[0][0]]),
                   "l2": "inputs larger than L2: weight copies rotated, no copy reused within 16 calls",
                   "grid": plan["num_ctas"], "stages": plan["stages"], "parallelism": f"replicas x{world}"},
        "per_call": per_call,
        "quantize": quant,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
