"""Benchmark of the paged GQA decode step on GB300.

Workload (default): Qwen3-0.6B-shaped decode -- 28 layers, each with its own
paged bf16 KV cache of T = 8192 positions (Hkv = 8, D = 128, page size 16,
random block table; 896 MiB of KV in total), B = 1, Hq = 16. One step runs,
for every layer, the prologue (Q/K RMSNorm, RoPE, K/V append) and the
split-KV paged decode attention with its partition merge as one
decode_step_paged launch, all 28 captured in one CUDA graph. Each layer's 32 MiB is read once per step and 27 other layers
are read in between, so the working set (896 MiB) is far larger than L2.

Metric: decode-attention KV GB/s (K+V bytes the attention must read, divided
by the step time) and microseconds per layer-step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (fp64, plain C) on the host cores on a
bounded sample of the same workload. Under torchrun every rank runs an
independent replica (the step does not shard across GPUs) and rank 0 prints
one JSON line.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention KV GB/s (fraction of HBM peak); µs per layer-step at T=8K"
WORKLOAD = "qwen3_0p6b_t8k"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_step_kernel_qwen3_t8k.md")
# GB300's nominal HBM3e bandwidth, reported beside the measured copy peak
NOMINAL_HBM_GBS = 7900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=[WORKLOAD, "ragged_b64", "long_split_kv_t128k", "host_tiled_t64k",
                             "qwen3_0p6b_t8k_m4", "qwen3_0p6b_t8k_int8"],
                    help="the headline step (default) or one of the larger parity workloads, "
                         "measured on their own (one JSON line per variant, not the headline line)")
    ap.add_argument("--ragged-batch", type=int, default=None,
                    help="with --workload ragged_b64: only the first N sequences (a smaller case for captures)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layers per step (default 28); a smaller count is only for profiling captures")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def slowest_rank_ms(ms: float, world: int, device) -> float:
    """The job's time for a timed region: the largest over the ranks (each
    rank times its own replica; collectives only here, never on the data
    path)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: float, world: int, step_s: float) -> float:
    """Whole-job throughput: every rank's bytes of a step over the slowest
    rank's step time (replicas: per-rank work is fixed, weak scaling)."""
    return world * bytes_per_rank_step / step_s / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_gqa_decode_head_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the split kernel from the committed ncu summary,
    only if it was taken on the current kernel sources."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    text = open(PROFILE_SUMMARY).read()
    sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    traffic = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not sha or not traffic or sha.group(1) != kernel_source_sha():
        return None
    return float(traffic.group(1))


def smi_gpu_id(dev) -> str:
    """nvidia-smi identifier (UUID when torch exposes it) of a torch device."""
    import torch

    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        idx = dev.index or 0
        if vis:
            return vis.split(",")[idx].strip()
        return str(idx)


def gpu_idle_check(gpu_id: str) -> dict:
    """Whether the GPU is idle before the benchmark starts: its utilization and
    the compute processes on it other than this one (nvidia-smi)."""
    out = {"util_pct": None, "other_processes": None}
    try:
        util = subprocess.run(["nvidia-smi", "-i", gpu_id, "--query-gpu=utilization.gpu",
                               "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
        apps = subprocess.run(["nvidia-smi", "-i", gpu_id, "--query-compute-apps=pid", "--format=csv,noheader"],
                              capture_output=True, text=True, timeout=20)
    except (OSError, subprocess.TimeoutExpired):
        return out
    try:
        out["util_pct"] = float(util.stdout.strip().splitlines()[0])
    except (ValueError, IndexError):
        pass
    if apps.returncode == 0:
        pids = [ln.strip() for ln in apps.stdout.splitlines() if ln.strip().isdigit()]
        out["other_processes"] = sum(1 for pid in pids if int(pid) != os.getpid())
    return out


class ClockSampler:
    """nvidia-smi clock/throttle samples in the background (200 ms period)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        window = [p for (t, p) in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        if not window:
            window = [p for (_, p) in self.samples]
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in window if num(p[1]) is not None]
        smax = [num(p[2]) for p in window if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in window:
            for name, val in zip(names, p[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(window)}


# ------------------------------------------------------------------ oracle (CPU) leg
def oracle_layer(layer, theta):
    import oracle

    kv, tok = layer
    q_ref, kc, vc = oracle.qk_norm_rope_append(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k, kv.context_lens,
                                               kv.block_table, kv.k_cache, kv.v_cache, kv.page_size, theta)
    oracle.decode_attention(q_ref, kc, vc, kv.block_table, kv.context_lens, 1.0 / math.sqrt(128))


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


def run_oracle_jobs(jobs, threads: int) -> float:
    """Run the callables on `threads` host threads (ctypes releases the GIL);
    returns the wall time in seconds."""
    t0 = time.perf_counter()
    if threads <= 1:
        for fn in jobs:
            fn()
    else:
        with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda fn: fn(), jobs))
    return time.perf_counter() - t0


def oracle_baseline(jobs, single_jobs, unit_bytes, single_bytes, sample: str, single_sample: str) -> dict:
    """The fp64 oracle timed on the host: `jobs` spread over all host cores
    (one thread per job at most) and `single_jobs` on one thread. Returns the
    cpu_baseline record (GB/s of KV the oracle gets through)."""
    import oracle

    oracle.build()
    threads = min(host_cores(), len(jobs))
    s_all = run_oracle_jobs(jobs, threads)
    s_one = run_oracle_jobs(single_jobs, 1)
    return {"value": unit_bytes / s_all / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{sample}, spread over {threads} host threads",
            "single_thread": {"value": single_bytes / s_one / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": single_sample}}


def kv_bytes_layer(T, Hkv=8, D=128):
    return 4 * T * Hkv * D


def headline_config(w, n_layers: int) -> dict:
    """The workload of the headline line, the same for both arms."""
    return {"workload": WORKLOAD, "layers": n_layers, "B": w["B"], "Hq": w["Hq"], "Hkv": w["Hkv"], "D": 128,
            "T": w["T"], "page_size": w["page_size"],
            "l2": "inputs larger than L2: 896 MiB of KV, each layer's 32 MiB read once per step"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from paged_gqa_decode_head_gb300 import inputs

    import oracle

    oracle.build()
    w = inputs.WORKLOADS[WORKLOAD]
    n_layers = args.layers or w["layers"]
    layers = inputs.qwen3_layers(layers=n_layers)
    jobs = [lambda lay=lay: oracle_layer(lay, w["theta"]) for lay in layers]
    threads = min(host_cores(), len(jobs))
    for _ in range(args.warmup):
        run_oracle_jobs(jobs, threads)
    total_s = 0.0
    for _ in range(args.steps):
        total_s += run_oracle_jobs(jobs, threads)
    step_s = total_s / args.steps
    gbs = kv_bytes_layer(w["T"]) * n_layers / step_s / 1e9
    sample = (f"one whole step per timed step: all {n_layers} layers (prologue + full-softmax attention, T={w['T']}), "
              f"fp64 oracle, layers spread over {threads} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "us_per_layer_step": step_s * 1e6 / n_layers,
        "config": headline_config(w, n_layers),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg
def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import paged_gqa_decode_head_gb300 as pg
    from paged_gqa_decode_head_gb300 import inputs
    from paged_gqa_decode_head_gb300.runner import DecodeStep

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # before any work of ours: the GPU should be idle (no other compute
    # process, no utilization left from an earlier job)
    idle = gpu_idle_check(smi_gpu_id(dev))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    pg.load_library()
    w = inputs.WORKLOADS[WORKLOAD]
    n_layers = args.layers or w["layers"]
    layers = inputs.qwen3_layers(layers=n_layers)

    # CPU-baseline leg first (rank 0, one GPU job only), before any GPU work
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        jobs = [lambda lay=lay: oracle_layer(lay, w["theta"]) for lay in layers]
        n_single = min(4, n_layers)
        cpu_baseline = oracle_baseline(
            jobs, jobs[:n_single], kv_bytes_layer(w["T"]) * n_layers, kv_bytes_layer(w["T"]) * n_single,
            f"one whole step ({n_layers} layers, prologue + full-softmax attention, T={w['T']}) of the fp64 oracle",
            f"{n_single} of the step's layers one after another on one host thread")

    step = DecodeStep(layers, Hq=w["Hq"], Hkv=w["Hkv"], rope_theta=w["theta"], device=dev)
    np_used = step.partitions
    attn_graph = step.capture(prologue=False)  # attention only, same buffers
    two_launch_graph = step.capture(prologue=True, fused=False)  # prologue + attention per layer
    step_graph = step.capture(prologue=True, fused=True)  # the step: decode_step_paged per layer
    stream = torch.cuda.current_stream(dev)

    kv_bytes = sum(kv_bytes_layer(int(kv.context_lens.sum())) for kv, _ in layers)
    Hq, Hkv = w["Hq"], w["Hkv"]
    # algorithmic bytes of one decode_step_paged launch (one layer): the K+V
    # history, the new token's q, k, v and the two gains read, the block
    # table, the appended K and V rows, the rotated q and both outputs written
    algo_bytes_step = (kv_bytes_layer(w["T"]) + 2 * (Hq + 2 * Hkv) * 128 + 2 * 2 * 128 + 4 * math.ceil(w["T"] / 16)
                       + 2 * 2 * Hkv * 128 + 2 * Hq * 128 + 6 * Hq * 128)
    # attention alone (decode_attn_paged): history, q, table, outputs
    algo_bytes_attn = kv_bytes_layer(w["T"]) + 2 * Hq * 128 + 4 * math.ceil(w["T"] / 16) + 6 * Hq * 128

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(fn, steps):
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        barrier()
        return slowest_rank_ms(e0.elapsed_time(e1), world, dev)

    for _ in range(max(3, args.warmup)):
        step_graph.replay()
    for _ in range(max(3, args.warmup)):
        attn_graph.replay()
        two_launch_graph.replay()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(smi_gpu_id(dev))
    sampler.start()
    time.sleep(0.5)
    t_wall0 = time.time()
    ms = timed(step_graph.replay, args.steps)
    t_wall1 = time.time()
    ms_attn = timed(attn_graph.replay, args.steps)
    ms_two = timed(two_launch_graph.replay, args.steps)
    t_wall2 = time.time()

    # end to end through the public API: per step the new tokens (q, k, v of
    # every layer, packed as the step's new_tokens buffer) come from pinned
    # host memory in one copy and the fp32 outputs of every layer go back in
    # one copy.
    host_in = torch.cat([torch.from_numpy(np.concatenate([a.reshape(-1).view("int16") for a in (tok.q, tok.k, tok.v)]))
                         for _, tok in layers]).view(torch.bfloat16).pin_memory()
    host_out = torch.empty(step.outputs.shape, dtype=torch.float32).pin_memory()
    assert host_in.numel() == step.new_tokens.numel()
    h2d = host_in.numel() * 2
    d2h = host_out.numel() * 4

    # the copies are recorded into the step's graph with it (DecodeStep.capture)
    e2e_graph = step.capture(prologue=True, fused=True, host_in=host_in, host_out=host_out)

    def e2e_step():
        e2e_graph.replay()

    for _ in range(3):
        e2e_step()
    e2e_steps = max(1, min(args.steps, 500))
    ms_e2e = timed(e2e_step, e2e_steps)
    t_wall3 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall3)
    assert pg.device_error_flags() == 0, "device error flags raised during the benchmark"

    step_s = ms / args.steps / 1e3
    value = job_gbs(kv_bytes, world, step_s)
    layer_attn_s = ms_attn / args.steps / 1e3 / n_layers
    achieved = algo_bytes_step / (step_s / n_layers) / 1e9
    achieved_attn = algo_bytes_attn / layer_attn_s / 1e9
    peak, peak_kind = load_peaks()
    e2e_s = ms_e2e / e2e_steps / 1e3
    # one decode_step_paged kernel per layer; the library merges up to 64
    # partitions inside it and launches merge_kernel only beyond that
    launches_per_layer = 1 + (1 if np_used > 64 else 0)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "storage_dtype": "bf16", "accumulate": "f32",
        "p_operand": "bf16 hi + lo pair (about 16 significant bits) in the P.V product; scores and sums in f32",
        "data": "synthetic",
        "us_per_layer_step": step_s * 1e6 / n_layers,
        "attention_us_per_layer": layer_attn_s * 1e6,
        "two_launch_us_per_layer_step": ms_two / args.steps / n_layers * 1e3,
        "hbm_fraction_of_step": value / world / peak,
        "config": headline_config(w, n_layers),
        "launch": {"num_partitions": np_used, "graph": f"one CUDA graph per step ({n_layers} launches)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": profiled_traffic(),
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "kernel": "decode_mma_kernel<2, fused> (decode_step_paged: prologue, split-KV attention, "
                               f"in-kernel merge), {n_layers} launches per step graph, CUDA events on the launch "
                               "stream; achieved = algorithmic bytes of one launch / (step time / launches)",
                     "bytes_per_launch": algo_bytes_step,
                     "attention_only": {"achieved": achieved_attn, "frac": achieved_attn / peak,
                                        "bytes_per_launch": algo_bytes_attn,
                                        "kernel": "decode_mma_kernel<2> (decode_attn_paged), attention-only graph"}},
        "e2e": {"value": job_gbs(kv_bytes, world, e2e_s), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": args.steps * n_layers * launches_per_layer,
        "clocks": clocks,
        "gpu_idle_at_start": idle,
        "cpu_baseline": cpu_baseline,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def host_tiled_overlap(trace, group_bytes: int) -> dict:
    """Summary of a traced host-tiled run: per copy group g the events
    [4g] copy start, [4g+1] copy end, [4g+2] update start, [4g+3] update end.
    Returns the run's span, the time the copy stream and the compute stream
    were busy, how much of the update time ran while a copy was in flight,
    and the link rate of the copies themselves."""
    t = [trace[0].elapsed_time(ev) * 1e3 for ev in trace]  # us after the first copy start
    G = len(t) // 4
    copies = [(t[4 * g], t[4 * g + 1]) for g in range(G)]
    updates = [(t[4 * g + 2], t[4 * g + 3]) for g in range(G)]
    span = max(e for _, e in updates) - copies[0][0]

    def overlap(a, b):
        return max(0.0, min(a[1], b[1]) - max(a[0], b[0]))

    copy_busy = sum(e - s_ for s_, e in copies)
    update_busy = sum(e - s_ for s_, e in updates)
    update_under_copy = sum(overlap(u, c) for u in updates for c in copies)
    waits = [updates[g][0] - copies[g][1] for g in range(G)]
    return {"groups": G, "span_us": span, "copy_busy_us": copy_busy, "update_busy_us": update_busy,
            "copy_busy_frac": copy_busy / span, "update_under_copy_frac": update_under_copy / max(update_busy, 1e-9),
            "copy_gbs": G * group_bytes / (copy_busy * 1e-6) / 1e9,
            "median_copy_us": statistics.median(e - s_ for s_, e in copies),
            "median_update_us": statistics.median(e - s_ for s_, e in updates),
            "median_copy_end_to_update_start_us": statistics.median(waits),
            "first_groups_us": [[round(x, 1) for x in (c[0], c[1], u[0], u[1])] for c, u in zip(copies[:4], updates[:4])]}


def run_secondary(args):
    """Bandwidth of one of the larger workloads: KV bytes per second of
    decode_attn_paged (ragged batch, long split-KV context), or bytes per second
    over the host link of the host-tiled copy pipeline and of the zero-copy
    variant, each against its own roofline (measured HBM copy bandwidth, or a
    256 MiB pinned host-to-device copy timed in the same run)."""
    import numpy as np
    import torch

    import paged_gqa_decode_head_gb300 as pg
    from paged_gqa_decode_head_gb300 import inputs
    from paged_gqa_decode_head_gb300.runner import to_device_bf16, to_device_i32

    import oracle

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    idle = gpu_idle_check(smi_gpu_id(dev))
    pg.load_library()
    w = inputs.WORKLOADS[args.workload]
    scale = 1.0 / math.sqrt(128)
    peak, peak_kind = load_peaks()
    iters = max(3, min(args.steps, 500))
    sampler = ClockSampler(smi_gpu_id(dev))
    state = {"cpu": None}

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        state["t0"] = time.time()
        e0.record()
        for _ in range(iters):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        state["t1"] = time.time()
        return e0.elapsed_time(e1) / iters / 1e3

    def emit(variant, nbytes, s, roof_peak, roof_unit, roof_kind, extra):
        gbs = nbytes / s / 1e9
        line = {"metric": f"{args.workload} {variant}", "value": gbs, "unit": "GB/s", "us": s * 1e6,
                "workload": args.workload, "variant": variant, "steps": iters, "data": "synthetic",
                "roofline": {"achieved": gbs, "peak": roof_peak, "unit": roof_unit, "frac": gbs / roof_peak,
                             "peak_kind": roof_kind, "bytes": nbytes}}
        if roof_unit == "GB/s" and roof_kind != "measured link":
            line["roofline"]["frac_of_nominal"] = gbs / NOMINAL_HBM_GBS
        line.update(extra)
        line["clocks"] = sampler.summary(state["t0"], state["t1"])
        line["gpu_idle_at_start"] = idle
        line["cpu_baseline"] = state["cpu"]
        print(json.dumps(line), flush=True)

    def baseline(jobs, n_single, bytes_of, sample, single_sample):
        """The oracle on the same inputs, before any GPU timing (skipped with
        --no-cpu-baseline)."""
        if args.no_cpu_baseline:
            return
        state["cpu"] = oracle_baseline(jobs, jobs[:n_single], sum(bytes_of), sum(bytes_of[:n_single]), sample,
                                       single_sample)

    if args.workload in ("ragged_b64", "long_split_kv_t128k"):
        if args.workload == "ragged_b64":
            kv, q = inputs.ragged_b64(args.ragged_batch)
            nps = [0]
            jobs = [lambda b=b: oracle.decode_attention(q[b:b + 1], kv.k_cache, kv.v_cache, kv.block_table[b:b + 1],
                                                        kv.context_lens[b:b + 1], scale)
                    for b in range(len(kv.context_lens))]
            sizes = [kv_bytes_layer(int(t), w["Hkv"]) for t in kv.context_lens]
            baseline(jobs, 8, sizes, f"all {len(jobs)} sequences of the batch, full-softmax attention",
                     "the first 8 sequences one after another on one host thread")
        else:
            kv, q = inputs.long_split_kv()
            nps = [w["T"] // w["partition"], 0]
            g = w["Hq"] // w["Hkv"]
            # one job per KV head (its group of query heads over its own copy of that head's cache)
            heads = [(q[:, h * g:(h + 1) * g].copy(), kv.k_cache[:, h:h + 1].copy(), kv.v_cache[:, h:h + 1].copy())
                     for h in range(w["Hkv"])]
            jobs = [lambda x=x: oracle.decode_attention(x[0], x[1], x[2], kv.block_table, kv.context_lens, scale)
                    for x in heads]
            baseline(jobs, 1, [kv_bytes_layer(w["T"], 1)] * len(jobs),
                     f"the whole T={w['T']} attention, one job per KV head (its {g} query heads)",
                     "one KV head's job on one host thread")
            del heads
        sampler.start()
        time.sleep(0.5)
        B, Hq, Hkv = len(kv.context_lens), w["Hq"], w["Hkv"]
        qd = to_device_bf16(q, dev)
        kc, vc = to_device_bf16(kv.k_cache, dev), to_device_bf16(kv.v_cache, dev)
        bt, ctx = to_device_i32(kv.block_table, dev), to_device_i32(kv.context_lens, dev)
        out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
        kv_bytes = 4 * int(kv.context_lens.sum()) * Hkv * 128
        for npr in nps:
            n = pg.decode_attn_workspace_size(B, Hq, Hkv, 128, kv.page_size, kv.max_pages, npr)
            ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
            np_used = pg.decode_attn_partition_count(B, Hkv, kv.page_size, kv.max_pages, npr)
            s = timed(lambda: pg.decode_attn_paged(qd, kc, vc, bt, ctx, scale, out_f32=out, workspace=ws,
                                                   num_partitions=npr))
            emit(f"decode_attn_paged NP={np_used}" + (" (automatic)" if npr == 0 else " (workload's 512-position partitions)"),
                 kv_bytes, s, peak, "GB/s", peak_kind,
                 {"config": {"B": B, "Hq": Hq, "Hkv": Hkv, "P": kv.page_size, "kv_bytes": kv_bytes,
                             "l2": "inputs larger than L2"}})
        # the same workload over an INT8 cache (timing only: uniform codes,
        # scales 1/127; parity is the test suite's)
        del kc, vc
        k8 = torch.from_numpy(inputs.int8_rows(w["seed"], kv.k_cache.shape, 72)).to(dev)
        v8 = torch.from_numpy(inputs.int8_rows(w["seed"], kv.v_cache.shape, 73)).to(dev)
        ks = torch.full(kv.k_cache.shape[:-1], 1.0 / 127, dtype=torch.float32, device=dev)
        vs = torch.full(kv.v_cache.shape[:-1], 1.0 / 127, dtype=torch.float32, device=dev)
        int8_bytes = kv_bytes // 512 * (2 * 128 + 2 * 4)
        for npr in nps:
            n = pg.decode_attn_int8_workspace_size(B, Hq, Hkv, 128, kv.page_size, kv.max_pages, npr)
            ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
            np_used = pg.decode_attn_partition_count(B, Hkv, kv.page_size, kv.max_pages, npr)
            s = timed(lambda: pg.decode_attn_paged_int8(qd, k8, v8, ks, vs, bt, ctx, scale, out_f32=out,
                                                        workspace=ws, num_partitions=npr))
            emit(f"decode_attn_paged_int8 NP={np_used}" +
                 (" (automatic)" if npr == 0 else " (workload's 512-position partitions)"),
                 int8_bytes, s, peak, "GB/s", peak_kind,
                 {"bf16_equivalent_gbs": kv_bytes / s / 1e9,
                  "config": {"B": B, "Hq": Hq, "Hkv": Hkv, "P": kv.page_size, "int8_bytes": int8_bytes,
                             "l2": "inputs larger than L2"}})
        sampler.stop()
        assert pg.device_error_flags() == 0
        return

    if args.workload == "qwen3_0p6b_t8k_m4":
        # multi-token verification: per layer the M-token prologue and the
        # M-token attention, 28 layers in one CUDA graph
        layers = inputs.qwen3_layers_multi()
        B, M, Hq, Hkv, T = w["B"], w["M"], w["Hq"], w["Hkv"], w["T"]

        def oracle_multi(layer):
            kv, q, k, v, gq, gk = layer
            q_ref, kc, vc = oracle.qk_norm_rope_append_multi(q, k, v, gq, gk, kv.context_lens, kv.block_table,
                                                             kv.k_cache, kv.v_cache, kv.page_size, w["theta"])
            oracle.decode_attention_multi(q_ref, kc, vc, kv.block_table, kv.context_lens, scale)

        jobs = [lambda lay=lay: oracle_multi(lay) for lay in layers]
        baseline(jobs, 2, [kv_bytes_layer(T, Hkv)] * len(jobs),
                 f"one whole step ({len(jobs)} layers, M={M}-token prologue + full-softmax attention)",
                 "2 of the step's layers one after another on one host thread")
        sampler.start()
        time.sleep(0.5)
        bufs = []
        for kv, q, k, v, gq, gk in layers:
            bufs.append(dict(kc=to_device_bf16(kv.k_cache, dev), vc=to_device_bf16(kv.v_cache, dev),
                             bt=to_device_i32(kv.block_table, dev), ctx=to_device_i32(kv.context_lens, dev),
                             q=to_device_bf16(q, dev), k=to_device_bf16(k, dev), v=to_device_bf16(v, dev),
                             gq=to_device_bf16(gq, dev), gk=to_device_bf16(gk, dev),
                             q_out=torch.empty((B, M, Hq, 128), dtype=torch.bfloat16, device=dev),
                             out=torch.empty((B, M, Hq, 128), dtype=torch.float32, device=dev)))
        P, max_pages = layers[0][0].page_size, layers[0][0].max_pages
        n = pg.decode_attn_multi_workspace_size(B, M, Hq, Hkv, 128, P, max_pages, 0)
        ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)

        def two_launch():
            for b_ in bufs:
                pg.qk_norm_rope_append_multi(b_["q"], b_["k"], b_["v"], b_["gq"], b_["gk"], b_["ctx"], b_["bt"],
                                             b_["kc"], b_["vc"], b_["q_out"], w["theta"])
                pg.decode_attn_paged_multi(b_["q_out"], b_["kc"], b_["vc"], b_["bt"], b_["ctx"], scale,
                                           out_f32=b_["out"], workspace=ws)

        def fused():
            for b_ in bufs:
                pg.decode_step_paged_multi(b_["q"], b_["k"], b_["v"], b_["gq"], b_["gk"], b_["ctx"], b_["bt"],
                                           b_["kc"], b_["vc"], scale, w["theta"], q_out=b_["q_out"],
                                           out_f32=b_["out"], workspace=ws)

        def capture(step):
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                step()
            torch.cuda.current_stream(dev).wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            return graph

        L = len(layers)
        kv_bytes = 4 * T * Hkv * 128 * L
        for name, step in (("decode_step_paged_multi (one launch per layer)", fused),
                           ("qk_norm_rope_append_multi + decode_attn_paged_multi", two_launch)):
            s = timed(capture(step).replay)
            emit(f"{name}, M={M}, {L} layers per graph", kv_bytes, s, peak, "GB/s", peak_kind,
                 {"us_per_layer_step": s * 1e6 / L,
                  "config": {"B": B, "M": M, "Hq": Hq, "Hkv": Hkv, "T": T, "P": P, "layers": L,
                             "num_partitions": pg.decode_attn_partition_count(B, Hkv, P, max_pages, 0),
                             "l2": "inputs larger than L2: 896 MiB of KV"}})
        sampler.stop()
        assert pg.device_error_flags() == 0
        return

    if args.workload == "qwen3_0p6b_t8k_int8":
        # the Qwen3-shaped 28-layer T = 8192 step over an INT8 cache: per layer
        # the quantizing prologue and the INT8 attention, one CUDA graph
        B, Hq, Hkv, T = w["B"], w["Hq"], w["Hkv"], w["T"]
        L = 28
        bufs = []
        host = []
        for i in range(L):
            seed = w["seed"] * 1000 + i
            kv = inputs.paged_kv(seed, [T] * B, Hkv=Hkv, page_size=w["page_size"], spare_pages=0,
                                 fill_unused="normal")
            tok = inputs.new_token(seed, B, Hq, Hkv)
            k8h = inputs.int8_rows(seed, kv.k_cache.shape, 70)
            v8h = inputs.int8_rows(seed, kv.v_cache.shape, 71)
            if i < 8:
                host.append((kv, tok, k8h, v8h))
            k8 = torch.from_numpy(k8h).to(dev)
            v8 = torch.from_numpy(v8h).to(dev)
            ks = torch.full(kv.k_cache.shape[:-1], 1.0 / 127, dtype=torch.float32, device=dev)
            vs = torch.full(kv.v_cache.shape[:-1], 1.0 / 127, dtype=torch.float32, device=dev)
            bufs.append(dict(k8=k8, v8=v8, ks=ks, vs=vs, bt=to_device_i32(kv.block_table, dev),
                             ctx=to_device_i32(kv.context_lens, dev), q=to_device_bf16(tok.q, dev),
                             k=to_device_bf16(tok.k, dev), v=to_device_bf16(tok.v, dev),
                             gq=to_device_bf16(tok.gamma_q, dev), gk=to_device_bf16(tok.gamma_k, dev),
                             q_out=torch.empty((B, Hq, 128), dtype=torch.bfloat16, device=dev),
                             out=torch.empty((B, Hq, 128), dtype=torch.float32, device=dev),
                             P=kv.page_size, mp=kv.max_pages))
        n = pg.decode_attn_int8_workspace_size(B, Hq, Hkv, 128, bufs[0]["P"], bufs[0]["mp"], 0)
        ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)

        def oracle_int8(layer):
            kv, tok, k8h, v8h = layer
            ks = np.full(kv.k_cache.shape[:-1], 1.0 / 127, dtype=np.float32)
            vs = np.full(kv.v_cache.shape[:-1], 1.0 / 127, dtype=np.float32)
            q_ref, kc, vc, ksc, vsc = oracle.qk_norm_rope_append_int8(
                tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k, kv.context_lens, kv.block_table, k8h, v8h, ks, vs,
                kv.page_size, w["theta"])
            oracle.decode_attention_int8(q_ref, kc, vc, ksc, vsc, kv.block_table, kv.context_lens, scale)

        jobs = [lambda lay=lay: oracle_int8(lay) for lay in host]
        baseline(jobs, 2, [(2 * 128 + 2 * 4) * T * Hkv] * len(jobs),
                 f"{len(jobs)} of the step's {L} layers (INT8 prologue + full-softmax attention over the codes)",
                 "2 layers one after another on one host thread")
        del host
        sampler.start()
        time.sleep(0.5)

        def attention_only():
            for b_ in bufs:
                pg.decode_attn_paged_int8(b_["q"], b_["k8"], b_["v8"], b_["ks"], b_["vs"], b_["bt"], b_["ctx"], scale,
                                          out_f32=b_["out"], workspace=ws)

        def step():
            for b_ in bufs:
                pg.qk_norm_rope_append_int8(b_["q"], b_["k"], b_["v"], b_["gq"], b_["gk"], b_["ctx"], b_["bt"],
                                            b_["k8"], b_["v8"], b_["ks"], b_["vs"], b_["q_out"], w["theta"])
                pg.decode_attn_paged_int8(b_["q_out"], b_["k8"], b_["v8"], b_["ks"], b_["vs"], b_["bt"], b_["ctx"],
                                          scale, out_f32=b_["out"], workspace=ws)

        def fused():
            for b_ in bufs:
                pg.decode_step_paged_int8(b_["q"], b_["k"], b_["v"], b_["gq"], b_["gk"], b_["ctx"], b_["bt"],
                                          b_["k8"], b_["v8"], b_["ks"], b_["vs"], scale, w["theta"],
                                          q_out=b_["q_out"], out_f32=b_["out"], workspace=ws)

        def capture(fn):
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                fn()
            torch.cuda.current_stream(dev).wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                fn()
            return graph

        int8_bytes = (2 * 128 + 2 * 4) * T * Hkv * L  # codes and scales of K and V
        bf16_bytes = 4 * T * Hkv * 128 * L
        for name, fn in (("decode_step_paged_int8 (one launch per layer)", fused),
                         ("decode_attn_paged_int8 alone", attention_only),
                         ("qk_norm_rope_append_int8 + decode_attn_paged_int8", step)):
            s = timed(capture(fn).replay)
            emit(f"{name}, {L} layers per graph", int8_bytes, s, peak, "GB/s", peak_kind,
                 {"us_per_layer_step": s * 1e6 / L, "bf16_equivalent_gbs": bf16_bytes / s / 1e9,
                  "config": {"B": B, "Hq": Hq, "Hkv": Hkv, "T": T, "P": bufs[0]["P"], "layers": L,
                             "bytes_per_row": "128 int8 codes + 1 float scale, K and V",
                             "l2": "inputs larger than L2: 462 MB of int8 KV"}})
        sampler.stop()
        assert pg.device_error_flags() == 0
        return

    # host_tiled_t64k: the copy pipeline and the zero-copy variant
    q, k, v = inputs.host_tiled_kv()
    B, Hq, Hkv, T, tile = w["B"], w["Hq"], w["Hkv"], w["T"], w["tile"]
    g = Hq // Hkv
    heads = [(q[:, h * g:(h + 1) * g].copy(), k[:, :, h:h + 1].copy(), v[:, :, h:h + 1].copy()) for h in range(Hkv)]
    jobs = [lambda x=x: oracle.attention_contiguous(x[0], x[1], x[2], scale) for x in heads]
    baseline(jobs, 1, [kv_bytes_layer(T, 1) * B] * len(jobs),
             f"the whole T={T} attention, one job per KV head (its {g} query heads)",
             "one KV head's job on one host thread")
    del heads
    sampler.start()
    time.sleep(0.5)
    hk = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
    nbytes = 2 * hk.numel() * 2
    probe = torch.empty(hk.numel(), dtype=torch.bfloat16, device=dev)
    link = max(hk.numel() * 2 / timed(lambda: probe.copy_(hk.view(-1), non_blocking=True)) / 1e9 for _ in range(3))
    del probe
    qd = to_device_bf16(q, dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    n_slots = 2
    m = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    l = torch.empty_like(m)
    acc = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    copy_stream = torch.cuda.Stream(dev)
    cfg = {"B": B, "Hq": Hq, "Hkv": Hkv, "T": T, "host_bytes": nbytes,
           "link_probe": "256 MiB pinned host-to-device cudaMemcpyAsync, best of 3"}
    # one tile per copy (the pages' pipeline), then eight 512-position tiles
    # per copy (8 MiB transfers), each tile still updated on its own
    for per_copy in (1, 8):
        slots_k = [torch.empty((B, tile * per_copy, Hkv, 128), dtype=torch.bfloat16, device=dev)
                   for _ in range(n_slots)]
        slots_v = [torch.empty((B, tile * per_copy, Hkv, 128), dtype=torch.bfloat16, device=dev)
                   for _ in range(n_slots)]
        events = [torch.cuda.Event() for _ in range(2 * n_slots)]
        s = timed(lambda: pg.attn_host_tiled_run(qd, hk, hv, scale, slots_k, slots_v, events, m, l, acc,
                                                 out_f32=out, tile_len=tile, tiles_per_copy=per_copy,
                                                 copy_stream=copy_stream))
        emit(f"attn_host_tiled_run ({tile}-position tiles, {per_copy} per copy, {n_slots} slots)", nbytes, s, link,
             "GB/s", "measured link", {"config": cfg})
        # one more run with an event pair around every copy and every group
        # of updates (attn_host_tiled_run_traced): how the copies and the
        # updates overlap
        n_groups = -(-T // (tile * per_copy))
        trace = [torch.cuda.Event(enable_timing=True) for _ in range(4 * n_groups)]
        pg.attn_host_tiled_run(qd, hk, hv, scale, slots_k, slots_v, events, m, l, acc, out_f32=out, tile_len=tile,
                               tiles_per_copy=per_copy, copy_stream=copy_stream, trace_events=trace)
        torch.cuda.synchronize(dev)
        print(json.dumps({"metric": f"{args.workload} attn_host_tiled_run pipeline trace ({per_copy} per copy)",
                          **host_tiled_overlap(trace, per_copy * tile * Hkv * 128 * 2 * 2 * B)}), flush=True)
        del slots_k, slots_v
    n = pg.attn_host_direct_workspace_size(B, Hq, Hkv, T, 0)
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device=dev)
    np_used = pg.attn_host_direct_partition_count(B, Hkv, T, 0)
    s = timed(lambda: pg.attn_host_direct(qd, hk, hv, scale, out_f32=out, workspace=ws))
    emit(f"attn_host_direct (zero-copy, NP={np_used})", nbytes, s, link, "GB/s", "measured link", {"config": cfg})
    sampler.stop()


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.gpus != world and world != 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload != WORKLOAD:
        if rank == 0:
            run_secondary(args)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
