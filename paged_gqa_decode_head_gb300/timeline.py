"""Per-phase timeline of the decode step chain (a measurement tool).

Builds libpgqa_timeline.so (the library with %globaltimer stamps compiled
into the split kernel), captures the 28-layer T = 8192 Qwen3-shaped step as
one CUDA graph (the fused step, then attention alone), replays it and prints,
for each phase of a layer, when it happens relative to the end of the
previous layer (the last CTA's merge): min, median and max over the layer's
CTAs, averaged over layers 4..27 and several replays. The stamps themselves
cost a little: the instrumented step runs a few tenths of a microsecond
slower per layer than the plain library, which the tool reports beside it.

    python -m paged_gqa_decode_head_gb300.timeline [--replays 10] [--partitions 0] [--int8 | --multi]

--int8 runs the same chain over an INT8 cache (decode_step_paged_int8 and
decode_attn_paged_int8; codes uniform in [-127, 127], scales 1/127, as the
benchmark's INT8 chain). --multi runs the M = 4 multi-token chain
(decode_step_paged_multi and decode_attn_paged_multi, the benchmark's
qwen3_0p6b_t8k_m4 workload).
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np

PHASES = [
    (0, "CTA start"),
    (1, "block-table entries in hand (warp 0)"),
    (2, "first requests issued (warp 0)"),
    (3, "grid dependency released"),
    (4, "query rotated (fused step)"),
    (5, "second chunk landed (warp 0)"),
    (6, "last chunk landed (latest warp)"),
    (7, "warp records merged"),
    (8, "partition state written"),
    (9, "ticket back"),
    (10, "merge done (last CTA)"),
]


def _layer_ends(d):
    """End of each launch: the last merge, else the last state/records write."""
    ends = []
    for x in d:
        cand = [x[:, s][x[:, s] > 0] for s in (10, 8, 7)]
        ends.append(max(int(c.max()) for c in cand if c.size))
    return ends


def summarise(d, first_layer: int = 4):
    """d: [layers][CTAs][slots] stamps (ns) -> {slot: (min, med, max)} in us
    after the previous layer's end, averaged over layers first_layer.."""
    ends = _layer_ends(d)
    acc = {s: [] for s, _ in PHASES}
    lens = []
    for l in range(first_layer, len(d)):
        ref = ends[l - 1]
        for s, _ in PHASES:
            v = d[l][:, s]
            v = v[v > 0]
            if v.size:
                acc[s].append(((v.min() - ref) / 1e3, (np.median(v) - ref) / 1e3, (v.max() - ref) / 1e3))
        lens.append((ends[l] - ref) / 1e3)
    out = {s: tuple(np.mean(np.array(a), axis=0)) for s, a in acc.items() if a}
    return out, float(np.mean(lens))


class Int8Chain:
    """The 28-layer T = 8192 chain over INT8 caches, with DecodeStep's
    partitions and capture() interface (the benchmark's INT8 leg)."""

    def __init__(self, layers: int, num_partitions: int):
        import torch

        from . import binding, inputs
        from .runner import to_device_bf16, to_device_i32

        w = inputs.WORKLOADS["qwen3_0p6b_t8k_int8"]
        self.w = w
        self.num_partitions = num_partitions
        self.bufs = []
        for i in range(layers):
            seed = w["seed"] * 1000 + i
            kv = inputs.paged_kv(seed, [w["T"]] * w["B"], Hkv=w["Hkv"], page_size=w["page_size"], spare_pages=0,
                                 fill_unused="normal")
            tok = inputs.new_token(seed, w["B"], w["Hq"], w["Hkv"])
            self.bufs.append(dict(
                k8=torch.from_numpy(inputs.int8_rows(seed, kv.k_cache.shape, 70)).cuda(),
                v8=torch.from_numpy(inputs.int8_rows(seed, kv.v_cache.shape, 71)).cuda(),
                ks=torch.full(kv.k_cache.shape[:-1], 1.0 / 127, dtype=torch.float32, device="cuda"),
                vs=torch.full(kv.v_cache.shape[:-1], 1.0 / 127, dtype=torch.float32, device="cuda"),
                bt=to_device_i32(kv.block_table, "cuda"), ctx=to_device_i32(kv.context_lens, "cuda"),
                q=to_device_bf16(tok.q, "cuda"), k=to_device_bf16(tok.k, "cuda"), v=to_device_bf16(tok.v, "cuda"),
                gq=to_device_bf16(tok.gamma_q, "cuda"), gk=to_device_bf16(tok.gamma_k, "cuda"),
                q_out=torch.empty((w["B"], w["Hq"], 128), dtype=torch.bfloat16, device="cuda"),
                out=torch.empty((w["B"], w["Hq"], 128), dtype=torch.float32, device="cuda"),
                P=kv.page_size, mp=kv.max_pages))
        b0 = self.bufs[0]
        n = binding.decode_attn_int8_workspace_size(w["B"], w["Hq"], w["Hkv"], 128, b0["P"], b0["mp"],
                                                     num_partitions)
        self.ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")

    @property
    def partitions(self) -> int:
        from . import binding

        b0 = self.bufs[0]
        return binding.decode_attn_partition_count(self.w["B"], self.w["Hkv"], b0["P"], b0["mp"],
                                                   self.num_partitions)

    def run(self, fused: bool):
        import math

        from . import binding

        scale = 1.0 / math.sqrt(128)
        for b_ in self.bufs:
            if fused:
                binding.decode_step_paged_int8(b_["q"], b_["k"], b_["v"], b_["gq"], b_["gk"], b_["ctx"], b_["bt"],
                                               b_["k8"], b_["v8"], b_["ks"], b_["vs"], scale, self.w["theta"],
                                               q_out=b_["q_out"], out_f32=b_["out"], workspace=self.ws,
                                               num_partitions=self.num_partitions)
            else:
                binding.decode_attn_paged_int8(b_["q"], b_["k8"], b_["v8"], b_["ks"], b_["vs"], b_["bt"], b_["ctx"],
                                               scale, out_f32=b_["out"], workspace=self.ws,
                                               num_partitions=self.num_partitions)

    def capture(self, prologue: bool = True, fused: bool = False):
        return _capture(lambda: self.run(fused))


class MultiChain:
    """The 28-layer T = 8192 chain with M = 4 new tokens per layer, with
    DecodeStep's partitions and capture() interface (the benchmark's M = 4
    leg). Attention alone runs on the raw queries."""

    def __init__(self, num_partitions: int):
        import torch

        from . import binding, inputs
        from .runner import to_device_bf16, to_device_i32

        w = inputs.WORKLOADS["qwen3_0p6b_t8k_m4"]
        self.w = w
        self.num_partitions = num_partitions
        B, M, Hq = w["B"], w["M"], w["Hq"]
        self.bufs = []
        for kv, q, k, v, gq, gk in inputs.qwen3_layers_multi():
            self.bufs.append(dict(
                kc=to_device_bf16(kv.k_cache, "cuda"), vc=to_device_bf16(kv.v_cache, "cuda"),
                bt=to_device_i32(kv.block_table, "cuda"), ctx=to_device_i32(kv.context_lens, "cuda"),
                q=to_device_bf16(q, "cuda"), k=to_device_bf16(k, "cuda"), v=to_device_bf16(v, "cuda"),
                gq=to_device_bf16(gq, "cuda"), gk=to_device_bf16(gk, "cuda"),
                q_out=torch.empty((B, M, Hq, 128), dtype=torch.bfloat16, device="cuda"),
                out=torch.empty((B, M, Hq, 128), dtype=torch.float32, device="cuda"),
                P=kv.page_size, mp=kv.max_pages))
        b0 = self.bufs[0]
        n = binding.decode_attn_multi_workspace_size(B, M, Hq, w["Hkv"], 128, b0["P"], b0["mp"], num_partitions)
        self.ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")

    @property
    def partitions(self) -> int:
        from . import binding

        b0 = self.bufs[0]
        return binding.decode_attn_partition_count(self.w["B"], self.w["Hkv"], b0["P"], b0["mp"],
                                                   self.num_partitions)

    def run(self, fused: bool):
        import math

        from . import binding

        scale = 1.0 / math.sqrt(128)
        for b_ in self.bufs:
            if fused:
                binding.decode_step_paged_multi(b_["q"], b_["k"], b_["v"], b_["gq"], b_["gk"], b_["ctx"], b_["bt"],
                                                b_["kc"], b_["vc"], scale, self.w["theta"], q_out=b_["q_out"],
                                                out_f32=b_["out"], workspace=self.ws,
                                                num_partitions=self.num_partitions)
            else:
                binding.decode_attn_paged_multi(b_["q"], b_["kc"], b_["vc"], b_["bt"], b_["ctx"], scale,
                                                out_f32=b_["out"], workspace=self.ws,
                                                num_partitions=self.num_partitions)

    def capture(self, prologue: bool = True, fused: bool = False):
        return _capture(lambda: self.run(fused))


def _capture(run):
    """Warm-up run on a side stream, then the same run captured as a graph."""
    import torch

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    return g


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--replays", type=int, default=10)
    ap.add_argument("--partitions", type=int, default=0, help="0: the library's automatic count")
    mode = ap.add_mutually_exclusive_group()
    mode.add_argument("--int8", action="store_true", help="the INT8 cache's step and attention instead of bf16")
    mode.add_argument("--multi", action="store_true", help="the M = 4 multi-token step and attention")
    ap.add_argument("--library", default=None,
                    help="an already built timeline library (default: build libpgqa_timeline.so here)")
    args = ap.parse_args(argv)

    import torch

    from . import binding, build, inputs
    from .runner import DecodeStep

    path = args.library or build.build(variant="timeline")
    lib = binding.load_library(path)
    lib.pgqa_timeline_attach.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.pgqa_timeline_attach.restype = ctypes.c_int
    slots = lib.pgqa_timeline_attach(None, 1)
    L = 28
    w = inputs.WORKLOADS["qwen3_0p6b_t8k"]
    if args.int8:
        step = Int8Chain(L, args.partitions)
    elif args.multi:
        step = MultiChain(args.partitions)
    else:
        step = DecodeStep(inputs.qwen3_layers(layers=L), Hq=w["Hq"], Hkv=w["Hkv"], rope_theta=w["theta"],
                          num_partitions=args.partitions)
    np_used = step.partitions
    grid = np_used * w["Hkv"]
    buf = torch.zeros(L * grid * slots, dtype=torch.int64, device="cuda")
    print(f"28 layers, B=1, Hq=16, Hkv=8, T=8192{', M=4' if args.multi else ''}, NP={np_used} "
          f"({grid} CTAs per launch)")
    keep = []
    for fused in (True, False):
        name = "fused step (decode_step_paged)" if fused else "attention alone (decode_attn_paged)"
        if args.int8:
            name = name.replace("paged)", "paged_int8)")
        if args.multi:
            name = name.replace("paged)", "paged_multi)")
        lib.pgqa_timeline_attach(None, 1)
        plain = step.capture(prologue=fused, fused=fused)
        # the capture's warm-up run takes the first L launch slots, the
        # captured launches the same slots again
        lib.pgqa_timeline_attach(ctypes.c_void_p(buf.data_ptr()), L)
        stamped = step.capture(prologue=fused, fused=fused)
        lib.pgqa_timeline_attach(None, 1)
        keep += [plain, stamped]

        def per_layer_us(g, n=100):
            for _ in range(5):
                g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / (n * L)

        t_plain = per_layer_us(plain)
        t_stamped = per_layer_us(stamped, 20)
        rows, lens = [], []
        for _ in range(args.replays):
            buf.zero_()
            torch.cuda.synchronize()
            stamped.replay()
            torch.cuda.synchronize()
            d = buf.view(L, grid, slots).cpu().numpy()
            r, ln = summarise(d)
            rows.append(r)
            lens.append(ln)
        print(f"\n{name}: {t_plain:.2f} us per layer (timeline library, stamps off), "
              f"{t_stamped:.2f} us per layer stamped")
        print(f"  {'phase (us after the previous layer end)':42s} {'min':>7s} {'median':>7s} {'max':>7s}")
        for s, label in PHASES:
            vals = [r[s] for r in rows if s in r]
            if not vals:
                continue
            m = np.mean(np.array(vals), axis=0)
            print(f"  {label:42s} {m[0]:7.2f} {m[1]:7.2f} {m[2]:7.2f}")
        print(f"  {'layer end (next layer starts from here)':42s} {np.mean(lens):7.2f}")
    flags = binding.device_error_flags()
    if flags:
        print(f"device error flags: {flags}", file=sys.stderr)
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
