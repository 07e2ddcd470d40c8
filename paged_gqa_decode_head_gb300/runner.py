"""Multi-layer decode step on one GPU, built on the C ABI.

A decode step runs, for every layer, the fused prologue
(qk_norm_rope_append) followed by decode attention (decode_attn_paged) over
that layer's paged KV cache. Buffers are allocated once with PyTorch at
construction (the hot path allocates nothing); ``capture()`` records the whole
step into one CUDA graph so that replays pay a single launch.

Inputs come as numpy bit patterns (see ``inputs``) and are uploaded once.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from . import binding
from .inputs import NewToken, PagedKV


def to_device_bf16(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> a bf16 tensor on `device` (bit for bit)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def to_device_i32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@dataclasses.dataclass
class LayerState:
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    context_lens: torch.Tensor
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    gamma_q: torch.Tensor
    gamma_k: torch.Tensor
    q_out: torch.Tensor
    out_f32: torch.Tensor
    out_bf16: torch.Tensor
    page_size: int


class DecodeStep:
    """One decode step over `len(layers)` layers of paged GQA attention."""

    def __init__(self, layers: list[tuple[PagedKV, NewToken]], Hq: int, Hkv: int, rope_theta: float,
                 eps: float = 1e-6, scale: float | None = None, num_partitions: int = 0,
                 device: str | torch.device = "cuda"):
        self.device = torch.device(device)
        self.Hq, self.Hkv = Hq, Hkv
        self.D = 128
        self.rope_theta = float(rope_theta)
        self.eps = float(eps)
        self.scale = float(scale) if scale is not None else 1.0 / math.sqrt(self.D)
        self.layers: list[LayerState] = []
        ws_bytes = 0
        # Every layer's new-token heads (q, k, v) live in one buffer and every
        # layer's fp32 output in another, so a step's inputs and results move
        # between host and device in one copy each (``new_tokens``,
        # ``outputs``); the per-layer tensors are views into them.
        B = int(layers[0][0].context_lens.shape[0]) if layers else 0
        if any(int(kv.context_lens.shape[0]) != B for kv, _ in layers):
            raise ValueError("every layer of a decode step has the same batch")
        q_n, kv_n = B * Hq * self.D, B * Hkv * self.D
        per_layer = q_n + 2 * kv_n
        self.new_tokens = torch.empty(len(layers) * per_layer, dtype=torch.bfloat16, device=self.device)
        self.outputs = torch.empty((len(layers), B, Hq, self.D), dtype=torch.float32, device=self.device)
        for i, (kv, tok) in enumerate(layers):
            heads = self.new_tokens[i * per_layer:(i + 1) * per_layer]
            q, k, v = (heads[:q_n].view(B, Hq, self.D), heads[q_n:q_n + kv_n].view(B, Hkv, self.D),
                       heads[q_n + kv_n:].view(B, Hkv, self.D))
            q.copy_(to_device_bf16(tok.q, self.device))
            k.copy_(to_device_bf16(tok.k, self.device))
            v.copy_(to_device_bf16(tok.v, self.device))
            st = LayerState(
                k_cache=to_device_bf16(kv.k_cache, self.device),
                v_cache=to_device_bf16(kv.v_cache, self.device),
                block_table=to_device_i32(kv.block_table, self.device),
                context_lens=to_device_i32(kv.context_lens, self.device),
                q=q,
                k=k,
                v=v,
                gamma_q=to_device_bf16(tok.gamma_q, self.device),
                gamma_k=to_device_bf16(tok.gamma_k, self.device),
                q_out=torch.empty((B, Hq, self.D), dtype=torch.bfloat16, device=self.device),
                out_f32=self.outputs[i],
                out_bf16=torch.empty((B, Hq, self.D), dtype=torch.bfloat16, device=self.device),
                page_size=kv.page_size,
            )
            self.layers.append(st)
            ws_bytes = max(ws_bytes, binding.decode_attn_workspace_size(
                B, Hq, Hkv, self.D, kv.page_size, kv.max_pages, num_partitions))
        self.num_partitions = int(num_partitions)
        self.workspace = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=self.device)
        self.graph: torch.cuda.CUDAGraph | None = None

    @property
    def partitions(self) -> int:
        st = self.layers[0]
        return binding.decode_attn_partition_count(st.block_table.shape[0], self.Hkv, st.page_size,
                                                   st.block_table.shape[1], self.num_partitions)

    def run_layer(self, i: int, stream=None, prologue: bool = True, fused: bool = False) -> None:
        st = self.layers[i]
        if prologue and fused:
            binding.decode_step_paged(st.q, st.k, st.v, st.gamma_q, st.gamma_k, st.context_lens, st.block_table,
                                      st.k_cache, st.v_cache, self.scale, self.rope_theta, self.eps, q_out=st.q_out,
                                      out_f32=st.out_f32, out_bf16=st.out_bf16, workspace=self.workspace,
                                      num_partitions=self.num_partitions, stream=stream)
            return
        if prologue:
            binding.qk_norm_rope_append(st.q, st.k, st.v, st.gamma_q, st.gamma_k, st.context_lens, st.block_table,
                                        st.k_cache, st.v_cache, st.q_out, st.page_size, self.rope_theta, self.eps,
                                        stream=stream)
        binding.decode_attn_paged(st.q_out, st.k_cache, st.v_cache, st.block_table, st.context_lens, self.scale,
                                  out_f32=st.out_f32, out_bf16=st.out_bf16, workspace=self.workspace,
                                  num_partitions=self.num_partitions, stream=stream)

    def run(self, stream=None, prologue: bool = True, fused: bool = False) -> None:
        """One step: per layer the prologue and the attention, as two launches
        or (fused=True) as one decode_step_paged launch."""
        for i in range(len(self.layers)):
            self.run_layer(i, stream=stream, prologue=prologue, fused=fused)

    def capture(self, prologue: bool = True, fused: bool = False, host_in: torch.Tensor | None = None,
                host_out: torch.Tensor | None = None) -> torch.cuda.CUDAGraph:
        """Record one whole step (every layer) into a CUDA graph.

        With ``host_in`` (pinned, bf16, shaped like ``new_tokens``) the graph
        starts with the copy of the step's new tokens from it; with
        ``host_out`` (pinned, fp32, shaped like ``outputs``) it ends with the
        copy of every layer's output into it. A replay is then one whole step
        from host inputs to host results; synchronise before reading
        ``host_out``."""
        if host_in is not None and (host_in.device.type != "cpu" or not host_in.is_pinned()
                                    or host_in.dtype != torch.bfloat16
                                    or host_in.numel() != self.new_tokens.numel()):
            raise ValueError("host_in must be pinned host bf16 memory with new_tokens' element count")
        if host_out is not None and (host_out.device.type != "cpu" or not host_out.is_pinned()
                                     or host_out.dtype != torch.float32
                                     or host_out.shape != self.outputs.shape):
            raise ValueError("host_out must be pinned host fp32 memory shaped like outputs")

        def step():
            if host_in is not None:
                self.new_tokens.copy_(host_in.view(-1), non_blocking=True)
            self.run(prologue=prologue, fused=fused)
            if host_out is not None:
                host_out.copy_(self.outputs, non_blocking=True)

        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            step()  # warm-up outside capture
        torch.cuda.current_stream(self.device).wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        self.graph = g
        return g

    def replay(self) -> None:
        assert self.graph is not None, "capture() first"
        self.graph.replay()

    def kv_bytes_per_step(self) -> int:
        """Algorithmic K+V bytes the attention reads in one step: 4*T*Hkv*D per sequence and layer."""
        total = 0
        for st in self.layers:
            total += 4 * int(st.context_lens.sum().item()) * self.Hkv * self.D
        return total
