"""Seeded synthetic inputs for the paged GQA decode step.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Both the CUDA path and the CPU oracle consume exactly the
bit patterns it produces (bf16 as ``uint16``, indices as ``int32``), so the
two sides see identical inputs.

Recipe (shared by the tests and the benchmark):
  * generator: numpy PCG64 seeded by ``SeedSequence([seed, stream])`` where
    ``stream`` names the tensor (one stream per tensor);
  * values: q/k/v/cache entries ~ N(0, 1) drawn in float32 and rounded to bf16
    (nearest, ties to even); RMSNorm gains ~ U(0.5, 1.5) the same way;
  * block tables: a seeded random permutation of a physical page pool, so
    logical pages land on scattered physical pages; entries past a
    sequence's last page hold an out-of-pool value that must never be read;
  * cache slots that no sequence owns (the tail of a last page, spare pages)
    are filled with bf16 NaN (0xFFFF) unless asked otherwise, so that any
    read of an unowned slot shows up in the result.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BF16_NAN = np.uint16(0xFFFF)
UNUSED_TABLE_ENTRY = np.int32(0x3FFFFFFF)

_CHUNK = 1 << 20


def generator(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, nearest with ties to even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(gen: np.random.Generator, shape) -> np.ndarray:
    """bf16 bit patterns of N(0, 1) draws. Generated through one reused chunk
    buffer (large fresh temporaries are slow to fault in on some hosts)."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint16)
    chunk = max(1, min(n, _CHUNK))
    f = np.empty(chunk, dtype=np.float32)
    u = f.view(np.uint32)
    t = np.empty(chunk, dtype=np.uint32)
    for s in range(0, n, chunk):
        m = min(n, s + chunk) - s
        gen.standard_normal(out=f[:m], dtype=np.float32)
        # nearest-even rounding to the top 16 bits, as in f32_to_bf16_bits
        np.right_shift(u[:m], np.uint32(16), out=t[:m])
        np.bitwise_and(t[:m], np.uint32(1), out=t[:m])
        np.add(t[:m], np.uint32(0x7FFF), out=t[:m])
        np.add(t[:m], u[:m], out=t[:m])
        np.right_shift(t[:m], np.uint32(16), out=t[:m])
        out[s:s + m] = t[:m]
    return out.reshape(shape)


def uniform_bf16(gen: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return f32_to_bf16_bits(gen.uniform(lo, hi, size=shape).astype(np.float32))


@dataclasses.dataclass
class PagedKV:
    """A paged KV pool and the tables that address it.

    k_cache, v_cache: uint16 [num_pages, Hkv, P, D]
    block_table:      int32  [B, max_pages]
    context_lens:     int32  [B]  (history length, new token included)
    """

    k_cache: np.ndarray
    v_cache: np.ndarray
    block_table: np.ndarray
    context_lens: np.ndarray
    page_size: int

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def paged_kv(seed: int, context_lens, Hkv: int, D: int = 128, page_size: int = 16,
             max_pages: int | None = None, spare_pages: int = 1, fill_unused: str = "nan",
             stream_base: int = 100) -> PagedKV:
    """Random paged KV pool for sequences of the given context lengths.

    Every sequence owns ceil(T_b / P) physical pages taken from one shared
    pool in seeded random order; ``spare_pages`` extra pages belong to nobody.
    """
    ctx = np.asarray(context_lens, dtype=np.int64)
    B = ctx.size
    pages_per_seq = [int(math.ceil(t / page_size)) for t in ctx]
    if max_pages is None:
        max_pages = max(1, max(pages_per_seq) if B else 1)
    total = sum(pages_per_seq) + spare_pages
    perm = generator(seed, stream_base).permutation(total).astype(np.int32)
    table = np.full((B, max_pages), UNUSED_TABLE_ENTRY, dtype=np.int32)
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[cursor:cursor + n]
        cursor += n
    shape = (total, Hkv, page_size, D)
    k_cache = normal_bf16(generator(seed, stream_base + 1), shape)
    v_cache = normal_bf16(generator(seed, stream_base + 2), shape)
    if fill_unused == "nan":
        owned = np.zeros((total, page_size), dtype=bool)
        for b, n in enumerate(pages_per_seq):
            for lp in range(n):
                valid = min(page_size, int(ctx[b]) - lp * page_size)
                owned[table[b, lp], :valid] = True
        k_cache.transpose(0, 2, 1, 3)[~owned] = BF16_NAN
        v_cache.transpose(0, 2, 1, 3)[~owned] = BF16_NAN
    elif fill_unused != "normal":
        raise ValueError(fill_unused)
    return PagedKV(k_cache, v_cache, table, ctx.astype(np.int32), page_size)


@dataclasses.dataclass
class NewToken:
    """The decode step's new token for one layer: q [B,Hq,D], k/v [B,Hkv,D],
    RMSNorm gains gamma_q/gamma_k [D] (all bf16 bit patterns)."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    gamma_q: np.ndarray
    gamma_k: np.ndarray


def new_token(seed: int, B: int, Hq: int, Hkv: int, D: int = 128, stream_base: int = 10) -> NewToken:
    return NewToken(
        q=normal_bf16(generator(seed, stream_base), (B, Hq, D)),
        k=normal_bf16(generator(seed, stream_base + 1), (B, Hkv, D)),
        v=normal_bf16(generator(seed, stream_base + 2), (B, Hkv, D)),
        gamma_q=uniform_bf16(generator(seed, stream_base + 3), (D,), 0.5, 1.5),
        gamma_k=uniform_bf16(generator(seed, stream_base + 4), (D,), 0.5, 1.5),
    )


def query(seed: int, B: int, Hq: int, D: int = 128, stream: int = 20) -> np.ndarray:
    """A post-prologue query [B,Hq,D] for attention-only cases."""
    return normal_bf16(generator(seed, stream), (B, Hq, D))


def int8_rows(seed: int, shape, stream: int) -> np.ndarray:
    """Uniform int8 codes in [-127, 127] (an INT8 cache's rows for timing)."""
    return generator(seed, stream).integers(-127, 128, size=shape, dtype=np.int8)


def ragged_lengths(seed: int, B: int, lo: int, hi: int, stream: int = 30) -> np.ndarray:
    """Per-sequence context lengths ~ U[lo, hi] (integers, both ends included)."""
    return generator(seed, stream).integers(lo, hi + 1, size=B).astype(np.int32)


def scale_key_outliers(kv: PagedKV, seed: int, fraction: float, factor: float, stream: int = 40):
    """Multiply the keys at ceil(fraction * T) seeded positions of sequence 0 by
    ``factor`` (a power of two, so the bf16 product is exact), all KV heads.
    Returns the chosen positions. Used to stress the running-max rescale."""
    T = int(kv.context_lens[0])
    n = int(math.ceil(fraction * T))
    pos = np.sort(generator(seed, stream).choice(T, size=n, replace=False))
    exp_shift = int(round(math.log2(factor)))
    assert 2.0 ** exp_shift == factor, "factor must be a power of two"
    P = kv.page_size
    for p in pos:
        page = kv.block_table[0, p // P]
        rows = kv.k_cache[page, :, p % P, :]
        f = bf16_bits_to_f32(rows) * np.float32(factor)
        kv.k_cache[page, :, p % P, :] = f32_to_bf16_bits(f)
    return pos


def contiguous_kv(seed: int, B: int, T: int, Hkv: int, D: int = 128, stream_base: int = 50):
    """Unpaged history K, V laid out [B, T, Hkv, D] (host-tiled variant)."""
    k = normal_bf16(generator(seed, stream_base), (B, T, Hkv, D))
    v = normal_bf16(generator(seed, stream_base + 1), (B, T, Hkv, D))
    return k, v


# Named workloads: seed = 1000 + workload index.
WORKLOADS = {
    "tiny_t512": dict(seed=1000, B=1, Hq=16, Hkv=8, D=128, T=512, page_size=16, theta=1e6),
    "qwen3_0p6b_t8k": dict(seed=1001, layers=28, B=1, Hq=16, Hkv=8, D=128, T=8192, page_size=16,
                           theta=1e6),
    "ragged_b64": dict(seed=1002, B=64, Hq=16, Hkv=8, D=128, T_lo=1, T_hi=32768, page_size=16,
                       theta=1e6),
    "long_split_kv_t128k": dict(seed=1003, B=1, Hq=32, Hkv=8, D=128, T=131072, page_size=16,
                                partition=512, outlier_fraction=0.01, outlier_factor=8.0),
    "host_tiled_t64k": dict(seed=1004, B=1, Hq=16, Hkv=8, D=128, T=65536, tile=512),
    "qwen3_0p6b_t8k_int8": dict(seed=1006, layers=28, B=1, Hq=16, Hkv=8, D=128, T=8192, page_size=16, theta=1e6),
    "qwen3_0p6b_t8k_m4": dict(seed=1005, layers=28, B=1, M=4, Hq=16, Hkv=8, D=128, T=8192, page_size=16,
                              theta=1e6),
}


# ---------------------------------------------------------------- workload builders
def qwen3_layers(layers: int | None = None, T: int | None = None):
    """Qwen3-0.6B-shaped decode: per layer a paged cache of T positions
    (Hkv=8, D=128, P=16, random block table over its own pool) and a new token
    (Hq=16). Returns [(PagedKV, NewToken)] * layers."""
    w = WORKLOADS["qwen3_0p6b_t8k"]
    L = w["layers"] if layers is None else layers
    T = w["T"] if T is None else T
    out = []
    for i in range(L):
        seed = w["seed"] * 1000 + i
        kv = paged_kv(seed, [T] * w["B"], Hkv=w["Hkv"], D=w["D"], page_size=w["page_size"], spare_pages=0,
                      fill_unused="normal")
        tok = new_token(seed, w["B"], w["Hq"], w["Hkv"], w["D"])
        out.append((kv, tok))
    return out


def qwen3_layers_multi(layers: int | None = None):
    """Multi-token verification step: the Qwen3-0.6B-shaped 28-layer cache at
    T = 8192 (T counting the M = 4 new tokens), per layer M new tokens
    q [B,M,Hq,D], k, v [B,M,Hkv,D]. Returns [(PagedKV, q, k, v, gamma_q, gamma_k)]."""
    w = WORKLOADS["qwen3_0p6b_t8k_m4"]
    out = []
    for i in range(w["layers"] if layers is None else layers):
        seed = w["seed"] * 1000 + i
        kv = paged_kv(seed, [w["T"]] * w["B"], Hkv=w["Hkv"], D=w["D"], page_size=w["page_size"], spare_pages=0,
                      fill_unused="normal")
        g = generator(seed, 60)
        q = normal_bf16(g, (w["B"], w["M"], w["Hq"], w["D"]))
        k = normal_bf16(g, (w["B"], w["M"], w["Hkv"], w["D"]))
        v = normal_bf16(g, (w["B"], w["M"], w["Hkv"], w["D"]))
        tok = new_token(seed, w["B"], w["Hq"], w["Hkv"], w["D"])
        out.append((kv, q, k, v, tok.gamma_q, tok.gamma_k))
    return out


def ragged_b64(batch: int | None = None):
    """Batched ragged decode: B=64, T_b ~ U[1, 32768], one shared page pool.
    `batch` keeps only the first sequences of the same draw (a smaller case
    of the same workload, for profiling captures)."""
    w = WORKLOADS["ragged_b64"]
    ctx = ragged_lengths(w["seed"], w["B"], w["T_lo"], w["T_hi"])
    q = query(w["seed"], w["B"], w["Hq"], w["D"])
    if batch is not None:
        ctx, q = ctx[:batch], q[:batch]
    max_pages = (w["T_hi"] + w["page_size"] - 1) // w["page_size"]
    kv = paged_kv(w["seed"], ctx, Hkv=w["Hkv"], D=w["D"], page_size=w["page_size"], max_pages=max_pages,
                  fill_unused="normal")
    return kv, q


def long_split_kv():
    """Long-context split-KV: B=1, Hq=32, Hkv=8, T=131072, keys at 1% of the
    positions multiplied by 8 (written straight into the cache)."""
    w = WORKLOADS["long_split_kv_t128k"]
    kv = paged_kv(w["seed"], [w["T"]], Hkv=w["Hkv"], D=w["D"], page_size=w["page_size"], spare_pages=0,
                  fill_unused="normal")
    scale_key_outliers(kv, w["seed"], w["outlier_fraction"], w["outlier_factor"])
    q = query(w["seed"], w["B"], w["Hq"], w["D"])
    return kv, q


def host_tiled_kv():
    """Host-tiled offload: B=1, Hq=16, Hkv=8, T=65536 history [B, T, Hkv, D]."""
    w = WORKLOADS["host_tiled_t64k"]
    k, v = contiguous_kv(w["seed"], w["B"], w["T"], w["Hkv"], w["D"])
    q = query(w["seed"], w["B"], w["Hq"], w["D"])
    return q, k, v
