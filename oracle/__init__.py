"""fp64 CPU oracle of the paged GQA decode step (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library and its Python binding
never import it, and it imports nothing from them.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
compiles it with gcc on first use and marshals numpy arrays to it through
ctypes. bf16 tensors travel as ``uint16`` bit patterns, index tensors as
``int32``. Each wrapper names the section of the pages its C routine follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, -O2, IEEE semantics)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_long
        D = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = D
        lib.oracle_round_bf16.argtypes = [D]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_head_rmsnorm.argtypes = [P, P, I, D, P]
        lib.oracle_head_rmsnorm.restype = None
        lib.oracle_rope_half.argtypes = [P, I, L, D, P]
        lib.oracle_rope_half.restype = None
        lib.oracle_kv_head.argtypes = [I, I, I]
        lib.oracle_kv_head.restype = I
        lib.oracle_cache_offset.argtypes = [P, I, I, I, I, L, I, I, I]
        lib.oracle_cache_offset.restype = L
        lib.oracle_qk_norm_rope_append.argtypes = [P] * 10 + [I] * 7 + [D, D]
        lib.oracle_qk_norm_rope_append.restype = I
        lib.oracle_decode_attention.argtypes = [P] * 5 + [I] * 7 + [D, P]
        lib.oracle_quantize_row_int8.argtypes = [P, I, P, P]
        lib.oracle_quantize_row_int8.restype = None
        lib.oracle_quantize_rows_int8.argtypes = [P, L, I, P, P]
        lib.oracle_quantize_rows_int8.restype = None
        lib.oracle_dequant_int8.argtypes = [ctypes.c_int8, ctypes.c_float]
        lib.oracle_dequant_int8.restype = D
        lib.oracle_qk_norm_rope_append_int8.argtypes = [P] * 12 + [I] * 7 + [D, D]
        lib.oracle_qk_norm_rope_append_int8.restype = I
        lib.oracle_decode_attention_int8.argtypes = [P] * 7 + [I] * 7 + [D, P]
        lib.oracle_decode_attention_int8.restype = I
        lib.oracle_decode_attention_multi.argtypes = [P] * 5 + [I] * 8 + [D, P]
        lib.oracle_decode_attention_multi.restype = I
        lib.oracle_qk_norm_rope_append_multi.argtypes = [P] * 10 + [I] * 8 + [D, D]
        lib.oracle_qk_norm_rope_append_multi.restype = I
        lib.oracle_decode_attention.restype = I
        lib.oracle_attention_contiguous.argtypes = [P, P, P, I, L, I, I, I, D, P]
        lib.oracle_attention_contiguous.restype = I
        lib.oracle_state_init.argtypes = [I, P, P, P]
        lib.oracle_state_init.restype = None
        lib.oracle_state_update.argtypes = [P, P, L, I, P, P, P]
        lib.oracle_state_update.restype = None
        lib.oracle_state_finalize.argtypes = [D, P, I, P]
        lib.oracle_state_finalize.restype = None
        lib.oracle_merge_partitions.argtypes = [P, P, P, I, I, P]
        lib.oracle_merge_partitions.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"bf16 bit patterns expected, got {a.dtype}"
    return a


def _i32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.int32, f"int32 expected, got {a.dtype}"
    return a


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


class OracleError(RuntimeError):
    pass


def _check(status: int, what: str) -> None:
    if status != 0:
        raise OracleError(f"{what}: oracle status {status}")


# --------------------------------------------------------------------------
# storage type (bf16-as-storage note; Qwen3 runtime s0.1)
# --------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns to float64, exactly."""
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    flat = b.reshape(-1)
    out = np.fromiter((lib.oracle_bf16_to_double(int(x)) for x in flat), dtype=np.float64, count=flat.size)
    return out.reshape(b.shape)


def round_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (nearest, ties to even)."""
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    flat = a.reshape(-1)
    out = np.fromiter((lib.oracle_round_bf16(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(a.shape)


# --------------------------------------------------------------------------
# A3, A4, A5, A7 building blocks
# --------------------------------------------------------------------------
def head_rmsnorm(x, gamma, eps: float = 1e-6) -> np.ndarray:
    """Per-head RMSNorm (Qwen3 runtime s2.1 / s2.3) of one D-vector."""
    lib = _load()
    x = _f64(x)
    g = _f64(gamma)
    out = np.empty_like(x)
    lib.oracle_head_rmsnorm(_ptr(x), _ptr(g), x.size, float(eps), _ptr(out))
    return out


def rope_half(x, pos: int, theta: float) -> np.ndarray:
    """Half-rotation RoPE (Qwen3 runtime s2.4) of one D-vector at position pos."""
    lib = _load()
    x = _f64(x)
    out = np.empty_like(x)
    lib.oracle_rope_half(_ptr(x), x.size, int(pos), float(theta), _ptr(out))
    return out


def kv_head(h: int, Hq: int, Hkv: int) -> int:
    """GQA head map (Qwen3 runtime s2.5)."""
    return int(_load().oracle_kv_head(h, Hq, Hkv))


def cache_offset(block_table, b: int, kvh: int, pos: int, Hkv: int, P: int, D: int, num_pages: int) -> int:
    """Element offset of (b, kvh, pos) in a [num_pages][Hkv][P][D] cache (s7.2)."""
    bt = _i32(block_table)
    max_pages = bt.shape[-1]
    return int(_load().oracle_cache_offset(_ptr(bt), max_pages, num_pages, b, kvh, int(pos), Hkv, P, D))


# --------------------------------------------------------------------------
# prologue and attention
# --------------------------------------------------------------------------
def qk_norm_rope_append(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache, v_cache,
                        page_size: int, rope_theta: float, eps: float = 1e-6):
    """Fused prologue (s2.3 + s2.4 + s7.2). Returns (q_out, k_cache', v_cache').

    q: u16 [B,Hq,D]; k, v: u16 [B,Hkv,D]; gammas u16 [D]; context_lens i32 [B];
    block_table i32 [B,max_pages]; caches u16 [num_pages,Hkv,P,D] (copied, not
    modified in place)."""
    lib = _load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    gq, gk = _u16(gamma_q), _u16(gamma_k)
    ctx, bt = _i32(context_lens), _i32(block_table)
    kc = _u16(k_cache).copy()
    vc = _u16(v_cache).copy()
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    q_out = np.zeros_like(q)
    st = lib.oracle_qk_norm_rope_append(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ctx), _ptr(bt), _ptr(kc), _ptr(vc),
        _ptr(q_out), B, Hq, Hkv, D, page_size, bt.shape[1], kc.shape[0], float(rope_theta), float(eps))
    _check(st, "qk_norm_rope_append")
    return q_out, kc, vc


def decode_attention(q, k_cache, v_cache, block_table, context_lens, scale: float) -> np.ndarray:
    """Direct-softmax decode attention over the paged cache (s2.5, s2.6, s7.2).

    Returns float64 [B, Hq, D]."""
    lib = _load()
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, ctx = _i32(block_table), _i32(context_lens)
    B, Hq, D = q.shape
    num_pages, Hkv, P, D2 = kc.shape
    assert D2 == D
    out = np.zeros((B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_attention(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(ctx), B, Hq, Hkv, D, P,
                                     bt.shape[1], num_pages, float(scale), _ptr(out))
    _check(st, "decode_attention")
    return out


def qk_norm_rope_append_multi(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache, v_cache,
                              page_size: int, rope_theta: float, eps: float = 1e-6):
    """Prologue for M new tokens per sequence at positions T-M .. T-1.

    q: u16 [B,M,Hq,D]; k, v: u16 [B,M,Hkv,D]. Returns (q_out [B,M,Hq,D], k_cache', v_cache')."""
    lib = _load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    gq, gk = _u16(gamma_q), _u16(gamma_k)
    ctx, bt = _i32(context_lens), _i32(block_table)
    kc = _u16(k_cache).copy()
    vc = _u16(v_cache).copy()
    B, M, Hq, D = q.shape
    Hkv = k.shape[2]
    q_out = np.zeros_like(q)
    st = lib.oracle_qk_norm_rope_append_multi(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ctx), _ptr(bt), _ptr(kc), _ptr(vc),
        _ptr(q_out), B, M, Hq, Hkv, D, page_size, bt.shape[1], kc.shape[0], float(rope_theta), float(eps))
    _check(st, "qk_norm_rope_append_multi")
    return q_out, kc, vc


def decode_attention_multi(q, k_cache, v_cache, block_table, context_lens, scale: float) -> np.ndarray:
    """Multi-query decode attention: token i of M (q [B,M,Hq,D]) attends causally to
    positions 0 .. T-M+i. Returns float64 [B, M, Hq, D]."""
    lib = _load()
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, ctx = _i32(block_table), _i32(context_lens)
    B, M, Hq, D = q.shape
    num_pages, Hkv, P, D2 = kc.shape
    assert D2 == D
    out = np.zeros((B, M, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_attention_multi(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(ctx), B, M, Hq, Hkv, D,
                                           P, bt.shape[1], num_pages, float(scale), _ptr(out))
    _check(st, "decode_attention_multi")
    return out


def quantize_rows_int8(rows):
    """Symmetric per-row INT8 quantization of bf16 rows [..., D] (u16 bits).

    Returns (codes int8 [..., D], scales float32 [...])."""
    rows = _u16(rows)
    D = rows.shape[-1]
    n = rows.size // D
    codes = np.zeros(rows.shape, dtype=np.int8)
    scales = np.zeros(rows.shape[:-1], dtype=np.float32)
    _load().oracle_quantize_rows_int8(_ptr(rows), n, D, _ptr(codes), _ptr(scales))
    return codes, scales


def dequantize_int8(codes, scales) -> np.ndarray:
    """codes * scale per row, float64 (exact)."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def qk_norm_rope_append_int8(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache8, v_cache8, k_scale,
                             v_scale, page_size: int, rope_theta: float, eps: float = 1e-6):
    """Prologue with an INT8 cache. Returns (q_out, k_cache8', v_cache8', k_scale', v_scale') (copies)."""
    lib = _load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    gq, gk = _u16(gamma_q), _u16(gamma_k)
    ctx, bt = _i32(context_lens), _i32(block_table)
    kc = np.ascontiguousarray(k_cache8, dtype=np.int8).copy()
    vc = np.ascontiguousarray(v_cache8, dtype=np.int8).copy()
    ks = np.ascontiguousarray(k_scale, dtype=np.float32).copy()
    vs = np.ascontiguousarray(v_scale, dtype=np.float32).copy()
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    q_out = np.zeros_like(q)
    st = lib.oracle_qk_norm_rope_append_int8(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gq), _ptr(gk), _ptr(ctx), _ptr(bt), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
        _ptr(q_out), B, Hq, Hkv, D, page_size, bt.shape[1], kc.shape[0], float(rope_theta), float(eps))
    _check(st, "qk_norm_rope_append_int8")
    return q_out, kc, vc, ks, vs


def decode_attention_int8(q, k_cache8, v_cache8, k_scale, v_scale, block_table, context_lens,
                          scale: float) -> np.ndarray:
    """Direct-softmax decode attention over an INT8 cache (dequantized rows). float64 [B, Hq, D]."""
    lib = _load()
    q = _u16(q)
    kc = np.ascontiguousarray(k_cache8, dtype=np.int8)
    vc = np.ascontiguousarray(v_cache8, dtype=np.int8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    bt, ctx = _i32(block_table), _i32(context_lens)
    B, Hq, D = q.shape
    num_pages, Hkv, P, _ = kc.shape
    out = np.zeros((B, Hq, D), dtype=np.float64)
    st = lib.oracle_decode_attention_int8(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(ctx), B,
                                          Hq, Hkv, D, P, bt.shape[1], num_pages, float(scale), _ptr(out))
    _check(st, "decode_attention_int8")
    return out


def attention_contiguous(q, k, v, scale: float) -> np.ndarray:
    """Direct-softmax decode attention over k, v laid out [B, T, Hkv, D]."""
    lib = _load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, D = q.shape
    _, T, Hkv, _ = k.shape
    out = np.zeros((B, Hq, D), dtype=np.float64)
    st = lib.oracle_attention_contiguous(_ptr(q), _ptr(k), _ptr(v), B, T, Hq, Hkv, D, float(scale), _ptr(out))
    _check(st, "attention_contiguous")
    return out


# --------------------------------------------------------------------------
# A1 online state and A2 merge
# --------------------------------------------------------------------------
def state_init(D: int):
    """(m, l, acc) = (-1e30, 0, 0) (KV-offload design, attn_init)."""
    lib = _load()
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(D)
    lib.oracle_state_init(D, _ptr(m), _ptr(l), _ptr(acc))
    return float(m[0]), float(l[0]), acc


def state_update(state, scores, values):
    """Fold keys one at a time into (m, l, acc) (online-softmax update step)."""
    lib = _load()
    m0, l0, acc0 = state
    s = _f64(scores)
    vals = _f64(values)
    n = s.size
    D = acc0.size
    assert vals.shape == (n, D)
    m = np.array([m0], dtype=np.float64)
    l = np.array([l0], dtype=np.float64)
    acc = _f64(acc0).copy()
    lib.oracle_state_update(_ptr(s), _ptr(vals), n, D, _ptr(m), _ptr(l), _ptr(acc))
    return float(m[0]), float(l[0]), acc


def state_finalize(state) -> np.ndarray:
    lib = _load()
    _, l, acc = state
    acc = _f64(acc)
    out = np.empty_like(acc)
    lib.oracle_state_finalize(float(l), _ptr(acc), acc.size, _ptr(out))
    return out


def merge_partitions(m, l, acc) -> np.ndarray:
    """Exact merge of partition states (s9.1). m, l: [NP]; acc: [NP, D] -> [D]."""
    lib = _load()
    m, l, acc = _f64(m), _f64(l), _f64(acc)
    NP, D = acc.shape
    out = np.empty(D)
    lib.oracle_merge_partitions(_ptr(m), _ptr(l), _ptr(acc), NP, D, _ptr(out))
    return out


def merge_partitions_batched(m, l, acc) -> np.ndarray:
    """Merge per (b, h): m, l [B, H, NP]; acc [B, H, NP, D] -> [B, H, D] float64."""
    m, l, acc = _f64(m), _f64(l), _f64(acc)
    B, H, NP, D = acc.shape
    out = np.empty((B, H, D))
    for b in range(B):
        for h in range(H):
            out[b, h] = merge_partitions(m[b, h], l[b, h], acc[b, h])
    return out


def tiled_state_reference(q, k, v, scale: float, tile: int):
    """State (m, l, acc) after folding [B,T,Hkv,D] keys tile by tile with the
    online update, starting from state_init. Returns m, l [B,Hq]; acc [B,Hq,D]."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, D = q.shape
    _, T, Hkv, _ = k.shape
    qd = bf16_widen(q)
    kd = bf16_widen(k)
    vd = bf16_widen(v)
    m = np.zeros((B, Hq))
    l = np.zeros((B, Hq))
    acc = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            kvh = kv_head(h, Hq, Hkv)
            st = state_init(D)
            for t0 in range(0, T, tile):
                keys = kd[b, t0:t0 + tile, kvh]
                vals = vd[b, t0:t0 + tile, kvh]
                scores = scale * (keys @ qd[b, h])
                st = state_update(st, scores, vals)
            m[b, h], l[b, h], acc[b, h] = st
    return m, l, acc


def bf16_widen(bits) -> np.ndarray:
    """Vectorised exact bf16 -> float64 widening (bits on top of a binary32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
