"""ctypes binding of libpgqa.so (include/pgqa.h), argument marshalling only.

Each function has the name of the C entry point it calls. It takes torch
tensors, checks their dtype/device/contiguity, passes raw pointers, sizes and
the current CUDA stream to the library, and raises PgqaError on a non-zero
status. Every step of the computation runs in the library's CUDA kernels;
there is no fallback of any kind: if the library cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libpgqa.so"
_lock = threading.Lock()
_lib = None

EXPORTED = (
    "pgqa_last_error",
    "pgqa_device_error",
    "pgqa_selftest_wait_timeout",
    "qk_norm_rope_append",
    "decode_attn_partition_count",
    "decode_attn_workspace_size",
    "decode_attn_paged",
    "decode_step_paged",
    "qk_norm_rope_append_multi",
    "decode_attn_multi_workspace_size",
    "decode_attn_paged_multi",
    "decode_step_paged_multi",
    "qk_norm_rope_append_int8",
    "decode_attn_int8_workspace_size",
    "decode_attn_paged_int8",
    "decode_step_paged_int8",
    "attn_partition_merge",
    "attn_tile_init",
    "attn_tile_update",
    "attn_tile_finalize",
    "attn_host_tiled_run",
    "attn_host_tiled_run_traced",
    "attn_host_direct_partition_count",
    "attn_host_direct_workspace_size",
    "attn_host_direct",
    "decode_attn_paged_static",
)

STATUS_NAMES = {
    0: "PGQA_OK",
    -1: "PGQA_ERR_INVALID_ARG",
    -2: "PGQA_ERR_UNSUPPORTED",
    -3: "PGQA_ERR_MISALIGNED",
    -4: "PGQA_ERR_WORKSPACE",
    -5: "PGQA_ERR_CUDA",
}

DEVERR_BAD_PAGE = 1
DEVERR_BAD_CONTEXT = 2
DEVERR_WAIT_TIMEOUT = 4


class PgqaError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load_library(path: str | None = None):
    """Load libpgqa.so (built by __graft_entry__.build()), or the library at
    `path` (the timeline build) on the first call; raise if missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or library_path()
        if not os.path.exists(path):
            raise PgqaError("load_library", -5, f"{path} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.pgqa_last_error.argtypes = []
        lib.pgqa_last_error.restype = ctypes.c_char_p
        lib.pgqa_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), I]
        lib.pgqa_device_error.restype = I
        lib.qk_norm_rope_append.argtypes = [P] * 10 + [I] * 7 + [F, F, P]
        lib.qk_norm_rope_append_multi.argtypes = [P] * 10 + [I] * 8 + [F, F, P]
        lib.qk_norm_rope_append_multi.restype = I
        lib.decode_attn_multi_workspace_size.argtypes = [I] * 8
        lib.decode_attn_multi_workspace_size.restype = S
        lib.decode_attn_paged_multi.argtypes = [P] * 5 + [I] * 8 + [F, I, P, P, P, S, P]
        lib.decode_attn_paged_multi.restype = I
        lib.decode_step_paged_multi.argtypes = [P] * 10 + [I] * 8 + [F, F, F, I, P, P, P, S, P]
        lib.decode_step_paged_multi.restype = I
        lib.qk_norm_rope_append_int8.argtypes = [P] * 12 + [I] * 7 + [F, F, P]
        lib.qk_norm_rope_append_int8.restype = I
        lib.decode_attn_int8_workspace_size.argtypes = [I] * 7
        lib.decode_attn_int8_workspace_size.restype = S
        lib.decode_attn_paged_int8.argtypes = [P] * 7 + [I] * 7 + [F, I, P, P, P, S, P]
        lib.decode_attn_paged_int8.restype = I
        lib.decode_step_paged_int8.argtypes = [P] * 12 + [I] * 7 + [F, F, F, I, P, P, P, S, P]
        lib.decode_step_paged_int8.restype = I
        lib.qk_norm_rope_append.restype = I
        lib.decode_attn_partition_count.argtypes = [I] * 5
        lib.decode_attn_partition_count.restype = I
        lib.decode_attn_workspace_size.argtypes = [I] * 7
        lib.decode_attn_workspace_size.restype = S
        lib.decode_attn_paged.argtypes = [P] * 5 + [I] * 7 + [F, I, P, P, P, S, P]
        lib.decode_attn_paged.restype = I
        lib.decode_step_paged.argtypes = [P] * 10 + [I] * 7 + [F, F, F, I, P, P, P, S, P]
        lib.decode_step_paged.restype = I
        lib.attn_partition_merge.argtypes = [P, P, P, I, I, I, I, P, P, P]
        lib.attn_partition_merge.restype = I
        lib.attn_tile_init.argtypes = [P, P, P, I, I, I, P]
        lib.attn_tile_init.restype = I
        lib.attn_tile_update.argtypes = [P, P, P, I, I, I, I, I, F, P, P, P, P]
        lib.attn_tile_update.restype = I
        lib.attn_tile_finalize.argtypes = [P, P, P, I, I, I, P, P, P]
        lib.attn_tile_finalize.restype = I
        lib.attn_host_tiled_run.argtypes = [P, P, P, I, I, I, I, I, F, I, I, I, P, P, P, P, P, P, P, P, P, P]
        lib.attn_host_tiled_run.restype = I
        lib.attn_host_tiled_run_traced.argtypes = [P, P, P, I, I, I, I, I, F, I, I, I, P, P, P, P, P, P, P, P, P, P,
                                                   P, I]
        lib.attn_host_tiled_run_traced.restype = I
        lib.attn_host_direct_partition_count.argtypes = [I, I, I, I]
        lib.attn_host_direct_partition_count.restype = I
        lib.attn_host_direct_workspace_size.argtypes = [I, I, I, I, I]
        lib.attn_host_direct_workspace_size.restype = S
        lib.attn_host_direct.argtypes = [P, P, P, I, I, I, I, I, F, I, P, P, P, S, P]
        lib.attn_host_direct.restype = I
        lib.pgqa_selftest_wait_timeout.argtypes = [P]
        lib.pgqa_selftest_wait_timeout.restype = I
        lib.decode_attn_paged_static.argtypes = [P] * 5 + [I] * 7 + [F, I, P, P, P]
        lib.decode_attn_paged_static.restype = I
        _lib = lib
        return lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        msg = load_library().pgqa_last_error().decode(errors="replace")
        raise PgqaError(fn, status, msg)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t, dtype, name, nullable=False):
    if t is None:
        if nullable:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _host(t, dtype, name):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CPU {dtype} tensor")
    if not t.is_pinned():
        raise ValueError(f"{name} must be in pinned host memory")
    return t.data_ptr()


def device_error_flags(clear: bool = True) -> int:
    """Sticky device-side flags (DEVERR_*) of the current device (synchronises)."""
    lib = load_library()
    v = ctypes.c_uint(0)
    _check("pgqa_device_error", lib.pgqa_device_error(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def qk_norm_rope_append(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache, v_cache, q_out,
                        page_size: int, rope_theta: float, eps: float = 1e-6, stream=None) -> None:
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    st = lib.qk_norm_rope_append(
        _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(gamma_q, bf, "gamma_q"),
        _dev(gamma_k, bf, "gamma_k"), _dev(context_lens, i32, "context_lens"),
        _dev(block_table, i32, "block_table"), _dev(k_cache, bf, "k_cache"), _dev(v_cache, bf, "v_cache"),
        _dev(q_out, bf, "q_out"), B, Hq, Hkv, D, page_size, block_table.shape[1], k_cache.shape[0],
        float(rope_theta), float(eps), _stream(stream))
    _check("qk_norm_rope_append", st)


def decode_attn_partition_count(B: int, Hkv: int, page_size: int, max_pages: int, num_partitions: int = 0) -> int:
    n = load_library().decode_attn_partition_count(B, Hkv, page_size, max_pages, num_partitions)
    if n < 1:
        _check("decode_attn_partition_count", n)
    return n


def decode_attn_workspace_size(B: int, Hq: int, Hkv: int, D: int, page_size: int, max_pages: int,
                               num_partitions: int = 0) -> int:
    return int(load_library().decode_attn_workspace_size(B, Hq, Hkv, D, page_size, max_pages, num_partitions))


def decode_attn_paged(q, k_cache, v_cache, block_table, context_lens, scale: float, out_f32=None, out_bf16=None,
                      workspace=None, num_partitions: int = 0, stream=None) -> None:
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    B, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_cache.shape
    ws_ptr = _dev(workspace, torch.uint8, "workspace", nullable=True)
    ws_bytes = workspace.numel() if workspace is not None else 0
    st = lib.decode_attn_paged(
        _dev(q, bf, "q"), _dev(k_cache, bf, "k_cache"), _dev(v_cache, bf, "v_cache"),
        _dev(block_table, i32, "block_table"), _dev(context_lens, i32, "context_lens"), B, Hq, Hkv, D, P,
        block_table.shape[1], num_pages, float(scale), int(num_partitions),
        _dev(out_f32, torch.float32, "out_f32", nullable=True), _dev(out_bf16, bf, "out_bf16", nullable=True),
        ws_ptr, ws_bytes, _stream(stream))
    _check("decode_attn_paged", st)


def qk_norm_rope_append_multi(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache, v_cache, q_out,
                              rope_theta: float, eps: float = 1e-6, stream=None) -> None:
    """Prologue for M new tokens per sequence: q [B, M, Hq, D], k/v [B, M, Hkv, D]."""
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    B, M, Hq, D = q.shape
    Hkv = k.shape[2]
    num_pages, _, P, _ = k_cache.shape
    st = lib.qk_norm_rope_append_multi(
        _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(gamma_q, bf, "gamma_q"),
        _dev(gamma_k, bf, "gamma_k"), _dev(context_lens, i32, "context_lens"),
        _dev(block_table, i32, "block_table"), _dev(k_cache, bf, "k_cache"), _dev(v_cache, bf, "v_cache"),
        _dev(q_out, bf, "q_out"), B, M, Hq, Hkv, D, P, block_table.shape[1], num_pages,
        float(rope_theta), float(eps), _stream(stream))
    _check("qk_norm_rope_append_multi", st)


def decode_attn_multi_workspace_size(B: int, M: int, Hq: int, Hkv: int, D: int, page_size: int, max_pages: int,
                                     num_partitions: int = 0) -> int:
    return int(load_library().decode_attn_multi_workspace_size(B, M, Hq, Hkv, D, page_size, max_pages,
                                                                num_partitions))


def decode_attn_paged_multi(q, k_cache, v_cache, block_table, context_lens, scale: float, out_f32=None,
                            out_bf16=None, workspace=None, num_partitions: int = 0, stream=None) -> None:
    """Attention for M new tokens per sequence: q and outputs [B, M, Hq, D]."""
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    B, M, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_cache.shape
    ws_ptr = _dev(workspace, torch.uint8, "workspace", nullable=True)
    ws_bytes = workspace.numel() if workspace is not None else 0
    st = lib.decode_attn_paged_multi(
        _dev(q, bf, "q"), _dev(k_cache, bf, "k_cache"), _dev(v_cache, bf, "v_cache"),
        _dev(block_table, i32, "block_table"), _dev(context_lens, i32, "context_lens"), B, M, Hq, Hkv, D, P,
        block_table.shape[1], num_pages, float(scale), int(num_partitions),
        _dev(out_f32, torch.float32, "out_f32", nullable=True), _dev(out_bf16, bf, "out_bf16", nullable=True),
        ws_ptr, ws_bytes, _stream(stream))
    _check("decode_attn_paged_multi", st)


def decode_step_paged_multi(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache, v_cache, scale: float,
                            rope_theta: float, eps: float = 1e-6, q_out=None, out_f32=None, out_bf16=None,
                            workspace=None, num_partitions: int = 0, stream=None) -> None:
    """Fused multi-token step: q [B, M, Hq, D], k/v [B, M, Hkv, D], outputs [B, M, Hq, D]."""
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    B, M, Hq, D = q.shape
    Hkv = k.shape[2]
    num_pages, _, P, _ = k_cache.shape
    ws_ptr = _dev(workspace, torch.uint8, "workspace", nullable=True)
    ws_bytes = workspace.numel() if workspace is not None else 0
    st = lib.decode_step_paged_multi(
        _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(gamma_q, bf, "gamma_q"),
        _dev(gamma_k, bf, "gamma_k"), _dev(context_lens, i32, "context_lens"), _dev(block_table, i32, "block_table"),
        _dev(k_cache, bf, "k_cache"), _dev(v_cache, bf, "v_cache"), _dev(q_out, bf, "q_out", nullable=True), B, M,
        Hq, Hkv, D, P, block_table.shape[1], num_pages, float(rope_theta), float(eps), float(scale),
        int(num_partitions), _dev(out_f32, torch.float32, "out_f32", nullable=True),
        _dev(out_bf16, bf, "out_bf16", nullable=True), ws_ptr, ws_bytes, _stream(stream))
    _check("decode_step_paged_multi", st)


def qk_norm_rope_append_int8(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache8, v_cache8, k_scale,
                             v_scale, q_out, rope_theta: float, eps: float = 1e-6, stream=None) -> None:
    """Prologue writing the new K/V rows into an INT8 cache (codes [pages, Hkv, P, D] int8, scales
    [pages, Hkv, P] float32)."""
    lib = load_library()
    bf, i32, i8, f32 = torch.bfloat16, torch.int32, torch.int8, torch.float32
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    num_pages, _, P, _ = k_cache8.shape
    st = lib.qk_norm_rope_append_int8(
        _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(gamma_q, bf, "gamma_q"),
        _dev(gamma_k, bf, "gamma_k"), _dev(context_lens, i32, "context_lens"), _dev(block_table, i32, "block_table"),
        _dev(k_cache8, i8, "k_cache8"), _dev(v_cache8, i8, "v_cache8"), _dev(k_scale, f32, "k_scale"),
        _dev(v_scale, f32, "v_scale"), _dev(q_out, bf, "q_out"), B, Hq, Hkv, D, P, block_table.shape[1], num_pages,
        float(rope_theta), float(eps), _stream(stream))
    _check("qk_norm_rope_append_int8", st)


def decode_attn_int8_workspace_size(B: int, Hq: int, Hkv: int, D: int, page_size: int, max_pages: int,
                                    num_partitions: int = 0) -> int:
    return int(load_library().decode_attn_int8_workspace_size(B, Hq, Hkv, D, page_size, max_pages, num_partitions))


def decode_attn_paged_int8(q, k_cache8, v_cache8, k_scale, v_scale, block_table, context_lens, scale: float,
                           out_f32=None, out_bf16=None, workspace=None, num_partitions: int = 0, stream=None) -> None:
    """Decode attention over an INT8 cache."""
    lib = load_library()
    bf, i32, i8, f32 = torch.bfloat16, torch.int32, torch.int8, torch.float32
    B, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_cache8.shape
    ws_ptr = _dev(workspace, torch.uint8, "workspace", nullable=True)
    ws_bytes = workspace.numel() if workspace is not None else 0
    st = lib.decode_attn_paged_int8(
        _dev(q, bf, "q"), _dev(k_cache8, i8, "k_cache8"), _dev(v_cache8, i8, "v_cache8"), _dev(k_scale, f32, "k_scale"),
        _dev(v_scale, f32, "v_scale"), _dev(block_table, i32, "block_table"), _dev(context_lens, i32, "context_lens"),
        B, Hq, Hkv, D, P, block_table.shape[1], num_pages, float(scale), int(num_partitions),
        _dev(out_f32, f32, "out_f32", nullable=True), _dev(out_bf16, bf, "out_bf16", nullable=True), ws_ptr, ws_bytes,
        _stream(stream))
    _check("decode_attn_paged_int8", st)


def decode_step_paged_int8(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache8, v_cache8, k_scale,
                           v_scale, scale: float, rope_theta: float, eps: float = 1e-6, q_out=None, out_f32=None,
                           out_bf16=None, workspace=None, num_partitions: int = 0, stream=None) -> None:
    """Fused qk_norm_rope_append_int8 + decode_attn_paged_int8 for one layer (one launch)."""
    lib = load_library()
    bf, i32, i8, f32 = torch.bfloat16, torch.int32, torch.int8, torch.float32
    B, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_cache8.shape
    ws_ptr = _dev(workspace, torch.uint8, "workspace", nullable=True)
    ws_bytes = workspace.numel() if workspace is not None else 0
    st = lib.decode_step_paged_int8(
        _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(gamma_q, bf, "gamma_q"),
        _dev(gamma_k, bf, "gamma_k"), _dev(context_lens, i32, "context_lens"), _dev(block_table, i32, "block_table"),
        _dev(k_cache8, i8, "k_cache8"), _dev(v_cache8, i8, "v_cache8"), _dev(k_scale, f32, "k_scale"),
        _dev(v_scale, f32, "v_scale"), _dev(q_out, bf, "q_out", nullable=True), B, Hq, Hkv, D, P,
        block_table.shape[1], num_pages, float(rope_theta), float(eps), float(scale), int(num_partitions),
        _dev(out_f32, f32, "out_f32", nullable=True), _dev(out_bf16, bf, "out_bf16", nullable=True), ws_ptr, ws_bytes,
        _stream(stream))
    _check("decode_step_paged_int8", st)


def decode_step_paged(q, k, v, gamma_q, gamma_k, context_lens, block_table, k_cache, v_cache, scale: float,
                      rope_theta: float, eps: float = 1e-6, q_out=None, out_f32=None, out_bf16=None, workspace=None,
                      num_partitions: int = 0, stream=None) -> None:
    """Fused qk_norm_rope_append + decode_attn_paged for one layer (one launch)."""
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    B, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_cache.shape
    ws_ptr = _dev(workspace, torch.uint8, "workspace", nullable=True)
    ws_bytes = workspace.numel() if workspace is not None else 0
    st = lib.decode_step_paged(
        _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(gamma_q, bf, "gamma_q"),
        _dev(gamma_k, bf, "gamma_k"), _dev(context_lens, i32, "context_lens"), _dev(block_table, i32, "block_table"),
        _dev(k_cache, bf, "k_cache"), _dev(v_cache, bf, "v_cache"), _dev(q_out, bf, "q_out", nullable=True), B, Hq,
        Hkv, D, P, block_table.shape[1], num_pages, float(rope_theta), float(eps), float(scale), int(num_partitions),
        _dev(out_f32, torch.float32, "out_f32", nullable=True), _dev(out_bf16, bf, "out_bf16", nullable=True),
        ws_ptr, ws_bytes, _stream(stream))
    _check("decode_step_paged", st)


def attn_partition_merge(m, l, acc, out_f32=None, out_bf16=None, stream=None) -> None:
    lib = load_library()
    B, Hq, NP, D = acc.shape
    f32 = torch.float32
    st = lib.attn_partition_merge(
        _dev(m, f32, "m"), _dev(l, f32, "l"), _dev(acc, f32, "acc"), B, Hq, D, NP,
        _dev(out_f32, f32, "out_f32", nullable=True), _dev(out_bf16, torch.bfloat16, "out_bf16", nullable=True),
        _stream(stream))
    _check("attn_partition_merge", st)


def attn_tile_init(m, l, acc, stream=None) -> None:
    lib = load_library()
    B, Hq, D = acc.shape
    f32 = torch.float32
    _check("attn_tile_init", lib.attn_tile_init(_dev(m, f32, "m"), _dev(l, f32, "l"), _dev(acc, f32, "acc"),
                                                B, Hq, D, _stream(stream)))


def attn_tile_update(q, k_tile, v_tile, m, l, acc, scale: float, n_pos: int | None = None, stream=None) -> None:
    lib = load_library()
    B, Hq, D = q.shape
    _, tile_len, Hkv, _ = k_tile.shape
    n = tile_len if n_pos is None else int(n_pos)
    f32, bf = torch.float32, torch.bfloat16
    st = lib.attn_tile_update(_dev(q, bf, "q"), _dev(k_tile, bf, "k_tile"), _dev(v_tile, bf, "v_tile"), n, B, Hq,
                              Hkv, D, float(scale), _dev(m, f32, "m"), _dev(l, f32, "l"), _dev(acc, f32, "acc"),
                              _stream(stream))
    _check("attn_tile_update", st)


def attn_tile_finalize(m, l, acc, out_f32=None, out_bf16=None, stream=None) -> None:
    lib = load_library()
    B, Hq, D = acc.shape
    f32 = torch.float32
    st = lib.attn_tile_finalize(_dev(m, f32, "m"), _dev(l, f32, "l"), _dev(acc, f32, "acc"), B, Hq, D,
                                _dev(out_f32, f32, "out_f32", nullable=True),
                                _dev(out_bf16, torch.bfloat16, "out_bf16", nullable=True), _stream(stream))
    _check("attn_tile_finalize", st)


def attn_host_tiled_run(q, host_k, host_v, scale: float, k_slots, v_slots, events, m, l, acc, out_f32=None,
                        out_bf16=None, tile_len: int = 512, tiles_per_copy: int = 1, compute_stream=None,
                        copy_stream=None, trace_events=None) -> None:
    """host_k/host_v: pinned CPU bf16 [B, T, Hkv, D]; k_slots/v_slots: lists of device
    [B, tiles_per_copy * tile_len, Hkv, D] buffers; events: 2*len(k_slots) torch.cuda.Event objects.
    trace_events (optional): 4 * G torch.cuda.Event(enable_timing=True) objects, recorded around
    the first G copy groups (attn_host_tiled_run_traced)."""
    lib = load_library()
    bf, f32 = torch.bfloat16, torch.float32
    B, Hq, D = q.shape
    _, T, Hkv, _ = host_k.shape
    n = len(k_slots)
    if len(v_slots) != n or len(events) != 2 * n:
        raise ValueError("need equally many K and V slots and 2 events per slot")
    kp = (ctypes.c_void_p * n)(*[_dev(t, bf, "k_slot") for t in k_slots])
    vp = (ctypes.c_void_p * n)(*[_dev(t, bf, "v_slot") for t in v_slots])
    for ev in events:
        if ev.cuda_event == 0:
            ev.record()  # materialise the lazily created torch event
    ep = (ctypes.c_void_p * (2 * n))(*[ev.cuda_event for ev in events])
    if copy_stream is None:
        raise ValueError("copy_stream is required (a stream other than the compute stream)")
    args = (_dev(q, bf, "q"), _host(host_k, bf, "host_k"), _host(host_v, bf, "host_v"), T, B, Hq, Hkv, D,
            float(scale), int(tile_len), int(tiles_per_copy), n, ctypes.cast(kp, ctypes.c_void_p),
            ctypes.cast(vp, ctypes.c_void_p), ctypes.cast(ep, ctypes.c_void_p), _dev(m, f32, "m"),
            _dev(l, f32, "l"), _dev(acc, f32, "acc"), _dev(out_f32, f32, "out_f32", nullable=True),
            _dev(out_bf16, bf, "out_bf16", nullable=True), _stream(compute_stream), _stream(copy_stream))
    if trace_events is None:
        _check("attn_host_tiled_run", lib.attn_host_tiled_run(*args))
        return
    if len(trace_events) % 4:
        raise ValueError("trace_events: 4 events per traced copy group")
    for ev in trace_events:
        if ev.cuda_event == 0:
            ev.record()  # materialise the lazily created torch event
    tp = (ctypes.c_void_p * max(1, len(trace_events)))(*[ev.cuda_event for ev in trace_events])
    _check("attn_host_tiled_run_traced",
           lib.attn_host_tiled_run_traced(*args, ctypes.cast(tp, ctypes.c_void_p), len(trace_events) // 4))


def attn_host_direct_partition_count(B: int, Hkv: int, T: int, num_partitions: int = 0) -> int:
    n = load_library().attn_host_direct_partition_count(B, Hkv, T, num_partitions)
    if n < 0:
        _check("attn_host_direct_partition_count", n)
    return n


def attn_host_direct_workspace_size(B: int, Hq: int, Hkv: int, T: int, num_partitions: int = 0) -> int:
    return int(load_library().attn_host_direct_workspace_size(B, Hq, Hkv, T, num_partitions))


def attn_host_direct(q, host_k, host_v, scale: float, out_f32=None, out_bf16=None, workspace=None,
                     num_partitions: int = 0, stream=None) -> None:
    """Zero-copy attention over a history in pinned host memory.

    q: device bf16 [B, Hq, D]; host_k/host_v: pinned CPU bf16 [B, T, Hkv, D]."""
    lib = load_library()
    bf = torch.bfloat16
    B, Hq, D = q.shape
    Bk, T, Hkv, Dk = host_k.shape
    if tuple(host_v.shape) != tuple(host_k.shape) or Bk != B or Dk != D:
        raise ValueError("attn_host_direct: host_k and host_v must both be [B, T, Hkv, D]")
    ws_ptr = _dev(workspace, torch.uint8, "workspace", nullable=True)
    ws_bytes = workspace.numel() if workspace is not None else 0
    hk = _host(host_k, bf, "host_k") if T > 0 else None
    hv = _host(host_v, bf, "host_v") if T > 0 else None
    st = lib.attn_host_direct(_dev(q, bf, "q"), hk, hv, T, B, Hq,
                              Hkv, D, float(scale), int(num_partitions),
                              _dev(out_f32, torch.float32, "out_f32", nullable=True),
                              _dev(out_bf16, bf, "out_bf16", nullable=True), ws_ptr, ws_bytes, _stream(stream))
    _check("attn_host_direct", st)


def selftest_wait_timeout(stream=None) -> None:
    """Run the bounded-wait self-test kernel (raises DEVERR_WAIT_TIMEOUT on the device)."""
    _check("pgqa_selftest_wait_timeout", load_library().pgqa_selftest_wait_timeout(_stream(stream)))


STATIC_SCRATCH_BYTES = 8 << 20  # PGQA_STATIC_SCRATCH_BYTES in include/pgqa.h


def decode_attn_paged_static(q, k_cache, v_cache, block_table, context_lens, scale: float, out_f32=None,
                             out_bf16=None, num_partitions: int = 0, stream=None) -> None:
    """decode_attn_paged without a workspace, for callers that cannot allocate:
    the partition scratch is the library's built-in array (see include/pgqa.h)."""
    lib = load_library()
    bf, i32 = torch.bfloat16, torch.int32
    B, Hq, D = q.shape
    num_pages, Hkv, P, _ = k_cache.shape
    st = lib.decode_attn_paged_static(
        _dev(q, bf, "q"), _dev(k_cache, bf, "k_cache"), _dev(v_cache, bf, "v_cache"),
        _dev(block_table, i32, "block_table"), _dev(context_lens, i32, "context_lens"), B, Hq, Hkv, D, P,
        block_table.shape[1], num_pages, float(scale), int(num_partitions),
        _dev(out_f32, torch.float32, "out_f32", nullable=True), _dev(out_bf16, bf, "out_bf16", nullable=True),
        _stream(stream))
    _check("decode_attn_paged_static", st)
