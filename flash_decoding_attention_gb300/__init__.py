"""Python binding of libfdattn.so, the GB300 flash-decoding C-ABI library.

The functions named ``fd_*`` mirror the C entry points of
``include/fd_attention.h`` one to one and only marshal arguments (torch
tensors to device pointers, torch streams and events to handles); every step
of the computation runs in the library's CUDA kernels.  ``decode_attention``
is a convenience wrapper that also allocates the output, the LSE and the
workspace with torch.

The library must have been built (``flash_decoding_attention_gb300.build``);
loading fails loudly when it is missing, and there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

from . import build as _build_mod

LIB_PATH = _build_mod.LIB_PATH

FD_OK = 0
FD_ERR_INVALID_ARG = 1
FD_ERR_UNSUPPORTED = 2
FD_ERR_WORKSPACE_TOO_SMALL = 3
FD_ERR_CUDA = 4
FD_ERR_DEVICE_BOUNDS = 5
FD_ERR_DEVICE_TIMEOUT = 6

FD_F16 = 0
FD_BF16 = 1
FD_E4M3 = 2
FD_I8 = 3

# element format names used by the input generators -> fd_dtype codes
DTYPE_CODES = {"f16": FD_F16, "bf16": FD_BF16, "e4m3": FD_E4M3, "i8": FD_I8}

FD_KERNEL_AUTO = 0
FD_KERNEL_SIMT = 1
FD_KERNEL_MMA = 2
FD_KERNEL_TC = 3
FD_KERNEL_FMA = 4

FD_SCALE_TENSOR = 0
FD_SCALE_HEAD = 1
FD_SCALE_TOKEN = 2

EXPORTED = [
    "fd_workspace_bytes", "fd_decode_attention", "fd_check_device_error", "fd_status_string",
    "fd_set_kernel", "fd_selected_kernel", "fd_selected_kernel_scaled", "fd_set_split_events",
    "fd_debug_read_plan",
    "fd_debug_gather_kv", "fd_decode_attention_noalloc", "fd_decode_attention_scaled",
    "fd_append_kv", "fd_decode_attention_append", "fd_decode_attention_multi",
    "fd_debug_set_wait_limit", "fd_debug_plan_segments",
]


class FdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fd_status_string(status)} (status {status})")


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None):
    """Loads libfdattn.so and declares the C signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build the CUDA library first "
                               "(flash_decoding_attention_gb300.build.build())")
        lib = ctypes.CDLL(p)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        lib.fd_workspace_bytes.restype = sz
        lib.fd_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.fd_decode_attention.restype = i32
        lib.fd_decode_attention.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, i32, i32, i32, i32,
                                            i32, f32, f32, f32, i32, i32, vp, vp, vp, sz, vp]
        lib.fd_decode_attention_scaled.restype = i32
        lib.fd_decode_attention_scaled.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, i32, i32, i32,
                                                   i32, i32, f32, f32, f32, i32, vp, vp, i32, i32,
                                                   vp, vp, vp, sz, vp]
        lib.fd_decode_attention_multi.restype = i32
        lib.fd_decode_attention_multi.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, i32, i32, i32,
                                                  i32, i32, i32, f32, f32, f32, i32, vp, vp, i32,
                                                  i32, vp, vp, vp, sz, vp]
        lib.fd_append_kv.restype = i32
        lib.fd_append_kv.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i64, i32, i32, i32, i32, i32,
                                     f32, f32, i32, vp, vp, i32, i32, vp, sz, vp]
        lib.fd_decode_attention_append.restype = i32
        lib.fd_decode_attention_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i64,
                                                   i32, i32, i32, i32, i32, i32, f32, f32, f32,
                                                   i32, vp, vp, i32, i32, vp, vp, vp, sz, vp]
        lib.fd_decode_attention_noalloc.restype = i32
        lib.fd_decode_attention_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, i64, i32, i32,
                                                    i32, i32, i32, f32, f32, f32, i32, i32, vp,
                                                    vp, vp]
        lib.fd_check_device_error.restype = i32
        lib.fd_check_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int64)]
        lib.fd_status_string.restype = ctypes.c_char_p
        lib.fd_status_string.argtypes = [i32]
        lib.fd_set_kernel.restype = i32
        lib.fd_set_kernel.argtypes = [i32]
        lib.fd_selected_kernel.restype = i32
        lib.fd_selected_kernel.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.fd_selected_kernel_scaled.restype = i32
        lib.fd_selected_kernel_scaled.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
        lib.fd_set_split_events.restype = i32
        lib.fd_set_split_events.argtypes = [vp, vp]
        lib.fd_debug_read_plan.restype = i32
        lib.fd_debug_read_plan.argtypes = [vp, vp, vp, i32]
        lib.fd_debug_gather_kv.restype = i32
        lib.fd_debug_gather_kv.argtypes = [vp, vp, vp, i32, vp, i64, i32, i32, i32, i32, i32, vp,
                                           vp, vp]
        lib.fd_debug_set_wait_limit.restype = i32
        lib.fd_debug_set_wait_limit.argtypes = [i64, i32]
        lib.fd_debug_plan_segments.restype = i32
        lib.fd_debug_plan_segments.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                               vp, i64, i32, ctypes.POINTER(ctypes.c_int), vp, sz,
                                               vp]
        if path is None:
            _lib = lib
        return lib


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _q_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FD_F16
    if t.dtype == torch.bfloat16:
        return FD_BF16
    raise ValueError(f"q must be float16 or bfloat16, got {t.dtype}")


def _kv_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FD_F16
    if t.dtype == torch.bfloat16:
        return FD_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return FD_E4M3
    if t.dtype == torch.int8:
        return FD_I8
    raise ValueError(f"k/v cache must be float16, bfloat16, e4m3 bytes (uint8) or int8 codes, "
                     f"got {t.dtype}")


# ---------------------------------------------------------------------------
# one-to-one wrappers of the C ABI
# ---------------------------------------------------------------------------

def fd_status_string(status: int) -> str:
    return load_library().fd_status_string(int(status)).decode()


def fd_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load_library().fd_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim))


def fd_decode_attention(q, k_cache, v_cache, kv_start_idx, block_table, seq_len, kv_rows: int,
                        num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                        softmax_scale: float, k_scale: float, v_scale: float, out, lse, workspace,
                        stream=None, q_dtype: Optional[int] = None,
                        kv_dtype: Optional[int] = None, check: bool = True) -> int:
    """Enqueues one decode step; raises FdError on a non-OK status when
    ``check`` (else returns the status)."""
    lib = load_library()
    batch = int(seq_len.shape[0])
    stride = int(block_table.shape[1]) if block_table is not None else 0
    st = lib.fd_decode_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_start_idx), _ptr(block_table), stride,
        _ptr(seq_len), int(kv_rows), batch, int(num_q_heads), int(num_kv_heads), int(head_dim),
        int(page_size), float(softmax_scale), float(k_scale), float(v_scale),
        _q_dtype(q) if q_dtype is None else int(q_dtype),
        _kv_dtype(k_cache) if kv_dtype is None else int(kv_dtype),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream_handle(stream))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_attention")
    return st


def fd_decode_attention_scaled(q, k_cache, v_cache, kv_start_idx, block_table, seq_len,
                               kv_rows: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                               page_size: int, softmax_scale: float, k_scale: float,
                               v_scale: float, scale_kind: int, k_scales, v_scales, out, lse,
                               workspace, stream=None, q_dtype: Optional[int] = None,
                               kv_dtype: Optional[int] = None, check: bool = True) -> int:
    """fd_decode_attention with per-KV-head (FD_SCALE_HEAD, fp32 [KVH]) or
    per-token (FD_SCALE_TOKEN, fp32 [kv_rows, KVH]) K/V scales on top of
    k_scale / v_scale."""
    lib = load_library()
    batch = int(seq_len.shape[0])
    stride = int(block_table.shape[1]) if block_table is not None else 0
    st = lib.fd_decode_attention_scaled(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_start_idx), _ptr(block_table), stride,
        _ptr(seq_len), int(kv_rows), batch, int(num_q_heads), int(num_kv_heads), int(head_dim),
        int(page_size), float(softmax_scale), float(k_scale), float(v_scale), int(scale_kind),
        _ptr(k_scales), _ptr(v_scales),
        _q_dtype(q) if q_dtype is None else int(q_dtype),
        _kv_dtype(k_cache) if kv_dtype is None else int(kv_dtype),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream_handle(stream))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_attention_scaled")
    return st


def fd_decode_attention_multi(q, k_cache, v_cache, kv_start_idx, block_table, seq_len,
                              kv_rows: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                              page_size: int, softmax_scale: float, k_scale: float,
                              v_scale: float, scale_kind: int, k_scales, v_scales, out, lse,
                              workspace, stream=None, q_dtype: Optional[int] = None,
                              kv_dtype: Optional[int] = None, check: bool = True) -> int:
    """q_len query tokens per sequence (q, out: [B, QH, q_len, D]; lse
    [B, QH, q_len]), causal among the last q_len tokens of each sequence."""
    lib = load_library()
    batch = int(seq_len.shape[0])
    q_len = int(q.shape[2])
    stride = int(block_table.shape[1]) if block_table is not None else 0
    st = lib.fd_decode_attention_multi(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_start_idx), _ptr(block_table), stride,
        _ptr(seq_len), int(kv_rows), batch, q_len, int(num_q_heads), int(num_kv_heads),
        int(head_dim), int(page_size), float(softmax_scale), float(k_scale), float(v_scale),
        int(scale_kind), _ptr(k_scales), _ptr(v_scales),
        _q_dtype(q) if q_dtype is None else int(q_dtype),
        _kv_dtype(k_cache) if kv_dtype is None else int(kv_dtype),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream_handle(stream))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_attention_multi")
    return st


def fd_append_kv(k_new, v_new, k_cache, v_cache, kv_start_idx, block_table, positions,
                 kv_rows: int, num_kv_heads: int, head_dim: int, page_size: int, k_scale: float,
                 v_scale: float, scale_kind: int, k_scales, v_scales, workspace, stream=None,
                 new_dtype: Optional[int] = None, kv_dtype: Optional[int] = None,
                 check: bool = True) -> int:
    """Writes the new tokens of every sequence (k_new, v_new: [B, KVH, D] for
    one, [B, n_new, KVH, D] for n_new) into the caches from ``positions``
    (int32 [B], the first new token's index, < 0: none), quantising for 8-bit
    caches; per-token scales are written into ``k_scales`` / ``v_scales``."""
    lib = load_library()
    batch = int(positions.shape[0])
    n_new = int(k_new.shape[1]) if k_new.dim() == 4 else 1
    stride = int(block_table.shape[1]) if block_table is not None else 0
    st = lib.fd_append_kv(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(kv_start_idx),
        _ptr(block_table), stride, _ptr(positions), int(kv_rows), batch, n_new,
        int(num_kv_heads), int(head_dim), int(page_size), float(k_scale), float(v_scale), int(scale_kind),
        _ptr(k_scales), _ptr(v_scales),
        _q_dtype(k_new) if new_dtype is None else int(new_dtype),
        _kv_dtype(k_cache) if kv_dtype is None else int(kv_dtype),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if check and st != FD_OK:
        raise FdError(st, "fd_append_kv")
    return st


def fd_decode_attention_append(q, k_new, v_new, k_cache, v_cache, kv_start_idx, block_table,
                               positions, seq_len, kv_rows: int, num_q_heads: int,
                               num_kv_heads: int, head_dim: int, page_size: int,
                               softmax_scale: float, k_scale: float, v_scale: float,
                               scale_kind: int, k_scales, v_scales, out, lse, workspace,
                               stream=None, q_dtype: Optional[int] = None,
                               kv_dtype: Optional[int] = None, check: bool = True) -> int:
    """fd_append_kv of the step's new tokens, then the attention over the
    caches holding them (``seq_len`` counts them), in one call.  One new token
    per sequence with q [B, QH, D] and k_new [B, KVH, D]; q_len of them with
    q [B, QH, q_len, D] and k_new [B, q_len, KVH, D]."""
    lib = load_library()
    batch = int(seq_len.shape[0])
    q_len = int(q.shape[2]) if q.dim() == 4 else 1
    stride = int(block_table.shape[1]) if block_table is not None else 0
    st = lib.fd_decode_attention_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(kv_start_idx),
        _ptr(block_table), stride, _ptr(positions), _ptr(seq_len), int(kv_rows), batch, q_len,
        int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size), float(softmax_scale),
        float(k_scale), float(v_scale), int(scale_kind), _ptr(k_scales), _ptr(v_scales),
        _q_dtype(q) if q_dtype is None else int(q_dtype),
        _kv_dtype(k_cache) if kv_dtype is None else int(kv_dtype),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream_handle(stream))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_attention_append")
    return st


def fd_decode_attention_noalloc(q, k_cache, v_cache, kv_start_idx, block_table, seq_len,
                                kv_rows: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                page_size: int, softmax_scale: float, k_scale: float,
                                v_scale: float, out, lse, stream=None,
                                q_dtype: Optional[int] = None, kv_dtype: Optional[int] = None,
                                check: bool = True) -> int:
    """Like fd_decode_attention, but the library supplies the scratch memory
    from a fixed array of its own, for callers that cannot allocate device
    memory.  Calls that may overlap on the GPU must be serialised."""
    lib = load_library()
    batch = int(seq_len.shape[0])
    stride = int(block_table.shape[1]) if block_table is not None else 0
    st = lib.fd_decode_attention_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_start_idx), _ptr(block_table), stride,
        _ptr(seq_len), int(kv_rows), batch, int(num_q_heads), int(num_kv_heads), int(head_dim),
        int(page_size), float(softmax_scale), float(k_scale), float(v_scale),
        _q_dtype(q) if q_dtype is None else int(q_dtype),
        _kv_dtype(k_cache) if kv_dtype is None else int(kv_dtype),
        _ptr(out), _ptr(lse), _stream_handle(stream))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_attention_noalloc")
    return st


def fd_check_device_error(workspace, stream=None):
    """Returns (status, info) and clears the workspace's device-error word."""
    info = ctypes.c_int64(0)
    st = load_library().fd_check_device_error(_ptr(workspace), _stream_handle(stream),
                                              ctypes.byref(info))
    return st, info.value


def fd_set_kernel(kernel: int) -> None:
    st = load_library().fd_set_kernel(int(kernel))
    if st != FD_OK:
        raise FdError(st, "fd_set_kernel")


def fd_selected_kernel(num_q_heads, num_kv_heads, head_dim, q_dtype, kv_dtype, paged,
                       page_size) -> int:
    return int(load_library().fd_selected_kernel(num_q_heads, num_kv_heads, head_dim, q_dtype,
                                                 kv_dtype, int(bool(paged)), page_size))


def fd_selected_kernel_scaled(num_q_heads, num_kv_heads, head_dim, q_dtype, kv_dtype, paged,
                              page_size, scale_kind) -> int:
    return int(load_library().fd_selected_kernel_scaled(num_q_heads, num_kv_heads, head_dim,
                                                        q_dtype, kv_dtype, int(bool(paged)),
                                                        page_size, int(scale_kind)))


def fd_set_split_events(before: Optional[torch.cuda.Event], after: Optional[torch.cuda.Event]):
    h0 = before.cuda_event if before is not None else None
    h1 = after.cuda_event if after is not None else None
    st = load_library().fd_set_split_events(h0, h1)
    if st != FD_OK:
        raise FdError(st, "fd_set_split_events")


def fd_debug_read_plan(workspace, stream=None, capacity: int = 1 << 16):
    buf = (ctypes.c_int32 * capacity)()
    st = load_library().fd_debug_read_plan(_ptr(workspace), _stream_handle(stream), buf, capacity)
    if st != FD_OK:
        raise FdError(st, "fd_debug_read_plan")
    head = list(buf[:8])
    S = head[0]
    return head, list(buf[8:8 + S + 1])


def fd_debug_gather_kv(cache, kv_start_idx, block_table, seq_len, kv_rows, num_kv_heads, head_dim,
                       page_size, dst, workspace, stream=None, kv_dtype: Optional[int] = None):
    stride = int(block_table.shape[1]) if block_table is not None else 0
    st = load_library().fd_debug_gather_kv(
        _ptr(cache), _ptr(kv_start_idx), _ptr(block_table), stride, _ptr(seq_len), int(kv_rows),
        int(seq_len.shape[0]), int(num_kv_heads), int(head_dim), int(page_size),
        _kv_dtype(cache) if kv_dtype is None else int(kv_dtype), _ptr(dst), _ptr(workspace),
        _stream_handle(stream))
    if st != FD_OK:
        raise FdError(st, "fd_debug_gather_kv")


def fd_debug_set_wait_limit(wait_ns: int, starve_first_stage: bool = False) -> None:
    st = load_library().fd_debug_set_wait_limit(int(wait_ns), int(bool(starve_first_stage)))
    if st != FD_OK:
        raise FdError(st, "fd_debug_set_wait_limit")


def fd_debug_plan_segments(seq_len, q_len: int, num_q_heads: int, num_kv_heads: int,
                           head_dim: int, paged: bool, page_size: int, q_dtype: int,
                           kv_dtype: int, workspace, capacity_per_cta: int = 64, stream=None,
                           kv_start_idx=None):
    """Segments (stream, t_begin, t_end, complete, slot) of every CTA of the
    split kernel for these sizes, as the device plans them: a list with one
    list of tuples per CTA."""
    sms = torch.cuda.get_device_properties(seq_len.device).multi_processor_count
    rows = 1 + 5 * capacity_per_cta
    dst = torch.full((4 * sms * rows,), -1, dtype=torch.int32, device=seq_len.device)
    grid = ctypes.c_int(0)
    st = load_library().fd_debug_plan_segments(
        _ptr(seq_len), _ptr(kv_start_idx), int(seq_len.shape[0]), int(q_len), int(num_q_heads), int(num_kv_heads),
        int(head_dim), int(bool(paged)), int(page_size), int(q_dtype), int(kv_dtype), _ptr(dst),
        dst.numel(), int(capacity_per_cta), ctypes.byref(grid), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != FD_OK:
        raise FdError(st, "fd_debug_plan_segments")
    torch.cuda.synchronize(seq_len.device)
    d = dst[:grid.value * rows].view(grid.value, rows).cpu().tolist()
    out = []
    for r in d:
        n = r[0]
        if n > capacity_per_cta:
            raise RuntimeError(f"a CTA has {n} segments, more than capacity {capacity_per_cta}")
        out.append([tuple(r[1 + 5 * k: 6 + 5 * k]) for k in range(n)])
    return out


# ---------------------------------------------------------------------------
# convenience API
# ---------------------------------------------------------------------------

def alloc_workspace(batch, num_q_heads, num_kv_heads, head_dim, device=None) -> torch.Tensor:
    n = fd_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim)
    if n == 0:
        raise FdError(FD_ERR_INVALID_ARG, "fd_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     seq_len: torch.Tensor, *, kv_start_idx: Optional[torch.Tensor] = None,
                     block_table: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
                     k_scale: float = 1.0, v_scale: float = 1.0,
                     workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, stream=None,
                     k_scales: Optional[torch.Tensor] = None,
                     v_scales: Optional[torch.Tensor] = None,
                     k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                     positions: Optional[torch.Tensor] = None):
    """Decode attention over a contiguous ([rows, KVH, D]) or paged
    ([pages, page_size, KVH, D]) cache; returns (out, lse).  Optional 8-bit
    ``k_scales`` / ``v_scales``: fp32 [KVH] (per KV head) or [kv_rows, KVH]
    (per token, by cache row), multiplying ``k_scale`` / ``v_scale``.  With
    ``k_new`` / ``v_new`` ([B, KVH, D], q's dtype) and ``positions`` (int32
    [B]) the step's new token is first written into the caches (quantised for
    8-bit caches, per-token scales written), and ``seq_len`` counts it.  A 4-d
    ``q`` ([B, QH, q_len, D]) asks for q_len query tokens per sequence, the
    last q_len cached tokens, causal among themselves (out and lse carry the
    q_len axis too); with it, k_new / v_new are [B, q_len, KVH, D] and
    ``positions`` holds the first new token's index."""
    multi = q.dim() == 4              # [B, QH, q_len, D]: multi-token queries
    B, QH, D = q.shape[0], q.shape[1], q.shape[-1]
    q_len = q.shape[2] if multi else 1
    if block_table is not None:
        pages, P, KVH, D2 = k_cache.shape
        kv_rows = pages * P
    else:
        rows, KVH, D2 = k_cache.shape
        kv_rows, P = rows, 0
    assert D2 == D
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(B, QH * q_len, KVH, D, q.device)
    if multi and k_new is None:
        kind = FD_SCALE_TENSOR if k_scales is None else (
            FD_SCALE_HEAD if k_scales.dim() == 1 else FD_SCALE_TOKEN)
        fd_decode_attention_multi(q, k_cache, v_cache, kv_start_idx, block_table, seq_len,
                                  kv_rows, QH, KVH, D, P, softmax_scale, k_scale, v_scale, kind,
                                  k_scales, v_scales, out, lse, workspace, stream)
    elif k_new is not None:
        kind = FD_SCALE_TENSOR if k_scales is None else (
            FD_SCALE_HEAD if k_scales.dim() == 1 else FD_SCALE_TOKEN)
        fd_decode_attention_append(q, k_new, v_new, k_cache, v_cache, kv_start_idx, block_table,
                                   positions, seq_len, kv_rows, QH, KVH, D, P, softmax_scale,
                                   k_scale, v_scale, kind, k_scales, v_scales, out, lse,
                                   workspace, stream)
    elif k_scales is None:
        fd_decode_attention(q, k_cache, v_cache, kv_start_idx, block_table, seq_len, kv_rows, QH,
                            KVH, D, P, softmax_scale, k_scale, v_scale, out, lse, workspace,
                            stream)
    else:
        kind = FD_SCALE_HEAD if k_scales.dim() == 1 else FD_SCALE_TOKEN
        fd_decode_attention_scaled(q, k_cache, v_cache, kv_start_idx, block_table, seq_len,
                                   kv_rows, QH, KVH, D, P, softmax_scale, k_scale, v_scale, kind,
                                   k_scales, v_scales, out, lse, workspace, stream)
    return out, lse
