"""CPU fp64 oracle for decode-step attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg import this package.  The library in
``flash_decoding_attention_gb300`` never does, and this package never imports
that library: the two share only the seeded input arrays of ``fd_workloads``.

The arithmetic lives in ``fd_oracle.c`` (plain C, fp64, full two-pass softmax,
no blocking or online rescaling); this module compiles it with gcc and
marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fd_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libfd_oracle.so")

_DTYPES = {"f16": 0, "bf16": 1, "e4m3": 2, "i8": 3}
_ERRORS = {1: "bad argument", 2: "cache row out of range", 3: "NaN FP8 code", 4: "out of memory"}


class OracleError(RuntimeError):
    pass


def compile_source(src: str, out_path: str) -> str:
    """gcc -O2 with OpenMP and strict IEEE fp64 (no fast-math)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile fd_oracle.c into oracle/_build/libfd_oracle.so (if stale)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


class Oracle:
    """ctypes binding of one compiled copy of fd_oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.fdo_e4m3_value.restype = ctypes.c_double
        lib.fdo_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.fdo_i8_value.restype = ctypes.c_double
        lib.fdo_i8_value.argtypes = [ctypes.c_uint8]
        lib.fdo_f16_value.restype = ctypes.c_double
        lib.fdo_f16_value.argtypes = [ctypes.c_uint16]
        lib.fdo_bf16_value.restype = ctypes.c_double
        lib.fdo_bf16_value.argtypes = [ctypes.c_uint16]
        vp = ctypes.c_void_p
        lib.fdo_decode_attention_q.restype = ctypes.c_int
        lib.fdo_decode_attention_q.argtypes = [
            vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_double, ctypes.c_double,
            ctypes.c_int, vp, vp,
            vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.c_int, vp]
        lib.fdo_e4m3_encode.restype = ctypes.c_uint8
        lib.fdo_e4m3_encode.argtypes = [ctypes.c_float]
        lib.fdo_i8_encode.restype = ctypes.c_uint8
        lib.fdo_i8_encode.argtypes = [ctypes.c_float]
        lib.fdo_append_kv.restype = ctypes.c_int
        lib.fdo_append_kv.argtypes = [
            vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
            ctypes.c_float, ctypes.c_int, vp, vp]
        self.lib = lib
        self.path = lib_path

    def e4m3_value(self, code: int) -> float:
        return self.lib.fdo_e4m3_value(int(code))

    def i8_value(self, code: int) -> float:
        return self.lib.fdo_i8_value(int(code))

    def e4m3_encode(self, x: float) -> int:
        return int(self.lib.fdo_e4m3_encode(float(x)))

    def i8_encode(self, x: float) -> int:
        return int(self.lib.fdo_i8_encode(float(x)))

    def append_kv(self, w, k_new, v_new, positions):
        """The KV append on copies of the workload's caches (and per-token
        scale arrays).  k_new, v_new: [B, KVH, D] (one new token) or
        [B, n_new, KVH, D] 16-bit patterns of the workload's q dtype;
        positions: int32 [B], the first new token's index (< 0: no append).  Returns
        (k_cache, v_cache, k_scales, v_scales); the scale arrays are None for
        per-tensor scales."""
        k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
        v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
        n_new = int(k_new.shape[1]) if k_new.ndim == 4 else 1
        positions = np.ascontiguousarray(positions, dtype=np.int32)
        kc = np.ascontiguousarray(w.k_cache).copy()
        vc = np.ascontiguousarray(w.v_cache).copy()
        kind = getattr(w, "scale_kind", 0)
        ks = vs = None
        if kind:
            ks = np.ascontiguousarray(w.k_scales, dtype=np.float32).copy()
            vs = np.ascontiguousarray(w.v_scales, dtype=np.float32).copy()
        bt_stride = int(w.block_table.shape[1]) if w.block_table is not None else 0
        rc = self.lib.fdo_append_kv(
            _ptr(k_new), _ptr(v_new), _DTYPES[w.q_dtype], _ptr(kc), _ptr(vc), _DTYPES[w.kv_dtype],
            _ptr(w.kv_start_idx), _ptr(w.block_table), bt_stride, _ptr(positions),
            int(w.kv_rows), int(w.batch), n_new, int(w.num_kv_heads), int(w.head_dim),
            int(w.page_size), float(w.k_scale), float(w.v_scale), int(kind), _ptr(ks), _ptr(vs))
        if rc != 0:
            raise OracleError(_ERRORS.get(rc, f"status {rc}"))
        return kc, vc, ks, vs

    def f16_value(self, bits: int) -> float:
        return self.lib.fdo_f16_value(int(bits))

    def bf16_value(self, bits: int) -> float:
        return self.lib.fdo_bf16_value(int(bits))

    def decode_attention_raw(self, q, q_dtype, k_cache, v_cache, kv_dtype, seq_len,
                             num_q_heads, num_kv_heads, head_dim, softmax_scale, k_scale,
                             v_scale, kv_start_idx=None, block_table=None, page_size=0,
                             kv_rows=None, pairs: Optional[Sequence[Tuple[int, int]]] = None,
                             nthreads: int = 0, want_weights: bool = False, scale_kind: int = 0,
                             k_scales=None, v_scales=None, q_len: int = 1):
        """Oracle on raw arrays.  Returns (out [B,QH,D] f64, lse [B,QH] f64,
        weights [B,QH,maxT] or None, threads used).  With ``pairs`` only those
        (b, qh) rows are computed; the rest of ``out``/``lse`` stays NaN.
        ``scale_kind`` 1 (per KV head, arrays [KVH]) or 2 (per token, arrays
        [kv_rows, KVH]) multiplies K and V elements by ``k_scales`` and
        ``v_scales`` on top of ``k_scale`` and ``v_scale``.  With ``q_len`` > 1,
        q is [B, QH, q_len, D] (the last q_len tokens of each sequence, causal
        among themselves) and out / lse / weights carry a q_len axis after QH."""
        q = np.ascontiguousarray(q)
        k_cache = np.ascontiguousarray(k_cache)
        v_cache = np.ascontiguousarray(v_cache)
        seq_len = np.ascontiguousarray(seq_len, dtype=np.int32)
        B = int(seq_len.shape[0])
        if kv_start_idx is not None:
            kv_start_idx = np.ascontiguousarray(kv_start_idx, dtype=np.int32)
        bt_stride = 0
        if block_table is not None:
            block_table = np.ascontiguousarray(block_table, dtype=np.int32)
            bt_stride = int(block_table.shape[1])
        if kv_rows is None:
            kv_rows = (k_cache.shape[0] * k_cache.shape[1]) if block_table is not None \
                else k_cache.shape[0]
        qax = (q_len,) if q_len > 1 else ()
        out = np.full((B, num_q_heads) + qax + (head_dim,), np.nan, np.float64)
        lse = np.full((B, num_q_heads) + qax, np.nan, np.float64)
        weights = None
        wstride = 0
        if want_weights:
            wstride = max(1, int(seq_len.max()) if B else 1)
            weights = np.zeros((B, num_q_heads) + qax + (wstride,), np.float64)
        pairs_arr = None
        n_pairs = 0
        if pairs is not None:
            pairs_arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
            n_pairs = int(pairs_arr.shape[0])
        if scale_kind:
            k_scales = np.ascontiguousarray(k_scales, dtype=np.float32)
            v_scales = np.ascontiguousarray(v_scales, dtype=np.float32)
        else:
            k_scales = v_scales = None
        used = ctypes.c_int(0)
        rc = self.lib.fdo_decode_attention_q(
            _ptr(q), _DTYPES[q_dtype], _ptr(k_cache), _ptr(v_cache), _DTYPES[kv_dtype],
            _ptr(kv_start_idx), _ptr(block_table), bt_stride, _ptr(seq_len), int(kv_rows),
            B, int(q_len), int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size),
            float(softmax_scale), float(k_scale), float(v_scale),
            int(scale_kind), _ptr(k_scales), _ptr(v_scales),
            _ptr(pairs_arr), n_pairs, int(nthreads), _ptr(out), _ptr(lse), _ptr(weights),
            wstride, ctypes.addressof(used))
        if rc != 0:
            raise OracleError(_ERRORS.get(rc, f"status {rc}"))
        return out, lse, weights, used.value

    def decode_attention(self, w, pairs=None, nthreads: int = 0, want_weights: bool = False):
        """Oracle on an ``fd_workloads.Workload``; returns (out, lse) or
        (out, lse, weights)."""
        out, lse, weights, _ = self.decode_attention_raw(
            w.q, w.q_dtype, w.k_cache, w.v_cache, w.kv_dtype, w.seq_len, w.num_q_heads,
            w.num_kv_heads, w.head_dim, w.softmax_scale, w.k_scale, w.v_scale,
            kv_start_idx=w.kv_start_idx, block_table=w.block_table, page_size=w.page_size,
            kv_rows=w.kv_rows, pairs=pairs, nthreads=nthreads, want_weights=want_weights,
            scale_kind=getattr(w, "scale_kind", 0), k_scales=getattr(w, "k_scales", None),
            v_scales=getattr(w, "v_scales", None), q_len=getattr(w, "q_len", 1))
        if want_weights:
            return out, lse, weights
        return out, lse


_default: Optional[Oracle] = None
_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def e4m3_value(code: int) -> float:
    return default().e4m3_value(code)


def i8_value(code: int) -> float:
    return default().i8_value(code)


def f16_value(bits: int) -> float:
    return default().f16_value(bits)


def bf16_value(bits: int) -> float:
    return default().bf16_value(bits)


def decode_attention_raw(*args, **kwargs):
    return default().decode_attention_raw(*args, **kwargs)


def decode_attention(w, pairs=None, nthreads: int = 0, want_weights: bool = False):
    return default().decode_attention(w, pairs=pairs, nthreads=nthreads,
                                      want_weights=want_weights)


def append_kv(w, k_new, v_new, positions):
    return default().append_kv(w, k_new, v_new, positions)
