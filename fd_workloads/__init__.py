"""Seeded synthetic decode-attention inputs.

This module only *generates* inputs (random draws, dtype casts, FP8 quantisation
and the placement of token rows into a contiguous or paged cache).  It holds no
attention arithmetic: both the CPU oracle and the CUDA library read the arrays
produced here, and neither is imported from here.

Every array is produced by ``numpy.random.Generator(PCG64(seed))`` with a fixed
draw order: sequence lengths, then Q, then K, then V, then the page permutation.

Shapes and recipes follow the five decode workloads of the flash-decoding
scope (tiny MQA; GQA bf16; FP8 ragged; FP8 paged; long-context MQA):

* Q is ``[B, QH, D]``; K/V caches are token-major ``[rows, KVH, D]`` for the
  contiguous layout (sequence ``b`` owns rows ``kv_start_idx[b] ...
  kv_start_idx[b] + seq_len[b] - 1``) and ``[num_pages, page_size, KVH, D]``
  for the paged layout, addressed through ``block_table[b, t // page_size]``.
* f16/bf16 tensors are stored as their raw 16-bit patterns (``uint16``),
  FP8-e4m3 tensors as raw bytes (``uint8``).
* FP8 K and V are quantised per tensor: ``scale = amax / 448`` in fp32, codes
  ``= e4m3fn(clamp(x / scale, -448, 448))`` rounded to nearest even.
* INT8 K and V (``kv_dtype='i8'``, stored as ``int8``) are quantised
  symmetrically per tensor: ``scale = amax / 127`` in fp32, codes
  ``= clamp(rint(x / scale), -127, 127)`` (round half to even, no zero point).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

E4M3_MAX = 448.0
I8_MAX = 127.0

# Values written where no sequence owns a row (gaps between contiguous
# sequences, unused pages, page tails).  A kernel that reads such a row
# produces a grossly wrong score or output, so parity fails loudly.
POISON_E4M3 = 0x7E          # +448
POISON_I8 = 127

SCALE_TENSOR, SCALE_HEAD, SCALE_TOKEN = 0, 1, 2
POISON_F16 = 30000.0


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    q_dtype: str              # 'f16' | 'bf16'  (out has the same dtype)
    kv_dtype: str             # 'f16' | 'bf16' | 'e4m3' | 'i8'
    softmax_scale: np.float32
    k_scale: np.float32
    v_scale: np.float32
    seq_len: np.ndarray       # int32 [B]
    q: np.ndarray             # uint16 [B, QH, D] raw bits
    k_cache: np.ndarray       # uint16/uint8 [rows, KVH, D] or [pages, P, KVH, D]
    v_cache: np.ndarray
    page_size: int = 0        # 0 = contiguous layout
    kv_start_idx: Optional[np.ndarray] = None   # int32 [B] (contiguous)
    block_table: Optional[np.ndarray] = None    # int32 [B, stride] (paged)
    # finer K/V scales on top of k_scale / v_scale: 0 none, 1 per KV head
    # (float32 [KVH]), 2 per token and KV head (float32 [kv_rows, KVH], by cache row)
    scale_kind: int = 0
    k_scales: Optional[np.ndarray] = None
    v_scales: Optional[np.ndarray] = None
    # query tokens per sequence: q is [B, QH, q_len, D] when q_len > 1 (the
    # last q_len tokens of each sequence, causal among themselves)
    q_len: int = 1

    @property
    def paged(self) -> bool:
        return self.page_size > 0

    @property
    def kv_rows(self) -> int:
        """Number of token rows the K/V buffers hold."""
        if self.paged:
            return int(self.k_cache.shape[0] * self.k_cache.shape[1])
        return int(self.k_cache.shape[0])

    @property
    def block_table_stride(self) -> int:
        return int(self.block_table.shape[1]) if self.paged else 0

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype in ("e4m3", "i8") else 2

    def algorithmic_bytes(self) -> int:
        """Bytes one decode step must move: K and V rows of every sequence,
        Q in, O out, and the index arrays it reads."""
        B, QH, KVH, D = self.batch, self.num_q_heads, self.num_kv_heads, self.head_dim
        total = int(self.seq_len.astype(np.int64).sum())
        kv = total * KVH * D * self.kv_elem_bytes * 2
        qo = 2 * B * QH * self.q_len * D * 2
        if self.paged:
            pages = int(sum((int(t) + self.page_size - 1) // self.page_size for t in self.seq_len))
            idx = 4 * B + 4 * pages
        else:
            idx = 8 * B
        if self.scale_kind == SCALE_HEAD:
            idx += 2 * 4 * KVH
        elif self.scale_kind == SCALE_TOKEN:
            idx += 2 * 4 * total * KVH
        return kv + qo + idx


# ----------------------------------------------------------------------------
# dtype helpers (casts of random draws into the stored formats)
# ----------------------------------------------------------------------------

def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x.astype(np.float16)).view(np.uint16)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def f32_to_e4m3_bytes(x: np.ndarray, scale: np.float32) -> np.ndarray:
    """Per-tensor quantisation to OCP e4m3fn codes (round to nearest even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = (t / torch.tensor(float(scale), dtype=torch.float32)).clamp_(-E4M3_MAX, E4M3_MAX)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def f32_to_i8(x: np.ndarray, scale: np.float32) -> np.ndarray:
    """Symmetric per-tensor INT8 quantisation (round half to even, clamp 127)."""
    t = np.ascontiguousarray(x, dtype=np.float32) / np.float32(scale)
    return np.clip(np.rint(t), -I8_MAX, I8_MAX).astype(np.int8)


def _cast16(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return f32_to_f16_bits(x)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def _poison_value(dtype: str):
    if dtype == "e4m3":
        return np.uint8(POISON_E4M3)
    if dtype == "i8":
        return np.int8(POISON_I8)
    return _cast16(np.array([POISON_F16], np.float32), dtype)[0]


def _quantise_pair(k: np.ndarray, v: np.ndarray, kv_dtype: str):
    """Cast the logical K/V draws to the stored format; return codes and scales."""
    if kv_dtype in ("e4m3", "i8"):
        top = np.float32(E4M3_MAX if kv_dtype == "e4m3" else I8_MAX)
        k_amax = np.float32(np.abs(k).max()) if k.size else np.float32(1.0)
        v_amax = np.float32(np.abs(v).max()) if v.size else np.float32(1.0)
        k_scale = np.float32(k_amax / top)
        v_scale = np.float32(v_amax / top)
        if k_scale == 0:
            k_scale = np.float32(1.0)
        if v_scale == 0:
            v_scale = np.float32(1.0)
        quant = f32_to_e4m3_bytes if kv_dtype == "e4m3" else f32_to_i8
        return quant(k, k_scale), quant(v, v_scale), k_scale, v_scale
    return _cast16(k, kv_dtype), _cast16(v, kv_dtype), np.float32(1.0), np.float32(1.0)


# ----------------------------------------------------------------------------
# generic builders
# ----------------------------------------------------------------------------

def make_contiguous(name: str, seed: int, seq_len, num_q_heads: int, num_kv_heads: int,
                    head_dim: int, q_dtype: str, kv_dtype: str, softmax_scale=None,
                    gap: int = 0, lead: int = 0, tail: int = 0,
                    rng: Optional[np.random.Generator] = None, q_len: int = 1) -> Workload:
    """Token-major contiguous cache.  ``gap`` poisoned rows separate consecutive
    sequences, ``lead``/``tail`` poisoned rows sit before the first and after the
    last one.  With all three zero, ``kv_start_idx`` is the exclusive prefix sum
    of ``seq_len``.  ``q_len`` > 1 draws q as [B, QH, q_len, D] (the same
    stream of draws as q_len = 1 extended)."""
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    seq_len = np.asarray(seq_len, dtype=np.int32)
    B = int(seq_len.shape[0])
    QH, KVH, D = num_q_heads, num_kv_heads, head_dim
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    total = int(seq_len.astype(np.int64).sum())

    q32 = rng.standard_normal((B, QH, q_len, D), dtype=np.float32)
    if q_len == 1:
        q32 = q32.reshape(B, QH, D)
    k32 = rng.standard_normal((total, KVH, D), dtype=np.float32)
    v32 = rng.standard_normal((total, KVH, D), dtype=np.float32)
    q = _cast16(q32, q_dtype)
    kq, vq, k_scale, v_scale = _quantise_pair(k32, v32, kv_dtype)
    del k32, v32

    starts = np.zeros(B, np.int32)
    rows = lead
    for b in range(B):
        starts[b] = rows
        rows += int(seq_len[b]) + (gap if b + 1 < B else 0)
    rows += tail
    rows = max(rows, 1)
    pv = _poison_value(kv_dtype)
    k_cache = np.full((rows, KVH, D), pv, dtype=kq.dtype)
    v_cache = np.full((rows, KVH, D), pv, dtype=vq.dtype)
    off = 0
    for b in range(B):
        n = int(seq_len[b])
        k_cache[starts[b]:starts[b] + n] = kq[off:off + n]
        v_cache[starts[b]:starts[b] + n] = vq[off:off + n]
        off += n
    return Workload(name=name, batch=B, num_q_heads=QH, num_kv_heads=KVH, head_dim=D,
                    q_dtype=q_dtype, kv_dtype=kv_dtype,
                    softmax_scale=np.float32(softmax_scale), k_scale=k_scale, v_scale=v_scale,
                    seq_len=seq_len, q=q, k_cache=k_cache, v_cache=v_cache,
                    page_size=0, kv_start_idx=starts, block_table=None, q_len=q_len)


def to_paged(w: Workload, page_size: int, seed: int, oversize: float = 1.2,
             rng: Optional[np.random.Generator] = None,
             extra_stride: int = 0) -> Workload:
    """Re-lay the logical rows of a contiguous workload into a paged pool.

    The pool holds ``ceil(oversize * sum_b ceil(T_b / page_size))`` pages; a
    seeded permutation of the pool's page ids is drawn and its first entries
    are handed to the sequences in order.  Unused pages and page tails are
    poisoned; block-table entries past a sequence's last page are -1."""
    assert not w.paged
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    P = int(page_size)
    B = w.batch
    npages = [(int(t) + P - 1) // P for t in w.seq_len]
    used = int(sum(npages))
    pool = max(1, int(math.ceil(oversize * used)))
    perm = rng.permutation(pool).astype(np.int32)
    stride = max(1, max(npages) if npages else 1) + extra_stride
    table = np.full((B, stride), -1, dtype=np.int32)
    pv = _poison_value(w.kv_dtype)
    shape = (pool, P, w.num_kv_heads, w.head_dim)
    k_pool = np.full(shape, pv, dtype=w.k_cache.dtype)
    v_pool = np.full(shape, pv, dtype=w.v_cache.dtype)
    nxt = 0
    for b in range(B):
        T = int(w.seq_len[b])
        s = int(w.kv_start_idx[b])
        for j in range(npages[b]):
            phys = int(perm[nxt])
            nxt += 1
            table[b, j] = phys
            lo, hi = j * P, min(T, (j + 1) * P)
            k_pool[phys, : hi - lo] = w.k_cache[s + lo:s + hi]
            v_pool[phys, : hi - lo] = w.v_cache[s + lo:s + hi]
    return dataclasses.replace(w, name=w.name + f"-paged{P}", k_cache=k_pool, v_cache=v_pool,
                               page_size=P, kv_start_idx=None, block_table=table)


def with_scales(w: Workload, kind: int, seed: int, powers_of_two: bool = False,
                span=(0.5, 2.0)) -> Workload:
    """Adds per-KV-head (kind 1) or per-token (kind 2) K/V scales to an e4m3
    or i8 workload.  They multiply k_scale / v_scale; seeded draws from ``span``,
    or from {1/4, 1/2, 1, 2, 4} with ``powers_of_two`` (products stay exact)."""
    assert w.kv_dtype in ("e4m3", "i8") and kind in (SCALE_HEAD, SCALE_TOKEN)
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (w.num_kv_heads,) if kind == SCALE_HEAD else (w.kv_rows, w.num_kv_heads)

    def draw():
        if powers_of_two:
            return np.exp2(rng.integers(-2, 3, size=shape)).astype(np.float32)
        return rng.uniform(span[0], span[1], size=shape).astype(np.float32)

    ks = draw()
    vs = draw()
    tag = "head" if kind == SCALE_HEAD else "token"
    return dataclasses.replace(w, name=w.name + f"-{tag}scales", scale_kind=kind, k_scales=ks,
                               v_scales=vs)


def share_prefix(w: Workload, shared_tokens: int) -> Workload:
    """Prefix-cache hit pattern on a paged workload: every sequence's first
    pages alias the physical pages of sequence 0 (the block tables point at
    the same pool pages; nothing is copied), as a serving system does when
    requests share a system prompt or a long context.  Only whole pages that
    both sequences fill are aliased, up to ``shared_tokens`` tokens; the
    pages a sequence gives up stay in the pool unused."""
    assert w.paged
    P = w.page_size
    table = w.block_table.copy()
    T0 = int(w.seq_len[0])
    for b in range(1, w.batch):
        k = min(int(shared_tokens) // P, T0 // P, int(w.seq_len[b]) // P)
        table[b, :k] = table[0, :k]
    return dataclasses.replace(w, name=w.name + f"-shared{int(shared_tokens)}", block_table=table)


def new_tokens(w: Workload, seed: int, std: float = 1.0, n_new: int = 1):
    """K and V of the new tokens of every sequence, [B, KVH, D] (one token) or
    [B, n_new, KVH, D] 16-bit patterns of the workload's q dtype (the
    projection's output dtype): N(0, std^2) draws, K then V."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = ((w.batch, w.num_kv_heads, w.head_dim) if n_new == 1
             else (w.batch, n_new, w.num_kv_heads, w.head_dim))
    k = rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
    v = rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
    return _cast16(k, w.q_dtype), _cast16(v, w.q_dtype)


def append_bytes(w: Workload, n_new: int = 1) -> int:
    """Bytes the KV append of n_new new tokens per sequence must move: the new
    K/V rows read (q dtype), the same rows written to the cache, the
    positions, and per-token scales written."""
    rows = w.batch * n_new * w.num_kv_heads * w.head_dim
    b = 2 * rows * 2 + 2 * rows * w.kv_elem_bytes + 4 * w.batch
    if w.scale_kind == SCALE_TOKEN:
        b += 2 * 4 * w.batch * n_new * w.num_kv_heads
    return b


def last_positions(w: Workload, n_new: int = 1) -> np.ndarray:
    """Index of the first of each sequence's last n_new tokens (the slots a
    decode or verify step appends into when seq_len already counts its new
    tokens); -1 for sequences shorter than n_new."""
    return np.where(w.seq_len >= n_new, w.seq_len - n_new, -1).astype(np.int32)


# ----------------------------------------------------------------------------
# the five decode workloads
# ----------------------------------------------------------------------------

def tiny_mqa() -> Workload:
    """B=2, seq_len {7, 33}, 4 query heads / 1 KV head, D=64, fp16 everywhere,
    contiguous (kv_start_idx {0, 7}), softmax_scale 1/8, seed 0."""
    return make_contiguous("tiny-mqa-f16", 0, [7, 33], 4, 1, 64, "f16", "f16",
                           softmax_scale=1.0 / 8.0)


def gqa_bf16(batch: int = 16, seq: int = 4096) -> Workload:
    """B=16, seq_len 4096, 32/8 heads, D=128, bf16, contiguous, seed 1."""
    return make_contiguous(f"gqa-bf16-B{batch}-T{seq}", 1, [seq] * batch, 32, 8, 128,
                           "bf16", "bf16")


def _kv_tag(kv_dtype: str) -> str:
    return "" if kv_dtype == "e4m3" else f"-{kv_dtype}"


def fp8_ragged(batch: int = 32, lo: int = 512, hi: int = 32768, kv_dtype: str = "e4m3") -> Workload:
    """B=32, seq_len ~ U{512..32768}, 32/8 heads, D=128, fp16 Q, e4m3 KV,
    contiguous, seed 2 (``kv_dtype='i8'``: the same draws quantised to INT8)."""
    rng = np.random.Generator(np.random.PCG64(2))
    seq = rng.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)
    return make_contiguous(f"fp8-ragged-B{batch}{_kv_tag(kv_dtype)}", 2, seq, 32, 8, 128, "f16",
                           kv_dtype, rng=rng)


def lognormal_lengths(rng: np.random.Generator, batch: int, median: float = 2048.0,
                      lo: int = 16, hi: int = 16384) -> np.ndarray:
    z = rng.standard_normal(batch)
    return np.clip(np.rint(median * np.exp(z)), lo, hi).astype(np.int32)


def fp8_paged(batch: int = 64, page_size: int = 64, kv_dtype: str = "e4m3") -> Workload:
    """B=64, seq_len lognormal (median 2048, sigma 1, clipped to [16, 16384]),
    64/8 heads, D=128, fp16 Q, e4m3 KV, page_size 64, 1.2x pool, seed 3
    (``kv_dtype='i8'``: the same draws quantised to INT8)."""
    rng = np.random.Generator(np.random.PCG64(3))
    seq = lognormal_lengths(rng, batch)
    w = make_contiguous(f"fp8-paged-B{batch}{_kv_tag(kv_dtype)}", 3, seq, 64, 8, 128, "f16",
                        kv_dtype, rng=rng)
    return to_paged(w, page_size, 3, rng=rng)


def long_mqa(batch: int = 4, seq: int = 131072, kv_dtype: str = "e4m3") -> Workload:
    """B=4, seq_len 131072, 16/1 heads, D=128, fp16 Q, e4m3 KV, contiguous, seed 4
    (``kv_dtype='i8'``: the same draws quantised to INT8)."""
    return make_contiguous(f"long-mqa-fp8-B{batch}-T{seq}{_kv_tag(kv_dtype)}", 4, [seq] * batch,
                           16, 1, 128, "f16", kv_dtype)


def with_q_len(w: Workload, q_len: int, seed: int) -> Workload:
    """The workload as a verify step of ``q_len`` query tokens per sequence
    (speculative decoding): the caches and lengths stay, and q is redrawn as
    [B, QH, q_len, D] from its own seed (the last q_len cached tokens of each
    sequence are the new ones)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q32 = rng.standard_normal((w.batch, w.num_q_heads, q_len, w.head_dim), dtype=np.float32)
    q = _cast16(q32, w.q_dtype)
    if q_len == 1:
        q = q.reshape(w.batch, w.num_q_heads, w.head_dim)
    return dataclasses.replace(w, name=w.name + f"-q{q_len}", q=q, q_len=q_len)


WORKLOADS = {
    1: tiny_mqa,
    2: gqa_bf16,
    3: fp8_ragged,
    4: fp8_paged,
    5: long_mqa,
}

WORKLOAD_NAMES = {
    1: "tiny MQA decode fp16: B=2, seq_len {7,33}, 4/1 heads, D=64, contiguous",
    2: "GQA decode bf16: B=16, seq_len 4096, 32/8 heads, D=128, contiguous",
    3: "FP8 ragged decode: B=32, seq_len U[512,32768], 32/8 heads, D=128, e4m3 KV, contiguous",
    4: "FP8 paged decode: B=64, seq_len lognormal(median 2048) in [16,16384], 64/8 heads, "
       "D=128, e4m3 KV, page 64, 1.2x permuted pool",
    5: "long-context MQA split-KV: B=4, seq_len 131072, 16/1 heads, D=128, e4m3 KV, contiguous",
}


# ----------------------------------------------------------------------------
# device copies (marshalling only)
# ----------------------------------------------------------------------------

def torch_dtypes(w: Workload):
    import torch
    qd = torch.float16 if w.q_dtype == "f16" else torch.bfloat16
    kd = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.uint8,
          "i8": torch.int8}[w.kv_dtype]
    return qd, kd


def to_torch(w: Workload, device="cuda", pin: bool = False) -> dict:
    """The workload's arrays as torch tensors on ``device`` (16-bit patterns
    reinterpreted as float16/bfloat16, e4m3 codes as uint8).  With
    ``device='cpu', pin=True`` the tensors are in pinned host memory."""
    import torch
    qd, kd = torch_dtypes(w)

    def mk(a, d=None):
        a = np.ascontiguousarray(a)
        if d is not None and a.dtype == np.uint16:
            t = torch.from_numpy(a.view(np.int16)).view(d)
        else:
            t = torch.from_numpy(a)
        if pin:
            return t.pin_memory()
        return t.to(device)

    out = {"q": mk(w.q, qd), "k": mk(w.k_cache, kd), "v": mk(w.v_cache, kd),
           "seq_len": mk(w.seq_len)}
    if w.paged:
        out["block_table"] = mk(w.block_table)
        out["kv_start_idx"] = None
    else:
        out["kv_start_idx"] = mk(w.kv_start_idx)
        out["block_table"] = None
    out["k_scales"] = mk(w.k_scales) if w.scale_kind else None
    out["v_scales"] = mk(w.v_scales) if w.scale_kind else None
    return out
