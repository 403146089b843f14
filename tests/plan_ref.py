"""Independent restatement of the library's split plan (stream-K over cost
units).

A work stream is (sequence b, one group of `hc` KV heads); there are
hg = num_kv_heads / hc streams per sequence, numbered s = b * hg + j.
Stream s has n_s = ceil(max(T_b, 0) / tile) tiles and costs
u_s = seg_units + n_s plan units when n_s > 0 (0 otherwise): `seg_units`
units for starting a segment, then one per tile.  The units of all streams,
concatenated in stream order, are dealt to `grid` CTAs in equal contiguous
runs of L = ceil(U / grid) units (U = sum u_s).  The tiles of a stream inside
one CTA's run form a segment (a run holding only some of a stream's leading
units holds none of it); a segment that is not the whole stream stores a
partial state in slot 2c (it continues a stream begun in an earlier CTA) or
2c + 1 (its stream continues in a later CTA).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List


@dataclass
class Seg:
    cta: int
    stream: int
    t_begin: int
    t_end: int
    complete: bool
    slot: int


def tiles_per_stream(seq_len, hg: int, tile: int) -> List[int]:
    out = []
    for T in seq_len:
        T = max(int(T), 0)
        n = -(-T // tile)
        out.extend([n] * hg)
    return out


def plan(seq_len, hg: int, tile: int, grid: int, seg_units: int = 0):
    """Returns (prefix [S+1] in units, total units, per_cta, segments)."""
    n = tiles_per_stream(seq_len, hg, tile)
    units = [x + seg_units if x > 0 else 0 for x in n]
    prefix = [0]
    for x in units:
        prefix.append(prefix[-1] + x)
    total = prefix[-1]
    per_cta = -(-total // grid) if total else 0
    segs = []
    for c in range(grid):
        g0, g1 = c * per_cta, min(total, (c + 1) * per_cta)
        for s in range(len(n)):
            a, e = max(g0, prefix[s]), min(g1, prefix[s + 1])
            if a >= e:
                continue
            first_tile_unit = prefix[s] + seg_units
            if e <= first_tile_unit:
                continue            # only leading units of the stream
            T = max(int(seq_len[s // hg]), 0)
            t0 = max(a, first_tile_unit) - first_tile_unit
            t1 = e - first_tile_unit
            starts_mid = a > first_tile_unit
            ends_mid = e < prefix[s + 1]
            segs.append(Seg(c, s, t0 * tile, min(t1 * tile, T),
                            not starts_mid and not ends_mid, 2 * c + (0 if starts_mid else 1)))
    return prefix, total, per_cta, segs


def merge_slots(prefix, total, grid, s, seg_units: int = 0):
    """Slots the combine step merges for stream s ([] if the stream is empty
    or held by one CTA): the CTAs holding its first and last tile units."""
    if prefix[s + 1] == prefix[s]:
        return []
    per_cta = -(-total // grid)
    c0, c1 = (prefix[s] + seg_units) // per_cta, (prefix[s + 1] - 1) // per_cta
    if c0 == c1:
        return []
    return [2 * c0 + 1] + [2 * c for c in range(c0 + 1, c1 + 1)]


def _next_pow2(x: int) -> int:
    p = 1
    while p < x:
        p <<= 1
    return p


def host_shape(kernel: int, num_q_heads: int, num_kv_heads: int, head_dim: int, kv_elem: int,
               sms: int, q_len: int = 1):
    """The host's choice of plan shape for a call, restated: returns
    (streams_per_sequence hg, tile tokens, grid, seg_units).

    kernel 2 (tensor cores): a 16-row head tile holds 16 query heads of one
    KV head; mt = next power of two of ceil(group / 16) tiles per KV head; a
    stream carries hc = 8 / mt KV heads (halved until it divides the KV
    heads), so that 8 consumer warps cover its mt * hc head tiles with
    wph = 8 / (mt * hc) warps each; a warp takes r sub-tiles of SUB tokens
    (32 for 8-bit caches, 16 for 16-bit ones) per stage, r = 65536 bytes of
    K+V over one r-step's bytes, clamped to [1, 4] and halved while a box
    would exceed 256 rows; tile = SUB * wph * r; a segment start costs
    ceil(128 KiB / stage bytes) tiles, twice that when wph > 1 (the warps of
    a head tile merge at every segment end); grid = one CTA per SM.
    kernel 1 (CUDA cores): streams of min(group, 16) query heads of one KV
    head, 32-token tiles, one CTA per SM, no start cost.
    kernel 4 (CUDA-core FMA form of kernel 2): kernel 2's shape.
    kernel 3 (tcgen05): a stream is one KV head with all its query rows;
    128-token tiles for groups of up to 64 rows, else 64-token tiles; one CTA
    per SM; a segment start costs ceil(128 KiB / stage bytes) tiles.
    """
    group = num_q_heads * q_len // num_kv_heads
    if kernel == 4:   # the CUDA-core form of kernel 2: the same plan shape
        kernel = 2
    if kernel == 3:
        tile = 128 if group <= 64 else 64
        return num_kv_heads, tile, sms, -(-131072 // (2 * tile * head_dim * kv_elem))
    if kernel == 1:
        hq = min(group, 16)
        return num_q_heads * q_len // hq, 32, sms, 0
    mt = _next_pow2(-(-group // 16))
    hc = 8 // mt
    while hc > 1 and num_kv_heads % hc:
        hc //= 2
    wph = 8 // (mt * hc)
    row = head_dim * kv_elem
    sub = 32 if kv_elem == 1 else 16
    r = max(1, min(4, 65536 // (sub * wph * hc * row * 2)))
    while r > 1 and sub * wph * r > 256:
        r //= 2
    tile = sub * wph * r
    stage = 2 * hc * tile * row
    return num_kv_heads // hc, tile, sms, (2 if wph > 1 else 1) * -(-131072 // stage)
