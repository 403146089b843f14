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
