"""CPU checks of the split-plan restatement: segments partition every
stream, a CTA's tiles plus the start costs it carries stay within L units,
and the combine's slot rule finds exactly the slots the segments wrote."""
import numpy as np
import pytest

import plan_ref


CASES = [
    ([7, 33], 1, 32, 152),
    ([4096] * 16, 8, 16, 152),
    ([131072] * 4, 1, 128, 152),
    ([0, 5, 0, 1000, 1], 2, 16, 7),
    ([1], 1, 16, 1),
    ([0, 0], 4, 16, 3),
]


@pytest.mark.parametrize("seg_units", [0, 2, 5])
@pytest.mark.parametrize("seq,hg,tile,grid", CASES + [
    (list(np.random.default_rng(i).integers(0, 3000, size=37)), hg, tile, grid)
    for i, (hg, tile, grid) in enumerate([(1, 32, 152), (8, 16, 148), (2, 128, 13), (4, 64, 300)])
])
def test_plan_partitions_streams(seq, hg, tile, grid, seg_units):
    prefix, total, per_cta, segs = plan_ref.plan(seq, hg, tile, grid, seg_units)
    S = len(seq) * hg
    assert len(prefix) == S + 1 and prefix[-1] == total
    per_stream = {s: [] for s in range(S)}
    per_cta_tiles = {}
    for g in segs:
        per_stream[g.stream].append(g)
        ntile = -(-(g.t_end - g.t_begin) // tile) if g.t_end > g.t_begin else 0
        per_cta_tiles[g.cta] = per_cta_tiles.get(g.cta, 0) + ntile
    for c, n in per_cta_tiles.items():
        assert n <= per_cta
    for s in range(S):
        T = max(int(seq[s // hg]), 0)
        ss = sorted(per_stream[s], key=lambda g: g.t_begin)
        if T == 0:
            assert ss == []
            assert plan_ref.merge_slots(prefix, total, grid, s, seg_units) == []
            continue
        assert ss[0].t_begin == 0 and ss[-1].t_end == T
        for a, b in zip(ss, ss[1:]):
            assert a.t_end == b.t_begin and a.cta < b.cta
        if len(ss) == 1:
            assert ss[0].complete and plan_ref.merge_slots(prefix, total, grid, s, seg_units) == []
        else:
            assert not any(g.complete for g in ss)
            assert plan_ref.merge_slots(prefix, total, grid, s, seg_units) == [g.slot for g in ss]
    # no slot is written twice
    slots = [g.slot for g in segs if not g.complete]
    assert len(slots) == len(set(slots))

    # start costs: a CTA whose run holds all leading units of a stream it
    # starts carries them on top of its tiles
    if per_cta:
        for c, n in per_cta_tiles.items():
            starts = [g for g in segs if g.cta == c and g.t_begin == 0
                      and prefix[g.stream] >= c * per_cta]
            assert n + seg_units * len(starts) <= per_cta


def test_start_cost_moves_tiles_off_busy_ctas():
    """With a start cost, CTAs that begin more segments receive fewer tiles:
    the most loaded CTA's tiles + starts * cost shrinks or stays."""
    rng = np.random.default_rng(11)
    seq = list(np.clip(np.round(2048 * np.exp(rng.normal(0, 1, 64))), 16, 16384).astype(int))
    def worst(seg_units, cost=2):
        _, _, _, segs = plan_ref.plan(seq, 1, 32, 152, seg_units)
        load = {}
        for g in segs:
            load[g.cta] = load.get(g.cta, 0) + -(-(g.t_end - g.t_begin) // 32) + cost
        return max(load.values())
    assert worst(2) <= worst(0)
