"""Host-side checks of the seeded input generators (no attention arithmetic)."""
import numpy as np

import fd_workloads as fw


def test_tiny_config_layout():
    w = fw.tiny_mqa()
    assert w.batch == 2 and list(w.seq_len) == [7, 33] and list(w.kv_start_idx) == [0, 7]
    assert w.q.shape == (2, 4, 64) and w.k_cache.shape == (40, 1, 64)
    assert w.q.dtype == np.uint16 and w.k_cache.dtype == np.uint16
    assert w.softmax_scale == np.float32(0.125)


def test_generation_is_deterministic():
    a = fw.make_contiguous("x", 5, [3, 9], 4, 2, 64, "f16", "e4m3", gap=2)
    b = fw.make_contiguous("x", 5, [3, 9], 4, 2, 64, "f16", "e4m3", gap=2)
    for f in ("q", "k_cache", "v_cache", "kv_start_idx"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert a.k_scale == b.k_scale and a.v_scale == b.v_scale


def test_ragged_lengths_match_seed():
    rng = np.random.Generator(np.random.PCG64(2))
    seq = rng.integers(512, 32768, size=32, endpoint=True)
    assert int(seq.sum()) == 519320
    assert seq.min() >= 512 and seq.max() <= 32768


def test_lognormal_lengths_are_clipped():
    rng = np.random.Generator(np.random.PCG64(3))
    seq = fw.lognormal_lengths(rng, 4096)
    assert seq.min() >= 16 and seq.max() <= 16384
    assert 1500 < np.median(seq) < 2700


def test_e4m3_quantisation_scale_and_saturation():
    w = fw.make_contiguous("q", 7, [50], 2, 1, 64, "f16", "e4m3")
    import torch
    k = torch.from_numpy(w.k_cache.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.abs(k).max() <= 448.0
    assert np.abs(k).max() >= 400.0          # the absmax element maps to ~448
    assert not np.any((w.k_cache & 0x7F) == 0x7F)   # no NaN codes


def test_paged_layout_covers_each_token_once():
    w = fw.make_contiguous("p", 8, [1, 63, 64, 65, 130], 4, 2, 64, "f16", "f16", gap=3)
    for P in (1, 16, 64):
        wp = fw.to_paged(w, P, 9)
        used = wp.block_table[wp.block_table >= 0]
        assert len(np.unique(used)) == len(used)            # no page shared
        assert used.max() < wp.k_cache.shape[0]
        for b in range(w.batch):
            T = int(w.seq_len[b])
            t = np.arange(T)
            phys = wp.block_table[b, t // P]
            got = wp.k_cache[phys, t % P]
            s = int(w.kv_start_idx[b])
            assert np.array_equal(got, w.k_cache[s:s + T])
            n = (T + P - 1) // P
            assert np.all(wp.block_table[b, n:] == -1)


def test_algorithmic_bytes_formula():
    w = fw.make_contiguous("b", 1, [10, 20], 8, 2, 128, "f16", "e4m3")
    assert w.algorithmic_bytes() == 30 * 2 * 128 * 1 * 2 + 2 * 2 * 8 * 128 * 2 + 8 * 2
    wp = fw.to_paged(w, 16, 2)
    assert wp.algorithmic_bytes() == 30 * 2 * 128 * 2 + 2 * 2 * 8 * 128 * 2 + 4 * 2 + 4 * (1 + 2)


def test_int8_quantisation_scale_and_range():
    """INT8 caches: symmetric per-tensor scale amax/127, codes in [-127, 127]
    with the largest magnitude on +-127, decoded values within half a step of
    the draws (checked against the e4m3 workload's same draws)."""
    a = fw.make_contiguous("q8", 7, [50, 20], 2, 1, 64, "f16", "i8", gap=1)
    e = fw.make_contiguous("q8", 7, [50, 20], 2, 1, 64, "f16", "e4m3", gap=1)
    assert a.k_cache.dtype == np.int8
    owned = np.ones(a.k_cache.shape[0], bool)
    owned[50] = False                                      # the gap row holds the poison code
    assert a.k_cache[~owned].min() == fw.POISON_I8
    k = a.k_cache[owned].astype(np.int32)
    assert k.min() >= -127 and k.max() <= 127 and np.abs(k).max() == 127
    # the same draws: e4m3 reconstructs them to 1/16 relative, int8 to half a step
    import torch
    ke = torch.from_numpy(e.k_cache[owned].copy()).view(torch.float8_e4m3fn).double().numpy()
    x = ke * float(e.k_scale)
    assert np.abs(k * float(a.k_scale) - x).max() <= 0.5 * float(a.k_scale) + 0.07 * np.abs(x).max()
    assert np.isclose(float(a.k_scale) * 127, float(e.k_scale) * 448, rtol=1e-6)


def test_multi_token_and_append_helpers():
    w = fw.make_contiguous("h", 8, [1, 4, 9], 4, 2, 64, "bf16", "e4m3", q_len=3)
    assert w.q.shape == (3, 4, 3, 64) and w.q_len == 3
    w1 = fw.make_contiguous("h", 8, [1, 4, 9], 4, 2, 64, "bf16", "e4m3")
    # q_len = 1 draws the same stream of numbers as the first token of a longer q
    assert w1.q.shape == (3, 4, 64)
    assert np.array_equal(fw.last_positions(w, 3), [-1, 1, 6])
    assert np.array_equal(fw.last_positions(w), [0, 3, 8])
    kn, vn = fw.new_tokens(w, 9, n_new=3)
    assert kn.shape == (3, 3, 2, 64) and kn.dtype == np.uint16 and not np.array_equal(kn, vn)
    k1, _ = fw.new_tokens(w, 9)
    assert k1.shape == (3, 2, 64)
    rows = 3 * 2 * 64
    assert fw.append_bytes(w) == 2 * rows * 2 + 2 * rows * 1 + 4 * 3
    assert fw.append_bytes(w, 3) == 3 * (2 * rows * 2 + 2 * rows) + 4 * 3
    v = fw.with_q_len(w1, 2, 10)
    assert v.q.shape == (3, 4, 2, 64) and v.q_len == 2
    assert v.algorithmic_bytes() - w1.algorithmic_bytes() == 2 * 3 * 4 * 64 * 2


def test_scales_and_shared_prefix_helpers():
    base = fw.make_contiguous("s", 11, [40, 70], 8, 2, 64, "f16", "e4m3")
    th = fw.with_scales(base, fw.SCALE_HEAD, 12)
    tt = fw.with_scales(base, fw.SCALE_TOKEN, 13, powers_of_two=True)
    assert th.k_scales.shape == (2,) and tt.k_scales.shape == (base.kv_rows, 2)
    assert set(np.unique(tt.k_scales)) <= {0.25, 0.5, 1.0, 2.0, 4.0}
    assert tt.algorithmic_bytes() - base.algorithmic_bytes() == 2 * 4 * 110 * 2
    paged = fw.to_paged(base, 16, 14)
    sh = fw.share_prefix(paged, 32)
    assert np.array_equal(sh.block_table[1, :2], sh.block_table[0, :2])
    assert not np.array_equal(paged.block_table[1, :2], paged.block_table[0, :2])
