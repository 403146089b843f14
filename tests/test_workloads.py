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
