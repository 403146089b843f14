"""Pins for the CPU oracle: checks that tie it to things other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` instance and raises AssertionError
(or the oracle's own error) when the oracle disagrees with

* the number formats' definitions, decoded by independent library routines
  (numpy float16 and int8, torch bfloat16 and float8_e4m3fn);
* closed forms of softmax attention (identical rows, one key, two keys,
  uniform weights, a dominant key, the empty sequence);
* invariants (weights sum to one, key permutation, GQA == MHA with
  replicated KV heads, paged == contiguous, scaling and shifting);
* an independent fp64 recomputation by the chunked online-softmax recurrence
  (running max, running sum, rescaled accumulator) over random chunk
  boundaries, with the two halves of each sequence merged by their
  log-sum-exp -- the recurrence of the online softmax loop in "SGLang Prefill
  optimisation: dissecting FlashAttention kernel bottlenecks with GPU Trace",
  section 2.2, and the split merge it implies.

The pins are collected in ``ALL_PINS`` so that a mutation test can run them
against deliberately broken copies of the oracle.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

import fd_workloads as fw


# ----------------------------------------------------------------------------
# independent decoders (library routines, not the oracle's)
# ----------------------------------------------------------------------------

def lib_decode(arr: np.ndarray, dtype: str) -> np.ndarray:
    arr = np.ascontiguousarray(arr)
    if dtype == "f16":
        return arr.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        t = torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16)
        return t.to(torch.float64).numpy()
    if dtype == "e4m3":
        t = torch.from_numpy(arr.view(np.uint8).copy()).view(torch.float8_e4m3fn)
        return t.to(torch.float64).numpy()
    if dtype == "i8":
        return arr.view(np.int8).astype(np.float64)
    raise ValueError(dtype)


def custom(q32, k32, v32, seq_len, q_dtype="f16", kv_dtype="f16", softmax_scale=0.125,
           k_scale=1.0, v_scale=1.0, kv_start_idx=None, name="custom") -> fw.Workload:
    """A contiguous workload from explicit float arrays (cast to the stored
    formats; e4m3 and i8 codes are taken from the values with scale 1)."""
    q32 = np.asarray(q32, np.float32)
    k32 = np.asarray(k32, np.float32)
    v32 = np.asarray(v32, np.float32)
    seq_len = np.asarray(seq_len, np.int32)
    B, QH, D = q32.shape
    KVH = k32.shape[1]
    if kv_start_idx is None:
        kv_start_idx = np.concatenate([[0], np.cumsum(seq_len)[:-1]]).astype(np.int32)
    q = fw._cast16(q32, q_dtype)
    if kv_dtype == "e4m3":
        k = fw.f32_to_e4m3_bytes(k32, np.float32(1.0))
        v = fw.f32_to_e4m3_bytes(v32, np.float32(1.0))
    elif kv_dtype == "i8":
        k = np.clip(np.rint(k32), -128, 127).astype(np.int8)
        v = np.clip(np.rint(v32), -128, 127).astype(np.int8)
    else:
        k = fw._cast16(k32, kv_dtype)
        v = fw._cast16(v32, kv_dtype)
    return fw.Workload(name=name, batch=B, num_q_heads=QH, num_kv_heads=KVH, head_dim=D,
                       q_dtype=q_dtype, kv_dtype=kv_dtype,
                       softmax_scale=np.float32(softmax_scale), k_scale=np.float32(k_scale),
                       v_scale=np.float32(v_scale), seq_len=seq_len, q=q, k_cache=k, v_cache=v,
                       page_size=0, kv_start_idx=np.asarray(kv_start_idx, np.int32))


# ----------------------------------------------------------------------------
# independent recomputation: chunked online softmax + LSE merge
# ----------------------------------------------------------------------------

def _online_state(scores: np.ndarray, vals: np.ndarray, rng, chunk_max: int):
    """Running max m, running sum l and rescaled accumulator acc over random
    chunks of the score sequence."""
    D = vals.shape[1]
    m, l, acc = -math.inf, 0.0, np.zeros(D)
    i = 0
    n = scores.shape[0]
    while i < n:
        j = min(n, i + int(rng.integers(1, chunk_max + 1)))
        s = scores[i:j]
        m_new = max(m, float(s.max()))
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        p = np.exp(s - m_new)
        l = l * alpha + float(p.sum())
        acc = acc * alpha + p @ vals[i:j]
        m = m_new
        i = j
    return m, l, acc


def _merge(states, D):
    ms = [s[0] for s in states if s[1] > 0]
    if not ms:
        return -math.inf, 0.0, np.zeros(D)
    M = max(ms)
    l = 0.0
    acc = np.zeros(D)
    for m, li, ai in states:
        if li > 0:
            f = math.exp(m - M)
            l += li * f
            acc = acc + ai * f
    return M, l, acc


def online_reference(w: fw.Workload, rng, chunk_max: int = 7):
    """fp64 out/lse by the online-softmax recurrence, each sequence cut at a
    random point into two partial states that are merged afterwards."""
    B, QH, KVH, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    g = QH // KVH
    qf = lib_decode(w.q, w.q_dtype).reshape(B, QH, D)
    kf = lib_decode(w.k_cache, w.kv_dtype).reshape(-1, KVH, D) * float(w.k_scale)
    vf = lib_decode(w.v_cache, w.kv_dtype).reshape(-1, KVH, D) * float(w.v_scale)
    out = np.zeros((B, QH, D))
    lse = np.zeros((B, QH))
    for b in range(B):
        T = int(w.seq_len[b])
        t = np.arange(T)
        if w.paged:
            P = w.page_size
            rows = w.block_table[b, t // P].astype(np.int64) * P + t % P
        else:
            rows = int(w.kv_start_idx[b]) + t
        for qh in range(QH):
            kvh = qh // g
            if T == 0:
                out[b, qh] = 0.0
                lse[b, qh] = -math.inf
                continue
            scores = float(w.softmax_scale) * (kf[rows, kvh, :] @ qf[b, qh])
            vals = vf[rows, kvh, :]
            cut = int(rng.integers(0, T + 1))
            st = [_online_state(scores[:cut], vals[:cut], rng, chunk_max),
                  _online_state(scores[cut:], vals[cut:], rng, chunk_max)]
            m, l, acc = _merge(st, D)
            out[b, qh] = acc / l
            lse[b, qh] = m + math.log(l)
    return out, lse


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    assert np.all(err <= lim), f"{what}: max err {err.max():.3e}"


def pin_e4m3_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = lib_decode(codes, "e4m3")
    got = np.array([orc.e4m3_value(c) for c in range(256)])
    nan = (codes & 0x7F) == 0x7F
    assert np.all(np.isnan(got[nan])), "S.1111.111 must decode to NaN"
    assert np.array_equal(got[~nan], ref[~nan]), "e4m3 decode differs from float8_e4m3fn"
    # values fixed by the format: largest normal, smallest subnormal,
    # smallest normal, one, negative zero
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9
    assert orc.e4m3_value(0x08) == 2.0 ** -6
    assert orc.e4m3_value(0x38) == 1.0
    assert orc.e4m3_value(0xB8) == -1.0
    assert math.copysign(1.0, orc.e4m3_value(0x80)) == -1.0 and orc.e4m3_value(0x80) == 0.0


def pin_i8_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = lib_decode(codes, "i8")
    got = np.array([orc.i8_value(int(c)) for c in codes])
    assert np.array_equal(got, ref), "i8 decode differs from numpy int8"
    # two's complement ends and the sign boundary
    assert orc.i8_value(0x7F) == 127.0 and orc.i8_value(0x80) == -128.0
    assert orc.i8_value(0xFF) == -1.0 and orc.i8_value(0x00) == 0.0


def pin_f16_codes(orc):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = lib_decode(codes, "f16")
    got = np.array([orc.f16_value(int(c)) for c in codes])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def pin_bf16_codes(orc):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = lib_decode(codes, "bf16")
    got = np.array([orc.bf16_value(int(c)) for c in codes])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def pin_identical_v_rows(orc):
    rng = np.random.default_rng(11)
    T, D = 37, 64
    q = rng.standard_normal((1, 4, D))
    k = rng.standard_normal((T, 2, D))
    row = rng.standard_normal((1, 2, D))
    v = np.repeat(row, T, axis=0)
    w = custom(q, k, v, [T], v_scale=0.75)
    out, lse = orc.decode_attention(w)
    expect = lib_decode(w.v_cache[0], "f16") * 0.75      # [KVH, D]
    for qh in range(4):
        _close(out[0, qh], expect[qh // 2], 1e-14, 1e-300, "identical V rows")


def pin_single_key(orc):
    """seq_len = 1: the only weight is 1, so out = v_0 and lse = s_0.  With a
    one-hot q and k the score is known exactly."""
    D = 64
    q = np.zeros((1, 1, D)); q[0, 0, 5] = 1.5
    k = np.zeros((3, 1, D)); k[1, 0, 5] = -2.0; k[1, 0, 6] = 7.0
    v = np.zeros((3, 1, D)); v[1, 0, :] = np.arange(D) / 8.0
    w = custom(q, k, v, [1], kv_start_idx=[1], softmax_scale=0.25, k_scale=0.5, v_scale=2.0)
    out, lse = orc.decode_attention(w)
    assert lse[0, 0] == 0.25 * 1.5 * (-2.0 * 0.5)
    assert np.array_equal(out[0, 0], 2.0 * np.arange(D) / 8.0)


def pin_zero_query(orc):
    """q = 0: all scores are 0, weights are 1/T, out = mean of V, lse = ln T."""
    rng = np.random.default_rng(12)
    T, D = 50, 128
    q = np.zeros((1, 2, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, D))
    w = custom(q, k, v, [T])
    out, lse = orc.decode_attention(w)
    vf = lib_decode(w.v_cache, "f16")[:, 0, :]
    for qh in range(2):
        _close(out[0, qh], vf.mean(axis=0), 1e-13, 1e-15, "zero query mean")
        _close(lse[0, qh], math.log(T), 1e-15, 0, "zero query lse")


def pin_identical_k_rows(orc):
    """All K rows equal: uniform weights, out = mean V, lse = s + ln T, where
    s is exact for a one-hot key."""
    rng = np.random.default_rng(13)
    T, D = 21, 64
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    q[0, 0, 3] = 0.625
    k = np.zeros((T, 1, D)); k[:, 0, 3] = 4.0
    v = rng.standard_normal((T, 1, D))
    w = custom(q, k, v, [T], softmax_scale=0.5)
    out, lse = orc.decode_attention(w)
    vf = lib_decode(w.v_cache, "f16")[:, 0, :]
    _close(out[0, 0], vf.mean(axis=0), 1e-13, 1e-15, "identical K mean")
    _close(lse[0, 0], 0.5 * 0.625 * 4.0 + math.log(T), 1e-15, 0, "identical K lse")


def pin_two_keys(orc):
    """T = 2: out = sigma(s0 - s1) v0 + sigma(s1 - s0) v1 and
    lse = logaddexp(s0, s1), with exact one-hot scores."""
    D = 64
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0; q[0, 0, 1] = 1.0
    k = np.zeros((2, 1, D)); k[0, 0, 0] = 3.0; k[1, 0, 1] = -1.25
    v = np.zeros((2, 1, D)); v[0, 0, :] = 1.0; v[1, 0, :] = -2.0; v[1, 0, 7] = 5.0
    w = custom(q, k, v, [2], softmax_scale=1.0)
    out, lse = orc.decode_attention(w)
    s0, s1 = 3.0, -1.25
    a0 = 1.0 / (1.0 + math.exp(s1 - s0))
    a1 = 1.0 / (1.0 + math.exp(s0 - s1))
    expect = a0 * lib_decode(w.v_cache, "f16")[0, 0] + a1 * lib_decode(w.v_cache, "f16")[1, 0]
    _close(out[0, 0], expect, 1e-14, 1e-15, "two keys out")
    _close(lse[0, 0], np.logaddexp(s0, s1), 1e-15, 0, "two keys lse")


def pin_dominant_key(orc):
    """One score exceeds all others by at least 40: out equals that key's V
    row to within e^-40 times the spread of V."""
    rng = np.random.default_rng(14)
    T, D = 64, 64
    q = np.zeros((1, 1, D)); q[0, 0, 9] = 8.0
    k = rng.uniform(-0.5, 0.5, (T, 1, D)); k[17, 0, 9] = 6.0
    v = rng.standard_normal((T, 1, D))
    w = custom(q, k, v, [T], softmax_scale=1.0)
    out, lse = orc.decode_attention(w)
    v17 = lib_decode(w.v_cache, "f16")[17, 0]
    assert np.max(np.abs(out[0, 0] - v17)) < 64 * math.exp(-40) * 10
    _close(lse[0, 0], 8.0 * float(lib_decode(w.k_cache, "f16")[17, 0, 9]), 1e-12, 0, "dominant lse")


def pin_empty_sequence(orc):
    rng = np.random.default_rng(15)
    D = 64
    q = rng.standard_normal((2, 2, D))
    k = rng.standard_normal((5, 1, D))
    v = rng.standard_normal((5, 1, D))
    w = custom(q, k, v, [0, 5], kv_start_idx=[0, 0])
    out, lse = orc.decode_attention(w)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1])) and np.all(np.isfinite(lse[1]))


def pin_weights_sum_to_one(orc):
    w = fw.make_contiguous("ws", 16, [1, 9, 130], 8, 2, 64, "f16", "e4m3", gap=3)
    out, lse, weights = orc.decode_attention(w, want_weights=True)
    for b, T in enumerate(w.seq_len):
        s = weights[b, :, :T].sum(axis=-1)
        assert np.all(np.abs(s - 1.0) < 1e-14), s
        assert np.all(weights[b, :, :T] >= 0)


def pin_key_permutation(orc):
    rng = np.random.default_rng(17)
    w = fw.make_contiguous("perm", 17, [45, 12], 4, 2, 128, "bf16", "bf16")
    out, lse = orc.decode_attention(w)
    k = w.k_cache.copy(); v = w.v_cache.copy()
    for b in range(w.batch):
        s, T = int(w.kv_start_idx[b]), int(w.seq_len[b])
        p = rng.permutation(T)
        k[s:s + T] = w.k_cache[s:s + T][p]
        v[s:s + T] = w.v_cache[s:s + T][p]
    out2, lse2 = orc.decode_attention(dataclasses.replace(w, k_cache=k, v_cache=v))
    _close(out2, out, 1e-12, 1e-14, "permutation out")
    _close(lse2, lse, 1e-13, 0, "permutation lse")


def pin_gqa_equals_replicated_mha(orc):
    w = fw.make_contiguous("gqa", 18, [33, 7], 8, 2, 64, "f16", "f16", gap=2)
    out, lse = orc.decode_attention(w)
    g = 4
    k = np.repeat(w.k_cache, g, axis=1)
    v = np.repeat(w.v_cache, g, axis=1)
    mha = dataclasses.replace(w, num_kv_heads=8, k_cache=k, v_cache=v)
    out2, lse2 = orc.decode_attention(mha)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_paged_equals_contiguous(orc):
    w = fw.make_contiguous("pg", 19, [1, 16, 17, 70], 4, 2, 64, "f16", "e4m3", gap=5)
    out, lse = orc.decode_attention(w)
    for P in (1, 4, 16):
        wp = fw.to_paged(w, P, 19 + P)
        out2, lse2 = orc.decode_attention(wp)
        assert np.array_equal(out, out2) and np.array_equal(lse, lse2), P


def pin_scale_factors(orc):
    """v_scale scales out and leaves lse; doubling k_scale equals doubling
    softmax_scale (both exact in fp64)."""
    w = fw.make_contiguous("sc", 20, [25, 3], 4, 1, 64, "f16", "e4m3")
    out, lse = orc.decode_attention(w)
    out2, lse2 = orc.decode_attention(dataclasses.replace(w, v_scale=np.float32(w.v_scale * 4)))
    assert np.array_equal(out2, 4 * out) and np.array_equal(lse2, lse)
    a = orc.decode_attention(dataclasses.replace(w, k_scale=np.float32(w.k_scale * 2)))
    b = orc.decode_attention(dataclasses.replace(w, softmax_scale=np.float32(w.softmax_scale * 2)))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert not np.allclose(a[1], lse)


def pin_score_shift(orc):
    """A component shared by every key shifts all scores of a head by the
    same amount: out is unchanged and lse moves by exactly that amount."""
    rng = np.random.default_rng(21)
    T, D = 40, 64
    q = rng.standard_normal((1, 1, D)); q[0, 0, 0] = 0.0
    k = rng.standard_normal((T, 1, D)); k[:, 0, 0] = 2.0
    v = rng.standard_normal((T, 1, D))
    w = custom(q, k, v, [T], softmax_scale=0.25)
    out, lse = orc.decode_attention(w)
    q2 = q.copy(); q2[0, 0, 0] = 1.5
    w2 = custom(q2, k, v, [T], softmax_scale=0.25)
    out2, lse2 = orc.decode_attention(w2)
    _close(out2, out, 1e-12, 1e-14, "shift out")
    _close(lse2, lse + 0.25 * 1.5 * 2.0, 1e-13, 0, "shift lse")


def pin_online_recurrence(orc):
    """Brute force on small inputs: the oracle equals the chunked online
    softmax with a split merge to 1e-12 (relative, fp64)."""
    rng = np.random.default_rng(22)
    cases = [
        fw.tiny_mqa(),
        fw.make_contiguous("a", 23, [1, 2, 63, 64, 65, 200], 8, 2, 128, "f16", "e4m3", gap=4, lead=3),
        fw.make_contiguous("b", 24, [129, 5], 32, 8, 64, "bf16", "bf16", gap=1),
        fw.to_paged(fw.make_contiguous("c", 25, [3, 64, 100], 16, 1, 128, "f16", "e4m3"), 16, 26),
        fw.make_contiguous("d", 27, [0, 31, 0], 4, 4, 64, "f16", "f16"),
    ]
    for w in cases:
        out, lse = orc.decode_attention(w)
        ref_out, ref_lse = online_reference(w, rng)
        _close(out, ref_out, 1e-12, 1e-13, f"online out {w.name}")
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse))
        _close(lse[fin], ref_lse[fin], 1e-12, 1e-13, f"online lse {w.name}")


def materialize_scales(w: fw.Workload) -> fw.Workload:
    """The same attention with the finer scales multiplied into an f16 cache
    (per-tensor scales only).  Exact when the scales are powers of two: an
    e4m3 value or an i8 code times 2^-2 .. 2^2 is an f16 value.  With
    per-tensor scales only, the codes are decoded into the f16 cache as they
    are."""
    KVH, D = w.num_kv_heads, w.head_dim
    kd = lib_decode(w.k_cache, w.kv_dtype).reshape(-1, KVH, D)
    vd = lib_decode(w.v_cache, w.kv_dtype).reshape(-1, KVH, D)
    if w.scale_kind == fw.SCALE_TENSOR:
        ks = vs = np.float64(1.0)
    elif w.scale_kind == fw.SCALE_HEAD:
        ks = w.k_scales.astype(np.float64)[None, :, None]
        vs = w.v_scales.astype(np.float64)[None, :, None]
    else:
        ks = w.k_scales.astype(np.float64).reshape(-1, KVH)[:, :, None]
        vs = w.v_scales.astype(np.float64).reshape(-1, KVH)[:, :, None]
    kf, vf = kd * ks, vd * vs
    k16 = fw.f32_to_f16_bits(kf.astype(np.float32)).reshape(w.k_cache.shape)
    v16 = fw.f32_to_f16_bits(vf.astype(np.float32)).reshape(w.v_cache.shape)
    assert np.array_equal(lib_decode(k16, "f16").reshape(kf.shape), kf)
    assert np.array_equal(lib_decode(v16, "f16").reshape(vf.shape), vf)
    return dataclasses.replace(w, kv_dtype="f16", k_cache=k16, v_cache=v16, scale_kind=0,
                               k_scales=None, v_scales=None)


def pin_head_scales_materialized(orc):
    """Per-KV-head scales equal an f16 cache holding scale * decoded code
    (GQA, two dtypes of q, different K and V scales per head)."""
    for seed, qdt in ((31, "f16"), (32, "bf16")):
        base = fw.make_contiguous("hs", seed, [1, 40, 129], 16, 4, 64, qdt, "e4m3", gap=3)
        w = fw.with_scales(base, fw.SCALE_HEAD, seed + 100, powers_of_two=True)
        assert len(set(w.k_scales.tolist())) > 1 and not np.array_equal(w.k_scales, w.v_scales)
        a = orc.decode_attention(w)
        b = orc.decode_attention(materialize_scales(w))
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def pin_token_scales_materialized(orc):
    """Per-token scales, indexed by cache row and KV head, equal an f16
    cache holding scale * decoded code: with gaps between sequences (row !=
    position) and through a shuffled page pool."""
    base = fw.make_contiguous("ts", 33, [1, 17, 64, 200], 8, 2, 64, "f16", "e4m3", gap=5, lead=2)
    cases = [base, fw.to_paged(base, 16, 34)]
    for i, c in enumerate(cases):
        w = fw.with_scales(c, fw.SCALE_TOKEN, 35 + i, powers_of_two=True)
        a = orc.decode_attention(w)
        b = orc.decode_attention(materialize_scales(w))
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), c.name


def pin_token_scales_single_key(orc):
    """One key: out = v_scale * vs(row) * v, lse = softmax_scale * k_scale *
    ks(row) * q.k (closed form, per head)."""
    rng = np.random.default_rng(36)
    D, KVH, QH = 64, 2, 4
    q = rng.standard_normal((1, QH, D))
    k = rng.standard_normal((1, KVH, D))
    v = rng.standard_normal((1, KVH, D))
    w = custom(q, k, v, [1], kv_dtype="e4m3", softmax_scale=0.25, k_scale=0.5, v_scale=2.0,
               kv_start_idx=[3])
    w = dataclasses.replace(w, k_cache=np.concatenate([np.full((3, KVH, D), 0x7E, np.uint8), w.k_cache]),
                            v_cache=np.concatenate([np.full((3, KVH, D), 0x7E, np.uint8), w.v_cache]))
    w = fw.with_scales(w, fw.SCALE_TOKEN, 37)
    out, lse = orc.decode_attention(w)
    qf = lib_decode(w.q, "f16").reshape(QH, D)
    kf = lib_decode(w.k_cache, "e4m3")[3]
    vf = lib_decode(w.v_cache, "e4m3")[3]
    for qh in range(QH):
        h = qh // (QH // KVH)
        ks, vs = float(w.k_scales[3, h]), float(w.v_scales[3, h])
        _close(out[0, qh], 2.0 * vs * vf[h], 1e-15, 0, "single key out")
        _close(lse[0, qh], 0.25 * 0.5 * ks * float(qf[qh] @ kf[h]), 1e-12, 1e-14, "single key lse")


def pin_i8_materialized(orc):
    """An INT8 cache equals an f16 cache holding its decoded codes times the
    finer scales: per tensor, per KV head (GQA, bf16 q) and per token through
    a shuffled page pool."""
    base = fw.make_contiguous("i8", 38, [1, 33, 150], 8, 2, 64, "f16", "i8", gap=4, lead=1)
    assert base.k_cache.dtype == np.int8 and base.k_cache.min() < -100 < 100 < base.k_cache.max()
    b16 = fw.make_contiguous("i8b", 39, [5, 70], 16, 4, 128, "bf16", "i8", gap=2)
    cases = [base, fw.with_scales(b16, fw.SCALE_HEAD, 40, powers_of_two=True),
             fw.with_scales(fw.to_paged(base, 16, 41), fw.SCALE_TOKEN, 42, powers_of_two=True)]
    for w in cases:
        a = orc.decode_attention(w)
        b = orc.decode_attention(materialize_scales(w))
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), w.name


def pin_i8_single_key_all_codes(orc):
    """Sequences of one key each: out = v_scale * V code row (every code
    -128 .. 127 appears in some V row) and lse = softmax_scale * k_scale *
    q . (K code row), closed forms."""
    rng = np.random.default_rng(43)
    D = 128
    q = rng.standard_normal((2, 2, D))
    codes = np.arange(-128, 128, dtype=np.float64).reshape(2, 1, D)
    k = codes[::-1] * 0.5
    w = custom(q, k, codes, [1, 1], kv_dtype="i8", softmax_scale=0.0625, k_scale=0.25,
               v_scale=0.125)
    out, lse = orc.decode_attention(w)
    qf = lib_decode(w.q, "f16").reshape(2, 2, D)
    kf = np.clip(np.rint(k), -128, 127)
    for b in range(2):
        for qh in range(2):
            _close(out[b, qh], 0.125 * codes[b, 0], 0, 0, "i8 single key out")
            _close(lse[b, qh], 0.0625 * 0.25 * float(qf[b, qh] @ kf[b, 0]), 1e-12, 1e-14,
                   "i8 single key lse")


# ----------------------------------------------------------------------------
# KV append: encoders against library casts, placement and scales
# ----------------------------------------------------------------------------

def lib_e4m3_encode(x: np.ndarray) -> np.ndarray:
    """torch's float8_e4m3fn cast (round to nearest even) after clamping to
    the finite range, as codes."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def lib_i8_encode(x: np.ndarray) -> np.ndarray:
    return np.clip(np.rint(np.asarray(x, np.float32)), -127, 127).astype(np.int8).view(np.uint8)


def _encoder_inputs(rng):
    vals = lib_decode(np.arange(0x7F, dtype=np.uint8), "e4m3")       # every finite magnitude
    mids = (vals[:-1] + vals[1:]) / 2                                  # ties (exact in fp32)
    x = np.concatenate([vals, -vals, mids, -mids, rng.standard_normal(3000) * 60,
                        rng.standard_normal(500) * 1e-3, [448.0, 463.9, 464.0, 500.0, 1e6, -1e6,
                                                          0.0, -0.0, 1e-12, -1e-12]])
    return x.astype(np.float32)


def pin_e4m3_encoder(orc):
    x = _encoder_inputs(np.random.default_rng(44))
    got = np.array([orc.e4m3_encode(v) for v in x], np.uint8)
    ref = lib_e4m3_encode(x)
    assert np.array_equal(got, ref), f"e4m3 encode differs at {x[got != ref][:5]}"


def pin_i8_encoder(orc):
    rng = np.random.default_rng(45)
    x = np.concatenate([np.arange(-131, 132), np.arange(-131, 131) + 0.5,
                        rng.standard_normal(2000) * 50, [1e6, -1e6, 0.0, -0.0, 0.49999997]])
    x = x.astype(np.float32)
    got = np.array([orc.i8_encode(v) for v in x], np.uint8)
    assert np.array_equal(got, lib_i8_encode(x))


def _appended_rows(w, positions):
    """Cache rows the append of ``positions`` writes (row per sequence or -1)."""
    rows = []
    for b in range(w.batch):
        t = int(positions[b])
        if t < 0:
            rows.append(-1)
        elif w.paged:
            rows.append(int(w.block_table[b, t // w.page_size]) * w.page_size + t % w.page_size)
        else:
            rows.append(int(w.kv_start_idx[b]) + t)
    return rows


def _check_append(orc, w, seed, n_new=1):
    k_new, v_new = fw.new_tokens(w, seed, std=3.0, n_new=n_new)
    pos = fw.last_positions(w, n_new)
    pos[0] = -1   # the first sequence gets no append
    kc, vc, ks, vs = orc.append_kv(w, k_new, v_new, pos)
    KVH, D = w.num_kv_heads, w.head_dim
    if n_new == 1:
        k_new, v_new = k_new[:, None], v_new[:, None]
    rows = [_appended_rows(w, np.where(pos >= 0, pos + i, -1)) for i in range(n_new)]
    for cache, old, new, scale, sarr, sarr_old in (
            (kc, w.k_cache, k_new, w.k_scale, ks, w.k_scales),
            (vc, w.v_cache, v_new, w.v_scale, vs, w.v_scales)):
        c2 = cache.reshape(-1, KVH, D)
        o2 = np.asarray(old).reshape(-1, KVH, D)
        touched = np.zeros(c2.shape[0], bool)
        touched[[r for ri in rows for r in ri if r >= 0]] = True
        assert np.array_equal(c2[~touched], o2[~touched]), f"{w.name}: rows outside the append changed"
        if sarr is not None and w.scale_kind == fw.SCALE_TOKEN:
            s2 = sarr.reshape(-1, KVH)
            assert np.array_equal(s2[~touched], np.asarray(sarr_old).reshape(-1, KVH)[~touched])
        x = lib_decode(new, w.q_dtype).astype(np.float32)      # [B, n_new, KVH, D], exact
        for b, i, r in ((b, i, rows[i][b]) for i in range(n_new) for b in range(w.batch)):
            if r < 0:
                continue
            if w.kv_dtype in ("f16", "bf16"):
                assert np.array_equal(c2[r], new[b, i]), "16-bit append must store the bits"
                continue
            qmax = 448.0 if w.kv_dtype == "e4m3" else 127.0
            for h in range(KVH):
                if w.scale_kind == fw.SCALE_TOKEN:
                    seff = np.float32(scale) * np.float32(sarr.reshape(-1, KVH)[r, h])
                elif w.scale_kind == fw.SCALE_HEAD:
                    seff = np.float32(scale) * np.float32(sarr[h])
                else:
                    seff = np.float32(scale)
                q = x[b, i, h] / seff                                # numpy fp32 IEEE division
                enc = lib_e4m3_encode(q) if w.kv_dtype == "e4m3" else lib_i8_encode(q)
                assert np.array_equal(c2[r, h].view(np.uint8), enc), f"{w.name} row {r} head {h}"
                if w.scale_kind == fw.SCALE_TOKEN:
                    # the row's largest element lands on the largest code, and
                    # nothing beyond it (no element saturates)
                    top = np.abs(lib_decode(c2[r, h], w.kv_dtype)).max()
                    assert top == qmax, (w.name, top)
                    assert abs(float(np.abs(q).max()) - qmax) <= qmax * 1e-6, (w.name, np.abs(q).max())


def pin_append_kv(orc):
    """The append writes exactly the new token's rows (contiguous with gaps
    and paged), stores 16-bit elements as they are and 8-bit codes equal to
    the library casts of x / s in fp32, with per-tensor, per-head and
    per-token scales; per-token scales put each row's largest element on the
    largest code and leave other rows' scales alone."""
    cases = []
    c1 = fw.make_contiguous("ap1", 46, [5, 1, 40, 0, 200], 8, 2, 64, "f16", "e4m3", gap=2, lead=1)
    cases.append(c1)
    cases.append(fw.with_scales(c1, fw.SCALE_HEAD, 47, powers_of_two=False))
    cases.append(fw.with_scales(fw.to_paged(c1, 16, 48), fw.SCALE_TOKEN, 49))
    c2 = fw.make_contiguous("ap2", 50, [9, 3, 70, 33], 16, 4, 128, "bf16", "i8", gap=1)
    cases.append(c2)
    cases.append(fw.with_scales(fw.to_paged(c2, 8, 51), fw.SCALE_TOKEN, 52))
    cases.append(fw.with_scales(c2, fw.SCALE_HEAD, 53))
    cases.append(fw.make_contiguous("ap3", 54, [4, 17], 4, 1, 64, "f16", "f16", gap=1))
    cases.append(fw.to_paged(fw.make_contiguous("ap4", 55, [4, 17, 2], 8, 2, 128, "bf16", "bf16"),
                             4, 56))
    for i, w in enumerate(cases):
        _check_append(orc, w, 60 + i)
    # several new tokens per sequence (a verify step's drafted tokens)
    _check_append(orc, cases[2], 70, n_new=3)
    _check_append(orc, cases[3], 71, n_new=2)


# ----------------------------------------------------------------------------
# multi-token query (speculative verify): causal among the new tokens
# ----------------------------------------------------------------------------

def pin_multi_token_equals_truncated_single(orc):
    """Query token j of q_len sees exactly the first T - (q_len - 1 - j)
    keys: each token's result equals the one-token oracle on the sequence
    cut there (bit for bit), with GQA, gaps, a paged pool, finer scales and
    sequences shorter than q_len."""
    base = fw.make_contiguous("mt", 88, [1, 2, 5, 40, 0, 130], 16, 4, 64, "f16", "e4m3", gap=2,
                              q_len=4)
    cases = [base, fw.with_scales(fw.to_paged(base, 8, 89), fw.SCALE_TOKEN, 90),
             fw.with_q_len(fw.make_contiguous("mt2", 91, [3, 77], 8, 1, 128, "bf16", "bf16"), 3, 92)]
    for w in cases:
        L = w.q_len
        out, lse = orc.decode_attention(w)
        assert out.shape == (w.batch, w.num_q_heads, L, w.head_dim)
        for j in range(L):
            cut = np.maximum(w.seq_len.astype(np.int64) - (L - 1 - j), 0).astype(np.int32)
            wj = dataclasses.replace(w, q=np.ascontiguousarray(w.q[:, :, j]), q_len=1, seq_len=cut)
            o1, l1 = orc.decode_attention(wj)
            assert np.array_equal(out[:, :, j], o1), (w.name, j)
            assert np.array_equal(lse[:, :, j], l1), (w.name, j)


def pin_multi_token_closed_form(orc):
    """All keys new (T = q_len) and identical: token j's weights are uniform
    over keys 0..j, so out_j = mean(v_0..v_j) and lse_j = s + ln(j + 1)."""
    rng = np.random.default_rng(93)
    L, D = 5, 64
    q = rng.standard_normal((1, 2, L, D))
    k = np.repeat(rng.standard_normal((1, 1, D)), L, axis=0)
    v = rng.standard_normal((L, 1, D))
    w = custom(q.reshape(1, 2 * L, D), k, v, [L], softmax_scale=0.125)
    w = dataclasses.replace(w, q=w.q.reshape(1, 2, L, D), num_q_heads=2, q_len=L)
    out, lse = orc.decode_attention(w)
    qf = lib_decode(w.q, "f16").reshape(2, L, D)
    kf = lib_decode(w.k_cache, "f16")[0, 0]
    vf = lib_decode(w.v_cache, "f16")[:, 0]
    for h in range(2):
        for j in range(L):
            _close(out[0, h, j], vf[: j + 1].mean(axis=0), 1e-14, 1e-15, "multi-token mean")
            _close(lse[0, h, j], 0.125 * float(qf[h, j] @ kf) + math.log(j + 1), 1e-13, 1e-14,
                   "multi-token lse")


ALL_PINS = [
    pin_e4m3_codes, pin_i8_codes, pin_i8_materialized, pin_i8_single_key_all_codes, pin_f16_codes, pin_bf16_codes, pin_identical_v_rows, pin_single_key,
    pin_zero_query, pin_identical_k_rows, pin_two_keys, pin_dominant_key, pin_empty_sequence,
    pin_weights_sum_to_one, pin_key_permutation, pin_gqa_equals_replicated_mha,
    pin_paged_equals_contiguous, pin_scale_factors, pin_score_shift, pin_online_recurrence,
    pin_head_scales_materialized, pin_token_scales_materialized, pin_token_scales_single_key,
    pin_e4m3_encoder, pin_i8_encoder, pin_append_kv, pin_multi_token_equals_truncated_single,
    pin_multi_token_closed_form,
]
