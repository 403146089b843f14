"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, for the five decode workloads at full size and for
edge cases (empty and one-token sequences, lengths around tile and page
boundaries, poisoned gaps and pages, every head grouping, both head
dimensions, every dtype pair, page sizes 1 .. 256)."""
import dataclasses
import functools

import numpy as np
import pytest
import torch

import fd_workloads as fw
import oracle
from gpu_util import lib, parity, run

pytestmark = pytest.mark.gpu

SIMT, MMA = 1, 2


def kernels_for(w):
    fda = lib()
    ks = []
    for k in (SIMT, MMA):
        fda.fd_set_kernel(k)
        sel = fda.fd_selected_kernel(w.num_q_heads, w.num_kv_heads, w.head_dim,
                                     0 if w.q_dtype == "f16" else 1,
                                     fda.DTYPE_CODES[w.kv_dtype], w.paged,
                                     max(w.page_size, 1))
        fda.fd_set_kernel(0)
        if sel == k:
            ks.append(k)
    return ks


@functools.lru_cache(maxsize=None)
def config(n):
    return fw.WORKLOADS[n]()


@functools.lru_cache(maxsize=None)
def oracle_of(n):
    return oracle.decode_attention(config(n))


def check_workload(w, ref=None, label=""):
    if ref is None:
        ref = oracle.decode_attention(w)
    ks = kernels_for(w)
    assert ks, "no kernel supports this case"
    for k in ks:
        out, lse, _, _ = run(w, k)
        parity(w, out, lse, ref[0], ref[1], label=f"{label or w.name} kernel={k}")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_config_full_size(n):
    check_workload(config(n), oracle_of(n), label=f"config{n}")


EDGE_LENGTHS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 1000]


@pytest.mark.parametrize("q_dtype,kv_dtype", [("f16", "f16"), ("bf16", "bf16"), ("f16", "e4m3"),
                                              ("bf16", "e4m3"), ("f16", "i8"), ("bf16", "i8")])
@pytest.mark.parametrize("D", [64, 128])
def test_edge_lengths_with_poisoned_gaps(q_dtype, kv_dtype, D):
    w = fw.make_contiguous(f"edge-{q_dtype}-{kv_dtype}-{D}", 100 + D, EDGE_LENGTHS, 8, 2, D,
                           q_dtype, kv_dtype, gap=3, lead=5, tail=7)
    check_workload(w)


NAN_BITS = {"e4m3": 0x7F, "f16": 0x7E00, "bf16": 0x7FC0}


def _fill_unowned_rows_with_nan(w):
    """Every cache row no sequence owns (gaps between sequences, page tails,
    unused pages) gets a NaN bit pattern; the oracle never reads them."""
    nan = NAN_BITS[w.kv_dtype]
    k, v = w.k_cache.copy(), w.v_cache.copy()
    if w.paged:
        owned = np.zeros(k.shape[:2], dtype=bool)       # [pages, page_size]
        for b in range(w.batch):
            T = int(w.seq_len[b])
            for j in range(-(-T // w.page_size)):
                owned[w.block_table[b, j], : min(w.page_size, T - j * w.page_size)] = True
    else:
        owned = np.zeros(k.shape[0], dtype=bool)
        for b in range(w.batch):
            s = int(w.kv_start_idx[b])
            owned[s:s + int(w.seq_len[b])] = True
    k[~owned] = nan
    v[~owned] = nan
    import dataclasses
    return dataclasses.replace(w, k_cache=k, v_cache=v)


@pytest.mark.parametrize("kv_dtype,P", [("e4m3", 0), ("e4m3", 16), ("e4m3", 64), ("f16", 0),
                                        ("f16", 16), ("bf16", 32), ("e4m3", 4), ("f16", 2)])
@pytest.mark.parametrize("qh,kvh", [(16, 2), (8, 8), (16, 1)])
def test_nan_in_rows_outside_sequences_never_leaks(kv_dtype, P, qh, kvh):
    """Rows past a sequence's end are loaded with its last tile (box rows,
    page tails): whatever bytes they hold must not reach the outputs."""
    q_dtype = "bf16" if kv_dtype == "bf16" else "f16"
    w = fw.make_contiguous(f"nan-{kv_dtype}-{P}-{qh}-{kvh}", 41, [100, 37, 300, 1, 0, 129], qh, kvh,
                           128, q_dtype, kv_dtype, gap=5, lead=3, tail=9)
    if P:
        w = fw.to_paged(w, P, 42)
    w = _fill_unowned_rows_with_nan(w)
    check_workload(w)


@pytest.mark.parametrize("P,shared", [(16, 256), (64, 1024), (64, 5000)])
def test_shared_prefix_pages(P, shared):
    """Block tables whose first entries alias the same physical pages
    (prefix-cache hits): read through the table like any other page."""
    base = fw.make_contiguous(f"prefix-{P}-{shared}", 51, [3000, 2048, 1500, 900, 64, 4500, 17, 0],
                              64, 8, 128, "f16", "e4m3", gap=2)
    w = fw.share_prefix(fw.to_paged(base, P, 52), shared)
    assert (w.block_table[1, :4] == w.block_table[0, :4]).all()
    check_workload(w)


@pytest.mark.parametrize("kv", ["e4m3", "i8"])
@pytest.mark.parametrize("kind", [fw.SCALE_HEAD, fw.SCALE_TOKEN], ids=["head", "token"])
@pytest.mark.parametrize("layout", [0, 16, 64], ids=["contiguous", "paged16", "paged64"])
@pytest.mark.parametrize("qh,kvh,qdt", [(64, 8, "f16"), (16, 1, "bf16"), (32, 4, "f16")])
def test_finer_kv_scales(kv, kind, layout, qh, kvh, qdt):
    """Per-KV-head and per-token FP8 / INT8 scales (fd_decode_attention_scaled).
    The bf16 bar (max-abs 1.6e-2) assumes outputs of the per-tensor workloads'
    size, and bf16 rounding grows with the value: the bf16 cases draw scales
    that keep the outputs there."""
    base = fw.make_contiguous(f"scales-{kv}-{kind}-{layout}-{qh}-{kvh}", 61,
                              [1, 100, 1000, 4097, 0, 33], qh, kvh, 128, qdt, kv, gap=3, lead=2)
    if layout:
        base = fw.to_paged(base, layout, 62)
    span = (0.25, 1.0) if qdt == "bf16" else (0.5, 2.0)
    check_workload(fw.with_scales(base, kind, 63, span=span))


@pytest.mark.parametrize("n,kind", [(4, fw.SCALE_TOKEN), (5, fw.SCALE_HEAD), (3, fw.SCALE_TOKEN)])
def test_config_full_size_finer_scales(n, kind):
    check_workload(fw.with_scales(config(n), kind, 64 + n), label=f"config{n}-scales{kind}")


@pytest.mark.parametrize("n,kind", [(3, fw.SCALE_TENSOR), (4, fw.SCALE_TENSOR), (5, fw.SCALE_TENSOR),
                                    (5, fw.SCALE_TOKEN)])
def test_config_full_size_int8(n, kind):
    """The 8-bit workloads with the same draws quantised to INT8."""
    w = fw.WORKLOADS[n](kv_dtype="i8")
    assert w.k_cache.dtype == np.int8
    if kind:
        w = fw.with_scales(w, kind, 74 + n)
    check_workload(w, label=f"config{n}-i8-scales{kind}")


@pytest.mark.parametrize("D,kvh", [(128, 8), (64, 1)])
def test_int8_one_signed_queries(D, kvh):
    """INT8 keys with f16 queries are widened biased (1152 + code) and the
    score subtracts 1152 * sum(q): queries of one sign make sum(q) large,
    the hardest case for that fold's fp32 accumulation."""
    w = fw.make_contiguous(f"i8-posq-{D}-{kvh}", 90 + D + kvh, [5, 600, 4000, 33], 8 * kvh, kvh, D,
                           "f16", "i8", gap=1)
    q = np.abs(w.q.view(np.float16).astype(np.float32)) * 2.0
    w = dataclasses.replace(w, q=fw.f32_to_f16_bits(q).view(w.q.dtype))
    check_workload(w)


@pytest.mark.parametrize("qh,kvh,D,P", [(16, 1, 64, 0), (64, 8, 128, 32), (40, 5, 128, 0),
                                        (8, 8, 64, 1), (32, 4, 128, 256)])
def test_int8_shapes(qh, kvh, D, P):
    """INT8 caches across head groupings, both head dims and page sizes."""
    w = fw.make_contiguous(f"i8-{qh}-{kvh}-{D}-{P}", 80 + qh + P, [3, 257, 1900, 0, 64], qh, kvh, D,
                           "bf16" if qh == 40 else "f16", "i8", gap=2, lead=1)
    if P:
        w = fw.to_paged(w, P, 81)
    check_workload(w)


@pytest.mark.parametrize("qh,kvh", [(8, 8), (8, 4), (16, 4), (32, 4), (64, 8), (16, 1), (32, 1),
                                    (64, 1), (128, 1), (12, 3), (40, 5)])
def test_head_groupings(qh, kvh):
    w = fw.make_contiguous(f"heads-{qh}-{kvh}", 200 + qh + kvh, [5, 130, 777], qh, kvh, 128,
                           "f16", "e4m3", gap=2)
    check_workload(w)


@pytest.mark.parametrize("P", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_paged_page_sizes(P):
    lens = [1, P - 1 if P > 1 else 2, P, P + 1, 3 * P + 5, 700]
    base = fw.make_contiguous(f"paged{P}", 300 + P, lens, 16, 2, 128, "f16", "e4m3")
    w = fw.to_paged(base, P, 301 + P, extra_stride=2)
    check_workload(w)


@pytest.mark.parametrize("P,D,kv,qh,kvh", [(2, 64, "e4m3", 16, 2), (8, 64, "e4m3", 64, 8),
                                           (4, 128, "bf16", 32, 8), (1, 64, "f16", 8, 8),
                                           (4, 128, "i8", 64, 8)])
def test_small_pages_on_tensor_cores(P, D, kv, qh, kvh):
    """Pages too small for a TMA box to start on a swizzle atom: the
    tensor-core kernel gathers their rows itself, and is what AUTO picks."""
    q = "bf16" if kv == "bf16" else "f16"
    base = fw.make_contiguous(f"small-pages{P}-{D}-{kv}", 330 + P + D, [1, 3, 9, 31, 200, 1100],
                              qh, kvh, D, q, kv)
    w = fw.to_paged(base, P, 331 + P)
    fda = lib()
    assert fda.fd_selected_kernel(w.num_q_heads, w.num_kv_heads, w.head_dim,
                                  0 if q == "f16" else 1, fda.DTYPE_CODES[kv], 1, P) == MMA
    check_workload(w)


def test_all_sequences_empty():
    w = fw.make_contiguous("empty", 7, [0, 0, 0], 8, 2, 128, "f16", "f16")
    ref = oracle.decode_attention(w)
    for k in kernels_for(w):
        out, lse, _, _ = run(w, k)
        assert np.all(out == 0) and np.all(np.isneginf(lse))
        parity(w, out, lse, ref[0], ref[1], label=f"empty kernel={k}")


def test_many_short_sequences():
    rng = np.random.default_rng(8)
    lens = rng.integers(0, 40, size=600)
    w = fw.make_contiguous("many-short", 8, lens, 32, 8, 128, "bf16", "e4m3", gap=1)
    check_workload(w)


def test_one_long_sequence_many_splits():
    w = fw.make_contiguous("one-long", 9, [200_003], 16, 1, 128, "f16", "e4m3")
    check_workload(w)


def test_paged_equals_contiguous_bitwise():
    base = fw.make_contiguous("pc", 10, [1, 64, 65, 1000, 4097], 64, 8, 128, "f16", "e4m3")
    paged = fw.to_paged(base, 64, 11)
    for k in kernels_for(base):
        if k not in kernels_for(paged):
            continue
        _, _, o1, l1 = run(base, k)
        _, _, o2, l2 = run(paged, k)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)), f"kernel={k}"
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32)), f"kernel={k}"


def test_repeated_calls_are_bitwise_identical():
    w = config(4)
    for k in kernels_for(w):
        _, _, o1, l1 = run(w, k)
        _, _, o2, l2 = run(w, k)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_nondefault_stream():
    w = fw.make_contiguous("stream", 12, [100, 2000], 16, 2, 128, "f16", "e4m3")
    ref = oracle.decode_attention(w)
    s = torch.cuda.Stream()
    out, lse, _, _ = run(w, 0, stream=s)
    parity(w, out, lse, ref[0], ref[1], label="side stream")


def test_cache_offsets_beyond_int32_elements():
    """Sequences whose rows lie past 2^31 cache elements (8 KV heads x 128
    dims = 1024 elements per row, rows from 2.1 M on): every element offset
    the kernels form must be 64-bit.  Contiguous and paged (page ids above
    2^31 / (16 x 1024))."""
    import dataclasses
    lead = 2_100_000
    w = fw.make_contiguous("beyond-int32", 90, [5, 300, 1000], 64, 8, 128, "f16", "e4m3", lead=lead)
    assert w.kv_rows * 8 * 128 > 2 ** 31
    check_workload(w)
    # paged: the same rows at page ids from 135,000 on in a 140,000-page pool
    P, pool, base = 16, 140_000, 135_000
    assert base * P * 8 * 128 > 2 ** 31
    k = np.full((pool, P, 8, 128), fw.POISON_E4M3, np.uint8)
    v = np.full((pool, P, 8, 128), fw.POISON_E4M3, np.uint8)
    npages = [-(-int(t) // P) for t in w.seq_len]
    table = np.full((w.batch, max(npages)), -1, np.int32)
    nxt = base
    for b in range(w.batch):
        s0, T = int(w.kv_start_idx[b]), int(w.seq_len[b])
        for j in range(npages[b]):
            lo, hi = j * P, min(T, (j + 1) * P)
            k[nxt, : hi - lo] = w.k_cache[s0 + lo:s0 + hi]
            v[nxt, : hi - lo] = w.v_cache[s0 + lo:s0 + hi]
            table[b, j] = nxt
            nxt += 1
    wp = dataclasses.replace(w, name="beyond-int32-paged16", k_cache=k, v_cache=v, page_size=P,
                             kv_start_idx=None, block_table=table)
    check_workload(wp)


@pytest.mark.parametrize("qh,kvh", [(64, 8), (16, 16)])
def test_multi_token_max_q_len(qh, kvh):
    """q_len 16, the largest: with 8 query heads per KV head that is 128 rows
    per KV head (8 MMA row tiles)."""
    w = fw.make_contiguous(f"q16-{qh}-{kvh}", 91, [1, 16, 17, 500], qh, kvh, 128, "f16", "e4m3",
                           gap=1, q_len=16)
    ref = oracle.decode_attention(w)
    fda = lib()
    ks = []
    for k in (SIMT, MMA):
        fda.fd_set_kernel(k)
        if fda.fd_selected_kernel(qh * 16, kvh, 128, 0, 2, 0, 1) == k:
            ks.append(k)
        fda.fd_set_kernel(0)
    assert ks
    for k in ks:
        out, lse, _, _ = run(w, k)
        parity(w, out, lse, ref[0], ref[1], label=f"{w.name} kernel={k}")


def test_many_sequences():
    """4,000 short sequences: thousands of streams for the plan's multi-pass
    branch and the combine."""
    rng = np.random.default_rng(92)
    lens = rng.integers(0, 70, size=4000)
    w = fw.make_contiguous("many-4000", 93, lens, 16, 2, 128, "f16", "e4m3", gap=1)
    check_workload(w)
