"""GPU parity of the tcgen05 split kernel (FD_KERNEL_TC: query groups of 17..128
rows per KV head, FP8-e4m3 caches, fp16 queries, head_dim 128) against the
oracle: one-token decode with large GQA/MQA groups, multi-token verify steps,
ragged and empty sequences, gaps between sequences, paged pools, per-KV-head
scales, and the shapes that the kernel must refuse."""
import numpy as np
import pytest

import fd_workloads as fw
import oracle
from gpu_util import lib, parity, run

pytestmark = pytest.mark.gpu

TC = 3

# empty, 1-token, tile-edge (63, 64, 65), several tiles, long sequences
LENS = [0, 1, 63, 64, 65, 129, 700, 5000, 2, 0, 31]


def selected(w):
    fda = lib()
    fda.fd_set_kernel(TC)
    try:
        return fda.fd_selected_kernel(w.num_q_heads * w.q_len, w.num_kv_heads, w.head_dim,
                                      0 if w.q_dtype == "f16" else 1, fda.DTYPE_CODES[w.kv_dtype],
                                      w.paged, max(w.page_size, 1))
    finally:
        fda.fd_set_kernel(0)


def check(w, label=""):
    assert selected(w) == TC, "the tcgen05 kernel does not take this shape"
    ref = oracle.decode_attention(w)
    out, lse, _, _ = run(w, TC)
    parity(w, out, lse, ref[0], ref[1], label=label or w.name)


@pytest.mark.parametrize("qh,kvh", [(32, 1), (24, 1), (64, 2), (128, 1), (17, 1), (96, 1)])
def test_tc_one_token_groups(qh, kvh):
    """Rows per KV head from 17 to 128 (M = 64 up to 64 rows, else 128)."""
    w = fw.make_contiguous(f"tc-{qh}-{kvh}", 600 + qh, LENS, qh, kvh, 128, "f16", "e4m3", gap=5,
                           lead=2, tail=3)
    check(w)


@pytest.mark.parametrize("qh,kvh,q_len", [(16, 1, 4), (16, 2, 3), (8, 1, 16), (64, 8, 4),
                                          (32, 8, 8), (12, 1, 2), (16, 1, 8)])
def test_tc_multi_token(qh, kvh, q_len):
    """Verify steps: q_len tokens per query head, causal among themselves."""
    w = fw.make_contiguous(f"tc-multi-{qh}-{kvh}-{q_len}", 610 + q_len, [1, 2, 3] + LENS, qh, kvh,
                           128, "f16", "e4m3", gap=3, lead=1, q_len=q_len)
    check(w)


@pytest.mark.parametrize("P", [8, 16, 32, 64, 128, 256])
def test_tc_paged(P):
    base = fw.make_contiguous(f"tc-paged-{P}", 620 + P, LENS, 48, 2, 128, "f16", "e4m3")
    check(fw.to_paged(base, P, 621 + P))


@pytest.mark.parametrize("P,q_len", [(16, 4), (64, 2), (8, 8)])
def test_tc_paged_multi_token(P, q_len):
    base = fw.make_contiguous(f"tc-paged-multi-{P}-{q_len}", 630 + P, [1, 2] + LENS, 16, 1, 128,
                              "f16", "e4m3", q_len=q_len)
    check(fw.to_paged(base, P, 631 + P))


def test_tc_head_scales():
    base = fw.make_contiguous("tc-head-scales", 640, LENS, 64, 2, 128, "f16", "e4m3", gap=1)
    check(fw.with_scales(base, fw.SCALE_HEAD, 641))


def test_tc_large_scores():
    """Scores spread wide (a large softmax scale): the running maximum moves
    by more than 2^8 between tiles, so O is rescaled in tensor memory."""
    w = fw.make_contiguous("tc-wide", 650, [4000, 129, 3000], 32, 1, 128, "f16", "e4m3",
                           softmax_scale=1.5)
    check(w)


def test_tc_many_segments():
    """More streams than SMs and long ones: every CTA starts several segments
    (Q and O buffers alternate) and streams are split across CTAs."""
    rng = np.random.default_rng(660)
    w = fw.make_contiguous("tc-many", 661, list(rng.integers(0, 3000, 300)), 64, 2, 128, "f16",
                           "e4m3", gap=2)
    check(w)


@pytest.mark.parametrize("qh,kvh,q_len,qdt,kv,D,paged,P", [
    (16, 1, 1, "f16", "e4m3", 128, 0, 1),    # 16 rows: the mma.sync kernel's shape
    (32, 1, 1, "bf16", "e4m3", 128, 0, 1),   # bf16 queries
    (32, 1, 1, "f16", "i8", 128, 0, 1),      # INT8 cache
    (32, 1, 1, "f16", "f16", 128, 0, 1),     # 16-bit cache
    (32, 1, 1, "f16", "e4m3", 64, 0, 1),     # head_dim 64
    (32, 1, 1, "f16", "e4m3", 128, 1, 4),    # pages under a swizzle atom
])
def test_tc_refuses(qh, kvh, q_len, qdt, kv, D, paged, P):
    fda = lib()
    fda.fd_set_kernel(TC)
    try:
        sel = fda.fd_selected_kernel(qh * q_len, kvh, D, 0 if qdt == "f16" else 1,
                                     fda.DTYPE_CODES[kv], paged, P)
    finally:
        fda.fd_set_kernel(0)
    assert sel == -1


def test_tc_bad_page_is_reported():
    """A block-table entry outside the pool: recorded as a device error, the
    tile skipped, and the sequence that does not touch it stays exact."""
    fda = lib()
    base = fw.make_contiguous("tc-bad", 670, [300, 500], 64, 2, 128, "f16", "e4m3")
    w = fw.to_paged(base, 16, 671)
    bt = w.block_table.copy()
    pool_pages = w.k_cache.shape[0]
    bt[1, 3] = pool_pages + 5
    w.block_table = bt
    assert selected(w) == TC
    ref = oracle.decode_attention(fw.to_paged(base, 16, 671))
    ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    out, lse, _, _ = run(w, TC, workspace=ws, check_errors=False)
    st, info = fda.fd_check_device_error(ws)
    assert st == fda.FD_ERR_DEVICE_BOUNDS and info == pool_pages + 5, (st, info)
    assert np.all(np.isfinite(out))
    sub = fw.to_paged(base, 16, 671)
    parity(sub, out[:1], lse[:1], ref[0][:1], ref[1][:1], label="tc-bad seq0")


def test_tc_config5_q_len4_full_size():
    """The long-context MQA workload as a 4-token verify step (64 rows per KV
    head) on the tcgen05 kernel, whole outputs against the oracle."""
    w = fw.with_q_len(fw.WORKLOADS[5](), 4, 545)
    check(w, label="config5-q4-tc")
