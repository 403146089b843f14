"""GPU parity of the CUDA-core FMA form of the split kernel (FD_KERNEL_FMA: the
mma.sync kernel's TMA pipeline and plan with FMA arithmetic) against the
oracle, on the shapes it takes: FP8-e4m3 caches, head_dim 128, at most 8 query
rows per KV head, KV heads a multiple of 8."""
import numpy as np
import pytest

import fd_workloads as fw
import oracle
from gpu_util import lib, parity, run

pytestmark = pytest.mark.gpu

FMA = 4
LENS = [0, 1, 31, 32, 33, 100, 700, 5000, 2]


def check(w, label=""):
    fda = lib()
    fda.fd_set_kernel(FMA)
    try:
        sel = fda.fd_selected_kernel(w.num_q_heads * w.q_len, w.num_kv_heads, w.head_dim,
                                     0 if w.q_dtype == "f16" else 1, fda.DTYPE_CODES[w.kv_dtype],
                                     w.paged, max(w.page_size, 1))
    finally:
        fda.fd_set_kernel(0)
    assert sel == FMA, "the FMA form does not take this shape"
    ref = oracle.decode_attention(w)
    out, lse, _, _ = run(w, FMA)
    parity(w, out, lse, ref[0], ref[1], label=label or w.name)


@pytest.mark.parametrize("qh,kvh,qdt", [(64, 8, "f16"), (32, 8, "f16"), (8, 8, "f16"),
                                         (64, 8, "bf16"), (128, 16, "f16")])
def test_fma_contiguous(qh, kvh, qdt):
    w = fw.make_contiguous(f"fma-{qh}-{kvh}-{qdt}", 700 + qh, LENS, qh, kvh, 128, qdt, "e4m3",
                           gap=3, lead=1, tail=2)
    check(w)


@pytest.mark.parametrize("P", [8, 16, 64, 128])
def test_fma_paged(P):
    base = fw.make_contiguous(f"fma-paged-{P}", 710 + P, LENS, 64, 8, 128, "f16", "e4m3")
    check(fw.to_paged(base, P, 711 + P))


def test_fma_head_scales():
    base = fw.make_contiguous("fma-head-scales", 720, LENS, 64, 8, 128, "f16", "e4m3", gap=1)
    check(fw.with_scales(base, fw.SCALE_HEAD, 721))


def test_fma_multi_token():
    """Two query tokens of 4 heads per KV head: 8 rows, causal among them."""
    w = fw.make_contiguous("fma-q2", 730, [1, 2, 3] + LENS, 32, 8, 128, "f16", "e4m3", q_len=2)
    check(w)


def test_fma_config4_full_size():
    """The FP8 paged decode workload, whole outputs against the oracle."""
    check(fw.WORKLOADS[4](), label="config4-fma")


@pytest.mark.parametrize("qh,kvh,kv,D", [(16, 2, "e4m3", 128),   # 2 KV heads: no 8-head stream
                                         (128, 8, "e4m3", 128),  # 16 rows per KV head
                                         (64, 8, "i8", 128), (64, 8, "f16", 128),
                                         (64, 8, "e4m3", 64)])
def test_fma_refuses(qh, kvh, kv, D):
    fda = lib()
    fda.fd_set_kernel(FMA)
    try:
        sel = fda.fd_selected_kernel(qh, kvh, D, 0, fda.DTYPE_CODES[kv], 0, 1)
    finally:
        fda.fd_set_kernel(0)
    assert sel == -1
