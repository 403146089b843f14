"""Seeded random parity cases against the oracle, on every split kernel that
takes each case: batch sizes, ragged and empty sequences, head layouts
(MHA, GQA, MQA), head_dim, query and cache dtypes, contiguous caches with
gaps or paged pools of every page size, finer K/V scales and query tokens
per sequence are drawn together, so that combinations no hand-written case
names still meet the parity bar."""
import numpy as np
import pytest

import fd_workloads as fw
import oracle
from gpu_util import lib, parity, run

pytestmark = pytest.mark.gpu

KERNELS = (0, 1, 2, 3, 4)   # the library's choice, then each kernel forced
N_CASES = 40
N_LARGE = 24


def _case(i):
    rng = np.random.default_rng(9000 + i)
    kvh = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8, 16, 32]))
    qh = kvh * g
    D = int(rng.choice([64, 128]))
    kv = str(rng.choice(["e4m3", "e4m3", "i8", "f16", "bf16"]))
    qdt = kv if kv in ("f16", "bf16") else str(rng.choice(["f16", "bf16"]))
    q_len = int(rng.choice([1, 1, 1, 2, 4]))
    if g * q_len > 128:
        q_len = 1
    B = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.choice([0, 1, 2, 31, 64, 65, 200, 1000, 3000], size=B)]
    w = fw.make_contiguous(f"fuzz-{i}", 9100 + i, lens, qh, kvh, D, qdt, kv,
                           gap=int(rng.integers(0, 4)), lead=int(rng.integers(0, 3)),
                           q_len=q_len)
    if rng.random() < 0.5:
        w = fw.to_paged(w, int(rng.choice([1, 2, 4, 8, 16, 64, 128])), 9200 + i)
    if kv in ("e4m3", "i8") and rng.random() < 0.4:
        kind = fw.SCALE_HEAD if rng.random() < 0.5 else fw.SCALE_TOKEN
        # (bf16 outputs: the span the bf16 bound is sized for, as in the other tests)
        w = fw.with_scales(w, kind, 9300 + i, span=(0.25, 1.0) if qdt == "bf16" else (0.5, 2.0))
    return w


def _large_group_case(i):
    """One or two KV heads with 16 to 128 query rows each (query heads times
    query tokens), FP8-e4m3 or 16-bit caches, longer sequences: the shapes
    on which the library's own choice can be the tcgen05 kernel."""
    rng = np.random.default_rng(9500 + i)
    kvh = int(rng.choice([1, 1, 2]))
    q_len = int(rng.choice([1, 1, 2, 4, 8]))
    g = int(rng.choice([g for g in (8, 16, 32, 64, 128) if g * q_len <= 128]))
    kv = str(rng.choice(["e4m3", "e4m3", "e4m3", "f16"]))
    qdt = "f16" if kv == "e4m3" and rng.random() < 0.8 else ("f16" if kv == "f16" else "bf16")
    B = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.choice([0, 1, 63, 64, 65, 127, 128, 129, 700, 4000, 9000], size=B)]
    w = fw.make_contiguous(f"fuzz-large-{i}", 9600 + i, lens, kvh * g, kvh, 128, qdt, kv,
                           gap=int(rng.integers(0, 3)), lead=int(rng.integers(0, 2)), q_len=q_len)
    if rng.random() < 0.5:
        w = fw.to_paged(w, int(rng.choice([8, 16, 32, 64, 128, 256])), 9700 + i)
    if kv == "e4m3" and rng.random() < 0.3:
        w = fw.with_scales(w, fw.SCALE_HEAD, 9800 + i, span=(0.5, 2.0) if qdt == "f16" else (0.25, 1.0))
    return w


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_every_kernel(i):
    _every_kernel(_case(i))


@pytest.mark.parametrize("i", range(N_LARGE))
def test_random_large_group_every_kernel(i):
    _every_kernel(_large_group_case(i))


def _every_kernel(w):
    fda = lib()
    ref = oracle.decode_attention(w)
    ran = 0
    for k in KERNELS:
        fda.fd_set_kernel(k)
        try:
            sel = fda.fd_selected_kernel_scaled(w.num_q_heads * w.q_len, w.num_kv_heads,
                                                w.head_dim, 0 if w.q_dtype == "f16" else 1,
                                                fda.DTYPE_CODES[w.kv_dtype], w.paged,
                                                max(w.page_size, 1), w.scale_kind)
        finally:
            fda.fd_set_kernel(0)
        if sel == -1:
            # the selection hook and the call agree: the call is refused
            assert k != 0, "the library's own choice refused a supported case"
            with pytest.raises(fda.FdError) as e:
                run(w, k)
            assert e.value.status == fda.FD_ERR_UNSUPPORTED
            continue
        assert k == 0 or sel == k, (k, sel)
        out, lse, _, _ = run(w, k)
        parity(w, out, lse, ref[0], ref[1], label=f"{w.name} kernel={k} (ran {sel})")
        ran += 1
    assert ran >= 1, "no kernel took the case"
