"""GPU parity of multi-token query decode (fd_decode_attention_multi: q_len
query tokens per sequence, causal among the last q_len cached tokens) against
the oracle, on every split kernel that takes the shape."""
import functools

import pytest

import fd_workloads as fw
import oracle
from gpu_util import lib, parity, run

pytestmark = pytest.mark.gpu

SIMT, MMA, TC = 1, 2, 3


def kernels_for(w):
    fda = lib()
    ks = []
    for k in (SIMT, MMA, TC):
        fda.fd_set_kernel(k)
        sel = fda.fd_selected_kernel(w.num_q_heads * w.q_len, w.num_kv_heads, w.head_dim,
                                     0 if w.q_dtype == "f16" else 1,
                                     fda.DTYPE_CODES[w.kv_dtype], w.paged, max(w.page_size, 1))
        fda.fd_set_kernel(0)
        if sel == k:
            ks.append(k)
    return ks


def check(w, ref=None, label=""):
    if ref is None:
        ref = oracle.decode_attention(w)
    ks = kernels_for(w)
    assert ks, "no kernel supports this case"
    for k in ks:
        out, lse, _, _ = run(w, k)
        parity(w, out, lse, ref[0], ref[1], label=f"{label or w.name} kernel={k}")


# lengths include sequences shorter than q_len (their first tokens see no key)
LENS = [1, 2, 3, 17, 64, 65, 300, 0, 1000]


@pytest.mark.parametrize("q_len", [2, 3, 4, 8])
@pytest.mark.parametrize("qh,kvh,qdt,kv", [(64, 8, "f16", "e4m3"), (16, 1, "f16", "e4m3"),
                                           (32, 8, "bf16", "bf16"), (8, 8, "f16", "f16"),
                                           (16, 2, "bf16", "i8")])
def test_multi_token_contiguous(q_len, qh, kvh, qdt, kv):
    if (qh // kvh) * q_len > 128:
        pytest.skip("group * q_len above 128")
    w = fw.make_contiguous(f"multi-{q_len}-{qh}-{kvh}-{kv}", 500 + q_len, LENS, qh, kvh, 128, qdt,
                           kv, gap=3, lead=1, q_len=q_len)
    check(w)


@pytest.mark.parametrize("P", [1, 16, 64])
@pytest.mark.parametrize("q_len", [2, 4])
def test_multi_token_paged(P, q_len):
    """Page size 1 runs on the CUDA-core kernel only, which takes groups
    (query heads x tokens per KV head) of up to 16 or multiples of 16."""
    base = fw.make_contiguous(f"multi-paged-{P}-{q_len}", 520 + P, LENS, 32, 4, 64, "f16", "e4m3",
                              q_len=q_len)
    check(fw.to_paged(base, P, 521))


@pytest.mark.parametrize("kind", [fw.SCALE_HEAD, fw.SCALE_TOKEN], ids=["head", "token"])
def test_multi_token_finer_scales(kind):
    base = fw.make_contiguous(f"multi-scales-{kind}", 530, LENS, 64, 8, 128, "f16", "e4m3", gap=1,
                              q_len=2)
    check(fw.with_scales(base, kind, 531))


@functools.lru_cache(maxsize=None)
def verify_workload(n, q_len):
    return fw.with_q_len(fw.WORKLOADS[n](), q_len, 540 + n)


@pytest.mark.parametrize("n,q_len", [(4, 2), (4, 4), (5, 4), (5, 8), (3, 2)])
def test_config_full_size_multi_token(n, q_len):
    """The decode workloads as verify steps: on the FP8 paged one, 2 tokens fill
    the 16-row MMA tile (8 query heads x 2 tokens per KV head)."""
    w = verify_workload(n, q_len)
    check(w, label=f"config{n}-q{q_len}")
