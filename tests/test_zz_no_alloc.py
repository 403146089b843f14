"""The allocation-free entry point, for callers that cannot allocate device
memory themselves (for example plugins of a framework whose allocator they
cannot reach, or code bound to a fixed memory budget).

fd_decode_attention_noalloc takes its scratch memory from a fixed array inside
the library instead of a caller workspace.  These checks call it through the C
ABI twice in a row and compare each result with the CPU oracle at the parity
bar, and with fd_decode_attention's on the same inputs bit for bit (the same
kernels run the same plan, so leftover scratch from an earlier call must not
change a single bit); they also check that sizes needing more scratch than the
array holds are refused before any launch.  The file is named so that pytest
collects it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

import fd_workloads as fw
from gpu_util import lib, parity

pytestmark = pytest.mark.gpu


def _cases():
    return [
        fw.tiny_mqa(),
        fw.to_paged(fw.make_contiguous("noalloc-paged", 31, [1, 70, 700, 3000], 64, 8, 128, "f16",
                                       "e4m3"), 64, 32),
        fw.make_contiguous("noalloc-long", 33, [60000, 5], 16, 1, 128, "f16", "e4m3"),
        fw.make_contiguous("noalloc-bf16", 34, [4096, 17], 32, 8, 128, "bf16", "bf16"),
    ]


def _with_workspace(fda, w, t):
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device="cuda")
    ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    fda.fd_decode_attention(t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"],
                            t["seq_len"], w.kv_rows, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            w.page_size, float(w.softmax_scale), float(w.k_scale),
                            float(w.v_scale), out, lse, ws)
    torch.cuda.synchronize()
    assert fda.fd_check_device_error(ws)[0] == fda.FD_OK
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _noalloc(fda, w, t):
    out = torch.full_like(t["q"], float("nan"))
    lse = torch.full(t["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    fda.fd_decode_attention_noalloc(t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"],
                                    t["seq_len"], w.kv_rows, w.num_q_heads, w.num_kv_heads,
                                    w.head_dim, w.page_size, float(w.softmax_scale),
                                    float(w.k_scale), float(w.v_scale), out, lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("case", range(4))
def test_noalloc_matches_oracle_and_workspace_entry_twice(case, orc):
    fda = lib()
    w = _cases()[case]
    t = fw.to_torch(w, "cuda")
    ws_out, ws_lse = _with_workspace(fda, w, t)
    ref_out, ref_lse = orc.decode_attention(w)
    for call in range(2):
        out, lse = _noalloc(fda, w, t)
        parity(w, out.astype(np.float64), lse.astype(np.float64), ref_out, ref_lse,
               label=f"{w.name} call {call}")
        # same kernels, same plan: identical bits, NaN nowhere
        assert np.array_equal(out, ws_out, equal_nan=False), f"call {call}: output bits differ"
        assert np.array_equal(lse, ws_lse), f"call {call}: lse bits differ"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    fda = lib()
    c = fda.load_library()
    # 128 query heads over 8 KV heads need about 20 MiB of partial states on
    # a 152-SM GPU, more than the 16 MiB array.
    need = fda.fd_workspace_bytes(4, 128, 8, 128)
    if need <= (16 << 20):
        pytest.skip("this GPU has too few SMs for the size to exceed the array")
    fake = ctypes.c_void_p(0x1000)
    st = c.fd_decode_attention_noalloc(fake, fake, fake, fake, None, 0, fake, 100, 4, 128, 8, 128,
                                       0, 0.1, 1.0, 1.0, 0, 2, fake, fake, None)
    assert st == fda.FD_ERR_WORKSPACE_TOO_SMALL
