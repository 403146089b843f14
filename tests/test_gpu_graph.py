"""A decode step captured in a CUDA graph and replayed.

Serving loops capture the decode step once and replay it every step with new
query vectors and new sequence lengths written in place.  The library reads
seq_len on the device (no host-side copy of it, no host sync), so a replay
must equal a fresh call on the rewritten inputs: each replay here is checked
against the oracle on those inputs, on the split kernel chosen by the library
and with its combine launched as a programmatic dependent inside the graph.
"""
import dataclasses

import numpy as np
import pytest
import torch

import fd_workloads as fw
import oracle
from gpu_util import lib, parity

pytestmark = pytest.mark.gpu


def _paged_gqa():
    base = fw.make_contiguous("graph-paged-fp8", 1200, [700, 3000, 65, 0, 1500, 129], 64, 8, 128,
                              "f16", "e4m3")
    return fw.to_paged(base, 64, 1201)


def _contiguous_bf16():
    return fw.make_contiguous("graph-contiguous-bf16", 1210, [1000, 31, 2500, 400], 32, 8, 128,
                              "bf16", "bf16", gap=2)


def _mqa_four_tokens():
    # 64 query rows for one KV head: the tcgen05 kernel when the library chooses
    return fw.make_contiguous("graph-mqa-4tok", 1220, [5000, 900, 3], 16, 1, 128, "f16", "e4m3",
                              q_len=4)


CASES = {"paged-fp8-gqa": _paged_gqa, "contiguous-bf16": _contiguous_bf16,
         "mqa-fp8-4-tokens": _mqa_four_tokens}


@pytest.mark.parametrize("name", list(CASES))
def test_replay_with_new_inputs(name):
    fda = lib()
    w = CASES[name]()
    dev = torch.device("cuda")
    t = fw.to_torch(w, dev)
    out = torch.full(t["q"].shape, float("nan"), dtype=t["q"].dtype, device=dev)
    lse = torch.full(t["q"].shape[:-1], float("nan"), dtype=torch.float32, device=dev)
    ws = fda.alloc_workspace(w.batch, w.num_q_heads * w.q_len, w.num_kv_heads, w.head_dim, dev)

    def step(stream):
        if w.q_len > 1:
            fda.fd_decode_attention_multi(
                t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"], t["seq_len"],
                w.kv_rows, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size,
                float(w.softmax_scale), float(w.k_scale), float(w.v_scale), w.scale_kind,
                t["k_scales"], t["v_scales"], out, lse, ws, stream)
        else:
            fda.fd_decode_attention(t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"],
                                    t["seq_len"], w.kv_rows, w.num_q_heads, w.num_kv_heads,
                                    w.head_dim, w.page_size, float(w.softmax_scale),
                                    float(w.k_scale), float(w.v_scale), out, lse, ws, stream)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step(side)   # eager first: one-time host setup happens outside the capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(side)

    rng = np.random.default_rng(1230)
    q_bits = w.q
    for it in range(3):
        if it == 0:
            new_q, new_len = w.q, w.seq_len
        else:
            # other query vectors (the same values, moved to other heads), and
            # every sequence cut to a random length no longer than it was
            new_q = np.ascontiguousarray(np.roll(q_bits, it, axis=1))
            new_len = np.array([rng.integers(0, n + 1) for n in w.seq_len], dtype=np.int32)
        t["q"].copy_(torch.from_numpy(new_q.view(np.int16)).view(t["q"].dtype).to(dev))
        t["seq_len"].copy_(torch.from_numpy(new_len).to(dev))
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize(dev)
        graph.replay()
        torch.cuda.synchronize(dev)
        st, info = fda.fd_check_device_error(ws)
        assert st == fda.FD_OK, (fda.fd_status_string(st), info)
        wi = dataclasses.replace(w, q=new_q, seq_len=new_len)
        ref_out, ref_lse = oracle.decode_attention(wi)
        parity(wi, out.float().cpu().numpy().astype(np.float64),
               lse.cpu().numpy().astype(np.float64), ref_out, ref_lse,
               label=f"{name} replay {it} seq_len {[int(x) for x in new_len]}")
