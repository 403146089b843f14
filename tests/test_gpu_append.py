"""GPU tests of the KV append (fd_append_kv) and of the decode step with its
append (fd_decode_attention_append), against the oracle's append and
attention.  Appended 8-bit codes and per-token scales must equal the
oracle's bit for bit (both take them from the same fp32 operations); a
negative zero and a positive zero e4m3 code count as the same code."""
import dataclasses

import numpy as np
import pytest
import torch

import fd_workloads as fw
import oracle
from gpu_util import lib, parity

pytestmark = pytest.mark.gpu


def _codes(a, kv_dtype):
    a = np.ascontiguousarray(a)
    if kv_dtype == "e4m3":
        c = a.view(np.uint8).copy()
        c[c == 0x80] = 0
        return c
    return a.view(np.uint8) if kv_dtype == "i8" else a.view(np.uint16)


def _expected(w, k_new, v_new, pos):
    kc, vc, ks, vs = oracle.append_kv(w, k_new, v_new, pos)
    upd = dataclasses.replace(w, k_cache=kc, v_cache=vc)
    if w.scale_kind == fw.SCALE_TOKEN:
        upd = dataclasses.replace(upd, k_scales=ks, v_scales=vs)
    return upd


def _device_inputs(w, k_new, v_new, pos):
    t = fw.to_torch(w, "cuda")
    qd, _ = fw.torch_dtypes(w)
    t["k_new"] = torch.from_numpy(k_new.view(np.int16)).view(qd).cuda()
    t["v_new"] = torch.from_numpy(v_new.view(np.int16)).view(qd).cuda()
    t["positions"] = torch.from_numpy(np.ascontiguousarray(pos, np.int32)).cuda()
    return t


def _check_caches(w, exp, t):
    torch.cuda.synchronize()
    for name, ref in (("k", exp.k_cache), ("v", exp.v_cache)):
        got = t[name].cpu()
        got = (got.view(torch.int16) if got.element_size() == 2 else got).numpy()
        assert np.array_equal(_codes(got, w.kv_dtype), _codes(ref, w.kv_dtype)), \
            f"{w.name}: {name} cache differs from the oracle's append"
    if w.scale_kind == fw.SCALE_TOKEN:
        for name, ref in (("k_scales", exp.k_scales), ("v_scales", exp.v_scales)):
            got = t[name].cpu().numpy()
            assert np.array_equal(got.view(np.uint32), np.asarray(ref, np.float32).view(np.uint32)), \
                f"{w.name}: {name} differ from the oracle's"


def _cases():
    out = []
    base8 = fw.make_contiguous("app-e4m3", 70, [1, 40, 0, 129, 300, 5], 16, 2, 128, "f16", "e4m3",
                               gap=2, lead=1)
    out.append(base8)
    out.append(fw.with_scales(base8, fw.SCALE_HEAD, 71))
    out.append(fw.with_scales(fw.to_paged(base8, 16, 72), fw.SCALE_TOKEN, 73))
    # bf16 outputs: scales from U(0.25, 1) keep the outputs at the size the
    # bf16 max-abs bar assumes (its rounding grows with the value)
    i8 = fw.make_contiguous("app-i8", 74, [3, 64, 65, 0, 700], 32, 4, 64, "bf16", "i8", gap=1)
    out.append(fw.to_paged(i8, 64, 75))
    out.append(fw.with_scales(i8, fw.SCALE_TOKEN, 76, span=(0.25, 1.0)))
    out.append(fw.with_scales(fw.to_paged(i8, 8, 77), fw.SCALE_HEAD, 78, span=(0.25, 1.0)))
    out.append(fw.make_contiguous("app-f16", 79, [2, 33, 0, 90], 8, 8, 128, "f16", "f16", gap=1))
    out.append(fw.to_paged(fw.make_contiguous("app-bf16", 80, [17, 1, 256], 16, 1, 64, "bf16",
                                              "bf16"), 32, 81))
    return out


CASES = _cases()


@pytest.mark.parametrize("i", range(len(CASES)), ids=[c.name for c in CASES])
def test_append_matches_oracle(i):
    fda = lib()
    w = CASES[i]
    k_new, v_new = fw.new_tokens(w, 200 + i, std=2.0)
    pos = fw.last_positions(w)
    pos[1] = -1                                       # one sequence gets no append
    exp = _expected(w, k_new, v_new, pos)
    t = _device_inputs(w, k_new, v_new, pos)
    ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    fda.fd_append_kv(t["k_new"], t["v_new"], t["k"], t["v"], t["kv_start_idx"], t["block_table"],
                     t["positions"], w.kv_rows, w.num_kv_heads, w.head_dim, w.page_size,
                     float(w.k_scale), float(w.v_scale), w.scale_kind, t["k_scales"],
                     t["v_scales"], ws)
    _check_caches(w, exp, t)
    st, info = fda.fd_check_device_error(ws)
    assert st == fda.FD_OK, (fda.fd_status_string(st), info)


def _fused(w, seed, kernel=0):
    """fd_decode_attention_append on device copies (w.q_len new tokens per
    sequence); returns (exp, t, out, lse)."""
    fda = lib()
    k_new, v_new = fw.new_tokens(w, seed, std=2.0, n_new=w.q_len)
    pos = fw.last_positions(w, w.q_len)
    exp = _expected(w, k_new, v_new, pos)
    t = _device_inputs(w, k_new, v_new, pos)
    out = torch.full(t["q"].shape, float("nan"), dtype=t["q"].dtype, device="cuda")
    lse = torch.full(t["q"].shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    ws = fda.alloc_workspace(w.batch, w.num_q_heads * w.q_len, w.num_kv_heads, w.head_dim)
    fda.fd_set_kernel(kernel)
    try:
        fda.fd_decode_attention_append(
            t["q"], t["k_new"], t["v_new"], t["k"], t["v"], t["kv_start_idx"], t["block_table"],
            t["positions"], t["seq_len"], w.kv_rows, w.num_q_heads, w.num_kv_heads, w.head_dim,
            w.page_size, float(w.softmax_scale), float(w.k_scale), float(w.v_scale),
            w.scale_kind, t["k_scales"], t["v_scales"], out, lse, ws)
        torch.cuda.synchronize()
    finally:
        fda.fd_set_kernel(0)
    st, info = fda.fd_check_device_error(ws)
    assert st == fda.FD_OK, (fda.fd_status_string(st), info)
    return exp, t, out, lse


@pytest.mark.parametrize("kernel", [1, 2], ids=["simt", "mma"])
@pytest.mark.parametrize("i", range(len(CASES)), ids=[c.name for c in CASES])
def test_decode_with_append_matches_oracle(i, kernel):
    """The step's new token is written and attended to in one call: caches as
    the oracle's append, outputs as the oracle's attention over them."""
    w = CASES[i]
    fda = lib()
    fda.fd_set_kernel(kernel)
    sel = fda.fd_selected_kernel(w.num_q_heads, w.num_kv_heads, w.head_dim,
                                 0 if w.q_dtype == "f16" else 1, fda.DTYPE_CODES[w.kv_dtype],
                                 w.paged, max(w.page_size, 1))
    fda.fd_set_kernel(0)
    if sel != kernel:
        pytest.skip("kernel does not support this shape")
    exp, t, out, lse = _fused(w, 300 + i, kernel)
    _check_caches(w, exp, t)
    ref_out, ref_lse = oracle.decode_attention(exp)
    parity(exp, out.float().cpu().numpy().astype(np.float64),
           lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, label=f"{w.name} append")


@pytest.mark.parametrize("n,kind", [(4, fw.SCALE_TENSOR), (5, fw.SCALE_TENSOR),
                                    (4, fw.SCALE_TOKEN)])
def test_config_full_size_with_append(n, kind):
    """The decode workloads' last token written by the step itself."""
    w = fw.WORKLOADS[n]()
    if kind:
        w = fw.with_scales(w, kind, 84 + n)
    exp, t, out, lse = _fused(w, 400 + n)
    _check_caches(w, exp, t)
    ref_out, ref_lse = oracle.decode_attention(exp)
    parity(exp, out.float().cpu().numpy().astype(np.float64),
           lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, label=f"config{n} append")


def test_append_out_of_range_is_reported_and_not_written():
    """A position whose page is not in the block table (entry -1) is recorded
    as a device bounds error and writes nothing; other sequences append."""
    fda = lib()
    base = fw.make_contiguous("app-oob", 85, [16, 40], 8, 2, 128, "f16", "e4m3")
    w = fw.to_paged(base, 16, 86)
    k_new, v_new = fw.new_tokens(w, 87)
    pos = np.array([16, 39], np.int32)      # sequence 0 has one page: page 1 is -1
    assert w.block_table[0, 1] == -1
    exp = _expected(w, k_new, v_new, np.array([-1, 39], np.int32))
    t = _device_inputs(w, k_new, v_new, pos)
    ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    fda.fd_append_kv(t["k_new"], t["v_new"], t["k"], t["v"], None, t["block_table"],
                     t["positions"], w.kv_rows, w.num_kv_heads, w.head_dim, w.page_size,
                     float(w.k_scale), float(w.v_scale), 0, None, None, ws)
    _check_caches(w, exp, t)
    st, info = fda.fd_check_device_error(ws)
    assert st == fda.FD_ERR_DEVICE_BOUNDS, (fda.fd_status_string(st), info)


@pytest.mark.parametrize("q_len", [2, 4])
@pytest.mark.parametrize("i", [0, 2, 5, 6], ids=[CASES[i].name for i in (0, 2, 5, 6)])
def test_verify_step_with_append(i, q_len):
    """A speculative verify step in one call: its q_len drafted tokens are
    appended (token j at position seq_len - q_len + j) and attended to
    causally; caches as the oracle's append, outputs as its attention."""
    w = fw.with_q_len(CASES[i], q_len, 600 + i)
    exp, t, out, lse = _fused(w, 610 + i)
    _check_caches(w, exp, t)
    ref_out, ref_lse = oracle.decode_attention(exp)
    parity(exp, out.float().cpu().numpy().astype(np.float64),
           lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, label=f"{w.name} verify")


@pytest.mark.parametrize("n,q_len", [(4, 2), (5, 4)])
def test_config_full_size_verify_with_append(n, q_len):
    w = fw.with_q_len(fw.WORKLOADS[n](), q_len, 620 + n)
    exp, t, out, lse = _fused(w, 630 + n)
    _check_caches(w, exp, t)
    ref_out, ref_lse = oracle.decode_attention(exp)
    parity(exp, out.float().cpu().numpy().astype(np.float64),
           lse.cpu().numpy().astype(np.float64), ref_out, ref_lse,
           label=f"config{n}-q{q_len} verify")
