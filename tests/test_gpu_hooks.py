"""GPU checks of the integer parts: the device split plan equals its Python
restatement bit for bit, the kernels' cache addressing gathers exactly the
bytes a CPU gather picks, and out-of-range rows or pages surface as a device
error status instead of a fault."""
import numpy as np
import pytest
import torch

import fd_workloads as fw
import plan_ref
from gpu_util import lib, run

pytestmark = pytest.mark.gpu


def _plan_cases():
    rng = np.random.default_rng(5)
    return [
        fw.tiny_mqa(),
        fw.make_contiguous("p1", 1, [0, 5, 0, 1000, 1], 16, 2, 128, "f16", "e4m3"),
        fw.make_contiguous("p2", 2, list(rng.integers(0, 5000, 40)), 32, 8, 128, "bf16", "bf16"),
        fw.make_contiguous("p3", 3, [40000, 3], 64, 8, 64, "f16", "e4m3"),
        fw.make_contiguous("p4", 4, [131072], 16, 1, 128, "f16", "e4m3"),
        # more streams than threads per CTA (the plan's multi-pass branch)
        fw.make_contiguous("p5", 6, list(rng.integers(0, 300, 700)), 8, 8, 64, "f16", "e4m3"),
        # 250 streams: one pass of the plan, most threads busy
        fw.make_contiguous("p6", 7, list(rng.integers(0, 900, 250)), 64, 8, 128, "f16", "e4m3"),
        # a paged pool (the plan reads seq_len only; the block table is not consulted)
        fw.to_paged(fw.make_contiguous("p7", 8, list(rng.integers(0, 3000, 24)), 32, 8, 128,
                                       "f16", "e4m3"), 16, 9),
        # query groups above 16 rows (the tcgen05 kernel's shapes)
        fw.make_contiguous("p8", 10, list(rng.integers(0, 9000, 12)), 64, 2, 128, "f16", "e4m3"),
        fw.to_paged(fw.make_contiguous("p9", 11, [0, 700, 40000, 5, 64], 128, 1, 128, "f16",
                                       "e4m3"), 16, 12),
    ]


def _takes(kernel, w):
    """Whether a forced kernel takes a plan case: the CUDA-core and mma.sync
    kernels take every case here; the tcgen05 kernel takes e4m3 caches with
    fp16 queries, head_dim 128 and 17..128 query rows per KV head."""
    rows = w.num_q_heads * w.q_len // w.num_kv_heads
    if kernel == 4:   # FMA form: e4m3, head_dim 128, <= 8 rows, 8 KV heads per stream
        return (w.kv_dtype == "e4m3" and w.head_dim == 128 and rows <= 8
                and w.num_kv_heads % 8 == 0 and (not w.paged or w.page_size >= 8))
    if kernel != 3:
        return True
    return (w.kv_dtype == "e4m3" and w.q_dtype == "f16" and w.head_dim == 128
            and 16 < rows <= 128 and (not w.paged or 8 <= w.page_size <= 256))


@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
@pytest.mark.parametrize("case", range(10))
def test_device_plan_matches_restatement(kernel, case):
    fda = lib()
    w = _plan_cases()[case]
    fda.fd_set_kernel(kernel)
    sel = fda.fd_selected_kernel(w.num_q_heads, w.num_kv_heads, w.head_dim,
                                 0 if w.q_dtype == "f16" else 1,
                                 fda.DTYPE_CODES[w.kv_dtype], w.paged, max(w.page_size, 1))
    fda.fd_set_kernel(0)
    if sel != kernel:
        # a forced kernel that does not take the shape refuses it outright
        assert sel == -1 and not _takes(kernel, w)
        return
    ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    run(w, kernel, workspace=ws)
    head, prefix = fda.fd_debug_read_plan(ws)
    S, hg, tile, grid, total, per_cta, k, seg_units = head
    assert k == kernel
    assert hg >= 1 and w.num_q_heads % hg == 0
    hq = w.num_q_heads // hg
    group = w.num_q_heads // w.num_kv_heads
    assert hq % group == 0 or group % hq == 0      # a stream never splits a KV head's reads
    assert S == w.batch * hg
    assert seg_units >= 0 and (kernel in (2, 3, 4) or seg_units == 0)
    # the host's choice of shape, restated
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    elem = 1 if w.kv_dtype in ("e4m3", "i8") else 2
    assert (hg, tile, grid, seg_units) == plan_ref.host_shape(
        kernel, w.num_q_heads, w.num_kv_heads, w.head_dim, elem, sms, w.q_len)
    p_prefix, p_total, p_per_cta, _ = plan_ref.plan(w.seq_len, hg, tile, grid, seg_units)
    assert prefix == p_prefix
    assert (total, per_cta) == (p_total, p_per_cta)


@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
@pytest.mark.parametrize("case", range(10))
def test_device_segments_match_restatement(kernel, case):
    """Every CTA's segments (stream, token range, complete, partial slot), as
    the split kernels' own plan and segment walk produce them on the device,
    equal the restatement's bit for bit."""
    fda = lib()
    w = _plan_cases()[case]
    fda.fd_set_kernel(kernel)
    try:
        qd = 0 if w.q_dtype == "f16" else 1
        kd = fda.DTYPE_CODES[w.kv_dtype]
        sel = fda.fd_selected_kernel(w.num_q_heads, w.num_kv_heads, w.head_dim, qd, kd, w.paged,
                                     max(w.page_size, 1))
        if sel != kernel:
            # a forced kernel that does not take the shape refuses it outright
            assert sel == -1 and not _takes(kernel, w)
            return
        ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
        seq = torch.from_numpy(w.seq_len).cuda()
        kvs = None if w.paged else torch.from_numpy(w.kv_start_idx).cuda()
        got = fda.fd_debug_plan_segments(seq, w.q_len, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                         w.paged, max(w.page_size, 1), qd, kd, ws,
                                         capacity_per_cta=1024, kv_start_idx=kvs)
        assert fda.fd_check_device_error(ws)[0] == fda.FD_OK
    finally:
        fda.fd_set_kernel(0)
    head, prefix = fda.fd_debug_read_plan(ws)
    S, hg, tile, grid, total, per_cta, k, seg_units = head
    assert k == kernel and len(got) == grid
    p_prefix, _, _, segs = plan_ref.plan(w.seq_len, hg, tile, grid, seg_units)
    assert prefix == p_prefix
    want = [[] for _ in range(grid)]
    for sg in segs:
        want[sg.cta].append((sg.stream, sg.t_begin, sg.t_end, int(sg.complete), sg.slot))
    assert got == want


def _cpu_gather(w, which):
    cache = w.k_cache if which == "k" else w.v_cache
    rows = cache.reshape(-1, w.num_kv_heads, w.head_dim)
    out = []
    for b in range(w.batch):
        t = np.arange(int(w.seq_len[b]))
        if w.paged:
            r = w.block_table[b, t // w.page_size].astype(np.int64) * w.page_size + t % w.page_size
        else:
            r = int(w.kv_start_idx[b]) + t
        out.append(rows[r])
    return np.concatenate(out) if out else rows[:0]


@pytest.mark.parametrize("paged,P", [(False, 0), (True, 1), (True, 16), (True, 64)])
def test_gather_is_byte_exact(paged, P):
    fda = lib()
    w = fw.make_contiguous("g", 21, [1, 17, 0, 300], 8, 2, 128, "f16", "e4m3", gap=4)
    if paged:
        w = fw.to_paged(w, P, 22)
    t = fw.to_torch(w, "cuda")
    total = int(w.seq_len.sum())
    for which in ("k", "v"):
        dst = torch.full((total, w.num_kv_heads, w.head_dim), 0xAB, dtype=torch.uint8,
                         device="cuda")
        ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        fda.fd_debug_gather_kv(t[which], t["kv_start_idx"], t["block_table"], t["seq_len"],
                               w.kv_rows, w.num_kv_heads, w.head_dim, max(P, 1), dst, ws)
        torch.cuda.synchronize()
        assert np.array_equal(dst.cpu().numpy(), _cpu_gather(w, which))
        assert fda.fd_check_device_error(ws)[0] == fda.FD_OK


def test_bad_page_id_is_reported_not_faulted():
    fda = lib()
    base = fw.make_contiguous("bad", 23, [100, 200], 16, 2, 128, "f16", "e4m3")
    w = fw.to_paged(base, 16, 24)
    bt = w.block_table.copy()
    pool_pages = w.k_cache.shape[0]
    bt[1, 3] = pool_pages + 5          # beyond the pool
    w.block_table = bt
    for k in (0, 1):
        ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
        out, lse, _, _ = run(w, k, workspace=ws, check_errors=False)
        st, info = fda.fd_check_device_error(ws)
        assert st == fda.FD_ERR_DEVICE_BOUNDS and info == pool_pages + 5, (k, st, info)
        # the word is cleared by the read
        assert fda.fd_check_device_error(ws)[0] == fda.FD_OK
        # sequence 0 does not touch the bad page and stays exact
        assert np.all(np.isfinite(out[0]))


def test_contiguous_row_overrun_is_reported():
    fda = lib()
    w = fw.make_contiguous("over", 25, [50, 60], 8, 2, 128, "f16", "f16")
    w.kv_start_idx = np.array([0, w.k_cache.shape[0] - 10], np.int32)   # runs 50 rows past the end
    ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    run(w, 0, workspace=ws, check_errors=False)
    st, _ = fda.fd_check_device_error(ws)
    assert st == fda.FD_ERR_DEVICE_BOUNDS


def test_workspace_too_small_is_rejected():
    fda = lib()
    w = fw.tiny_mqa()
    t = fw.to_torch(w, "cuda")
    need = fda.fd_workspace_bytes(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    assert need > 256
    ws = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device="cuda")
    st = fda.fd_decode_attention(t["q"], t["k"], t["v"], t["kv_start_idx"], None, t["seq_len"],
                                 w.kv_rows, 4, 1, 64, 0, 0.125, 1.0, 1.0, out, lse, ws,
                                 check=False)
    assert st == fda.FD_ERR_WORKSPACE_TOO_SMALL
