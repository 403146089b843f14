"""Helpers for the GPU tests: run a workload through the C ABI, compare with
the oracle at the tolerances of the decode-attention parity bar."""
from __future__ import annotations

import numpy as np
import torch

import fd_workloads as fw

# Parity bar: fp16 output max-abs 4e-3 and relative L2 1e-3; bf16 output
# max-abs 1.6e-2 (its own rounding alone gives a relative L2 near 1.7e-3, so
# the relative-L2 gate applies to fp16 only); LSE |d| <= 1e-4 * max(|lse|, 1).
TOL = {"f16": dict(max_abs=4e-3, rel_l2=1e-3), "bf16": dict(max_abs=1.6e-2, rel_l2=None)}
LSE_REL = 1e-4


def lib():
    import flash_decoding_attention_gb300 as fda
    fda.load_library()
    return fda


def run(w: fw.Workload, kernel: int = 0, workspace=None, stream=None, check_errors=True):
    """Returns (out fp64 numpy, lse fp64 numpy, raw out tensor, raw lse tensor)."""
    fda = lib()
    fda.fd_set_kernel(kernel)
    try:
        t = fw.to_torch(w, "cuda")
        out = torch.full(t["q"].shape, float("nan"), dtype=t["q"].dtype, device="cuda")
        lse = torch.full(t["q"].shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
        if workspace is None:
            workspace = fda.alloc_workspace(w.batch, w.num_q_heads * w.q_len, w.num_kv_heads,
                                            w.head_dim)
        if w.q_len > 1:
            fda.fd_decode_attention_multi(
                t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"], t["seq_len"],
                w.kv_rows, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size,
                float(w.softmax_scale), float(w.k_scale), float(w.v_scale), w.scale_kind,
                t["k_scales"], t["v_scales"], out, lse, workspace, stream)
        elif w.scale_kind:
            fda.fd_decode_attention_scaled(
                t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"], t["seq_len"],
                w.kv_rows, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size,
                float(w.softmax_scale), float(w.k_scale), float(w.v_scale), w.scale_kind,
                t["k_scales"], t["v_scales"], out, lse, workspace, stream)
        else:
            fda.fd_decode_attention(t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"],
                                    t["seq_len"], w.kv_rows, w.num_q_heads, w.num_kv_heads,
                                    w.head_dim, w.page_size, float(w.softmax_scale),
                                    float(w.k_scale), float(w.v_scale), out, lse, workspace,
                                    stream)
        torch.cuda.synchronize()
        if check_errors:
            st, info = fda.fd_check_device_error(workspace, stream)
            assert st == fda.FD_OK, (fda.fd_status_string(st), info)
    finally:
        fda.fd_set_kernel(fda.FD_KERNEL_AUTO)
    return (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            out, lse)


def parity(w: fw.Workload, out, lse, ref_out, ref_lse, pairs=None, label=""):
    """Asserts the parity bar; returns the measured errors."""
    if pairs is not None:
        idx = tuple(np.asarray(pairs).T)
        out, lse, ref_out, ref_lse = out[idx], lse[idx], ref_out[idx], ref_lse[idx]
    assert np.all(np.isfinite(out)), f"{label}: non-finite output"
    d = out - ref_out
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    nrm = float(np.linalg.norm(ref_out))
    rel_l2 = float(np.linalg.norm(d) / nrm) if nrm > 0 else float(np.linalg.norm(d))
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse)), f"{label}: lse finiteness differs"
    assert np.all(lse[~fin] == ref_lse[~fin]), f"{label}: lse of empty sequences"
    lse_err = float((np.abs(lse[fin] - ref_lse[fin]) / np.maximum(np.abs(ref_lse[fin]), 1.0)).max()) \
        if fin.any() else 0.0
    tol = TOL[w.q_dtype]
    msg = f"{label}: max_abs={max_abs:.3e} rel_l2={rel_l2:.3e} lse_rel={lse_err:.3e}"
    print(msg)
    assert max_abs <= tol["max_abs"], msg
    if tol["rel_l2"] is not None:
        assert rel_l2 <= tol["rel_l2"], msg
    assert lse_err <= LSE_REL, msg
    return max_abs, rel_l2, lse_err
