"""The bounded waits of the tensor-core split kernel, made to run out.

Every wait of that kernel on its copy pipeline is bounded; when a bound
expires the kernel records a timeout in the workspace's error word, stops
issuing copies, lets the copies it issued land, and returns, so that the
context stays usable and the host learns of it from fd_check_device_error
(the asynchronous reporting of device errors described in "SGLang Prefill
optimisation: dissecting FlashAttention kernel bottlenecks with GPU Trace",
section 4.2).  Here the producer is told to issue no copy at all and the
bound is cut to a few milliseconds, so the consumers' first wait runs out
with nothing in flight; the next call, with the defaults back, must be
exact again.
"""
import numpy as np
import pytest

import fd_workloads as fw
from gpu_util import lib, parity, run

pytestmark = pytest.mark.gpu


def _cases():
    return [
        fw.make_contiguous("timeout-mqa", 41, [3000, 70000], 16, 1, 128, "f16", "e4m3"),
        fw.to_paged(fw.make_contiguous("timeout-gqa", 42, [1, 500, 9000], 64, 8, 128, "f16",
                                       "e4m3"), 64, 43),
        fw.make_contiguous("timeout-bf16", 44, [2048, 100], 32, 8, 128, "bf16", "bf16"),
    ]


@pytest.mark.parametrize("case", range(3))
def test_starved_pipeline_reports_timeout_then_recovers(case, orc):
    fda = lib()
    w = _cases()[case]
    ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    try:
        fda.fd_debug_set_wait_limit(3_000_000, True)      # 3 ms, no copy issued
        run(w, fda.FD_KERNEL_MMA, workspace=ws, check_errors=False)
        st, info = fda.fd_check_device_error(ws)
    finally:
        fda.fd_debug_set_wait_limit(0, False)
    assert st == fda.FD_ERR_DEVICE_TIMEOUT, fda.fd_status_string(st)
    assert info == 2                                     # a consumer's wait ran out
    # the word is cleared by the read, and the defaults are back
    assert fda.fd_check_device_error(ws)[0] == fda.FD_OK
    out, lse, _, _ = run(w, fda.FD_KERNEL_MMA, workspace=ws)
    ref_out, ref_lse = orc.decode_attention(w)
    parity(w, out, lse, ref_out, ref_lse, label=w.name)


@pytest.mark.parametrize("kernel,qh,kvh,q_len", [(3, 16, 1, 4), (3, 128, 2, 1), (4, 64, 8, 1)])
def test_starved_pipeline_other_split_kernels(kernel, qh, kvh, q_len, orc):
    """The same on the tcgen05 kernel (its converter, softmax and MMA-issue
    waits are bounded alike; whichever runs out first is recorded) and on
    the CUDA-core FMA form (its consumers' waits)."""
    fda = lib()
    w = fw.make_contiguous(f"timeout-k{kernel}-{qh}-{kvh}", 45 + kernel, [3000, 700, 9000], qh, kvh,
                           128, "f16", "e4m3", q_len=q_len)
    ws = fda.alloc_workspace(w.batch, w.num_q_heads * q_len, w.num_kv_heads, w.head_dim)
    try:
        fda.fd_debug_set_wait_limit(3_000_000, True)      # 3 ms, no copy issued
        run(w, kernel, workspace=ws, check_errors=False)
        st, info = fda.fd_check_device_error(ws)
    finally:
        fda.fd_debug_set_wait_limit(0, False)
    assert st == fda.FD_ERR_DEVICE_TIMEOUT, fda.fd_status_string(st)
    # tcgen05: a converter (6), the MMA thread (7) or a softmax warp (11); FMA form: a consumer
    assert info in ({6, 7, 11} if kernel == 3 else {2}), info
    assert fda.fd_check_device_error(ws)[0] == fda.FD_OK
    out, lse, _, _ = run(w, kernel, workspace=ws)
    ref_out, ref_lse = orc.decode_attention(w)
    parity(w, out, lse, ref_out, ref_lse, label=w.name)


def test_wait_limit_alone_changes_nothing(orc):
    """A shortened bound that no wait reaches leaves the result exact."""
    fda = lib()
    w = _cases()[0]
    ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim)
    try:
        fda.fd_debug_set_wait_limit(200_000_000, False)   # 200 ms
        out, lse, _, _ = run(w, fda.FD_KERNEL_MMA, workspace=ws)
    finally:
        fda.fd_debug_set_wait_limit(0, False)
    ref_out, ref_lse = orc.decode_attention(w)
    parity(w, out, lse, ref_out, ref_lse, label=w.name)


def test_wait_limit_arguments():
    fda = lib()
    c = fda.load_library()
    assert c.fd_debug_set_wait_limit(-1, 0) == fda.FD_ERR_INVALID_ARG
    assert c.fd_debug_set_wait_limit(20_000_000_000, 0) == fda.FD_ERR_INVALID_ARG
    assert c.fd_debug_set_wait_limit(0, 0) == fda.FD_OK
