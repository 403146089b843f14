"""Concurrent calls from several host threads.

Each thread drives its own stream, workspace and workload (different shapes,
so different TMA descriptors and kernel variants), repeatedly and at the same
time as the others: the library's host-side caches (descriptors, per-device
SM count and shared-memory limits) are shared by the threads, and every
thread's last result must still match the oracle.  ctypes releases the
interpreter lock around each foreign call, so the calls overlap on the host.
"""
import threading

import numpy as np
import pytest
import torch

import fd_workloads as fw
import oracle
from gpu_util import lib, parity

pytestmark = pytest.mark.gpu

REPS = 25


def _workloads():
    return [
        fw.to_paged(fw.make_contiguous("thr-paged-fp8", 1300, [700, 2000, 65, 0, 900], 64, 8, 128,
                                       "f16", "e4m3"), 64, 1301),
        fw.make_contiguous("thr-contig-bf16", 1310, [1000, 31, 2500], 32, 8, 128, "bf16", "bf16",
                           gap=2),
        fw.make_contiguous("thr-mqa-fp8", 1320, [6000, 129], 16, 1, 128, "f16", "e4m3"),
        fw.to_paged(fw.make_contiguous("thr-paged16-d64", 1330, [300, 1, 1200, 77], 16, 4, 64,
                                       "f16", "f16"), 16, 1331),
    ]


def test_threads_share_the_library():
    fda = lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    jobs = []
    for w in _workloads():
        t = fw.to_torch(w, dev)
        out = torch.full(t["q"].shape, float("nan"), dtype=t["q"].dtype, device=dev)
        lse = torch.full(t["q"].shape[:-1], float("nan"), dtype=torch.float32, device=dev)
        ws = fda.alloc_workspace(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, dev)
        jobs.append((w, t, out, lse, ws, torch.cuda.Stream(device=dev)))
    torch.cuda.synchronize(dev)
    errors = []
    start = threading.Barrier(len(jobs))

    def work(w, t, out, lse, ws, stream):
        try:
            torch.cuda.set_device(dev.index)
            start.wait(timeout=120)
            for _ in range(REPS):
                fda.fd_decode_attention(t["q"], t["k"], t["v"], t["kv_start_idx"],
                                        t["block_table"], t["seq_len"], w.kv_rows, w.num_q_heads,
                                        w.num_kv_heads, w.head_dim, w.page_size,
                                        float(w.softmax_scale), float(w.k_scale),
                                        float(w.v_scale), out, lse, ws, stream)
            stream.synchronize()
        except Exception as e:   # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=job) for job in jobs]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize(dev)
    for w, t, out, lse, ws, stream in jobs:
        st, info = fda.fd_check_device_error(ws, stream)
        assert st == fda.FD_OK, (w.name, fda.fd_status_string(st), info)
        ref_out, ref_lse = oracle.decode_attention(w)
        parity(w, out.float().cpu().numpy().astype(np.float64),
               lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, label=w.name)
