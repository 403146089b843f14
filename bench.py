"""Decode-step benchmark: effective HBM GB/s and microseconds per decode step.

One step = one fd_decode_attention call (split kernel + combine kernel) over
one batch of synthetic, seeded inputs already resident in HBM.  Default
workload: FP8 paged decode (B=64, lognormal lengths with median 2048 clipped
to [16, 16384], 64 query / 8 KV heads, D=128, page 64, e4m3 K/V with
per-tensor scales, fp16 Q/out).  `--config N` picks another of the five
decode workloads.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on the host cores instead (the reference arm of this build).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import fd_workloads as fw  # noqa: E402

METRIC = "decode-attention effective HBM GB/s (% of GB300 peak) and \u00b5s per decode step"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "mma", "tc", "fma"])
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--scales", default="tensor", choices=["tensor", "head", "token"],
                    help="8-bit workloads: finer K/V scales per KV head or per token")
    ap.add_argument("--kv", default="e4m3", choices=["e4m3", "i8"],
                    help="8-bit K/V format of the FP8 workloads (configs 3-5): e4m3, or the same "
                         "draws quantised to INT8 (symmetric, amax/127)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence (a speculative-decoding verify step: the "
                         "last q_len cached tokens, causal among themselves)")
    ap.add_argument("--append", action="store_true",
                    help="the step also writes each sequence's last token (with --q-len, its "
                         "last q_len tokens: K/V rows, quantised for 8-bit caches) before "
                         "attending, in one call")
    ap.add_argument("--shared-prefix", type=int, default=0,
                    help="paged workloads: every sequence's first pages alias those of "
                         "sequence 0 up to this many tokens (prefix-cache hits)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config timings of the other workloads and variants")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def device_env(dev) -> dict:
    """GPU name, SM count, L2 size, CUDA runtime and driver versions."""
    import torch
    prop = torch.cuda.get_device_properties(dev)
    env = {"gpu": prop.name, "sms": prop.multi_processor_count,
           "l2_bytes": prop.L2_cache_size, "cuda_runtime": torch.version.cuda,
           "torch": torch.__version__}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                              "-i", str(dev.index or 0)], capture_output=True, text=True, timeout=20)
        env["driver"] = out.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        env["driver"] = None
    return env


def max_over_ranks(value: float, device) -> float:
    """Largest value over the ranks of the default process group (the
    slowest replica sets the whole job's time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units processed by all replicas (each does the same work) per second
    of the slowest one."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on the host cores
# ---------------------------------------------------------------------------

def oracle_sample(w: fw.Workload, budget_s: float, nthreads: int = 0, start: int = 0):
    """Times the oracle on the workload's (sequence, KV head) units -- the
    query heads of one KV head of one sequence; with a budget of a second or
    more, whole sequences per call -- taken in order from unit `start`
    (wrapping) until about `budget_s` seconds of wall time; returns (GB/s by
    the algorithmic-bytes formula, threads used, description, seconds)."""
    import oracle
    orc = oracle.default()
    g = w.num_q_heads // w.num_kv_heads
    per_call = w.num_kv_heads if budget_s >= 1.0 else 1     # KV heads per oracle call
    calls_per_seq = w.num_kv_heads // per_call
    n_calls = w.batch * calls_per_seq
    done_bytes = 0
    elapsed = 0.0
    threads = 0
    calls = 0
    for c in range(n_calls):
        u = (start + c) % n_calls
        b, h0 = u // calls_per_seq, (u % calls_per_seq) * per_call
        T = int(w.seq_len[b])
        pairs = [(b, h) for h in range(h0 * g, (h0 + per_call) * g)]
        t0 = time.perf_counter()
        _, _, _, threads = orc.decode_attention_raw(
            w.q, w.q_dtype, w.k_cache, w.v_cache, w.kv_dtype, w.seq_len, w.num_q_heads,
            w.num_kv_heads, w.head_dim, w.softmax_scale, w.k_scale, w.v_scale,
            kv_start_idx=w.kv_start_idx, block_table=w.block_table, page_size=w.page_size,
            kv_rows=w.kv_rows, pairs=pairs, scale_kind=w.scale_kind, k_scales=w.k_scales,
            v_scales=w.v_scales, q_len=w.q_len, nthreads=nthreads)
        elapsed += time.perf_counter() - t0
        done_bytes += per_call * (T * w.head_dim * w.kv_elem_bytes * 2
                                  + 2 * g * w.q_len * w.head_dim * 2)
        if h0 == 0:   # index bytes, once per sequence
            done_bytes += (4 + 4 * (-(-T // w.page_size))) if w.paged else 8
        calls += 1
        if elapsed >= budget_s:
            break
    gbs = done_bytes / elapsed / 1e9 if elapsed > 0 else 0.0
    what = "sequences (all query heads)" if per_call == w.num_kv_heads else \
        f"(sequence, KV head) units ({g} query heads each)"
    desc = (f"{calls} of {n_calls} {what} from unit {start % n_calls}, "
            f"{done_bytes / 1e6:.1f} MB algorithmic, {elapsed:.2f} s")
    return gbs, threads, desc, elapsed


def make_workload(args) -> fw.Workload:
    if args.kv != "e4m3":
        if args.config < 3:
            raise SystemExit("--kv needs an 8-bit workload (configs 3-5)")
        w = fw.WORKLOADS[args.config](kv_dtype=args.kv)
    else:
        w = fw.WORKLOADS[args.config]()
    if args.q_len > 1:
        w = fw.with_q_len(w, args.q_len, 540 + args.config)
    if args.shared_prefix:
        if not w.paged:
            raise SystemExit("--shared-prefix needs a paged workload")
        w = fw.share_prefix(w, args.shared_prefix)
    if args.scales != "tensor":
        if w.kv_dtype not in ("e4m3", "i8"):
            raise SystemExit("--scales needs an 8-bit workload")
        kind = fw.SCALE_HEAD if args.scales == "head" else fw.SCALE_TOKEN
        w = fw.with_scales(w, kind, 90 + args.config)
    return w


def workload_config(args) -> dict:
    c = {"workload": fw.WORKLOAD_NAMES[args.config]}
    if args.shared_prefix:
        c["shared_prefix_tokens"] = args.shared_prefix
    if args.kv != "e4m3":
        c["kv_dtype"] = f"{args.kv} (the workload's draws quantised to INT8, per-tensor amax/127)"
    if args.q_len > 1:
        c["q_len"] = args.q_len
    if args.append:
        c["append"] = ("each step first writes every sequence's last q_len tokens (K/V rows of "
                       "the projection dtype, quantised for 8-bit caches) into the cache, then "
                       "attends over them: fd_decode_attention_append")
    if args.scales != "tensor":
        c["kv_scales"] = f"per {args.scales} (fp32, on top of the per-tensor scales)"
    return c


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = make_workload(args)
    per_step = []
    gbs_all = []
    threads = 0
    desc = ""
    # each step samples the oracle for a bounded time, so that the whole
    # --steps / --warmup run stays within about two minutes
    budget = min(2.0, max(0.02, 120.0 / max(1, args.warmup + args.steps)))
    for i in range(args.warmup + args.steps):
        if args.append:
            # the oracle's append of the whole batch, then the attention sample
            import dataclasses
            import oracle
            k_new, v_new = fw.new_tokens(w, 500 + args.config, n_new=w.q_len)
            t0 = time.perf_counter()
            kc, vc, ks, vs = oracle.default().append_kv(w, k_new, v_new,
                                                        fw.last_positions(w, w.q_len))
            t_app = time.perf_counter() - t0
            wa = dataclasses.replace(w, k_cache=kc, v_cache=vc)
            if w.scale_kind == fw.SCALE_TOKEN:
                wa = dataclasses.replace(wa, k_scales=ks, v_scales=vs)
            gbs, threads, desc, el = oracle_sample(wa, budget_s=budget, start=i)
            el_all = el + t_app
            gbs = (gbs * el + fw.append_bytes(w, w.q_len) / 1e9) / el_all
            el = el_all
            desc += f"; plus the append of all {w.batch} new tokens ({t_app:.3f} s)"
        else:
            gbs, threads, desc, el = oracle_sample(w, budget_s=budget, start=i)
        if i >= args.warmup:
            per_step.append(el)
            gbs_all.append(gbs)
    value = statistics.median(gbs_all)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(per_step), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(args),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": "per step: " + desc},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled: bool):
        self.proc = None
        self.path = None
        self.index = index
        if not enabled:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        # nvidia-smi's start-up (NVML initialisation) can stall the GPU for a
        # while: wait for its first two samples before anything is timed
        t_end = time.time() + 10.0
        while time.time() < t_end and self.proc.poll() is None:
            try:
                with open(self.path) as f:
                    if sum(1 for _ in f) >= 2:
                        break
            except OSError:
                pass
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ln in open(self.path):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# sources that make up each split kernel (its traffic changes only with them)
# arithmetic of each split kernel, for the dtype label
TENSOR_LABEL = {"mma": "mma", "tc": "tcgen05"}

KERNEL_SOURCES = {"fma": ("fd_common.cuh", "fd_split_mma.cuh", "fd_split_fma.cu"),
                  "tc": ("fd_common.cuh", "fd_split_mma.cuh", "fd_split_tc.cu"),
                  "mma": ("fd_common.cuh", "fd_split_mma.cuh", "fd_split_mma.cu",
                          "fd_split_mma_e4m3.cu", "fd_split_mma_i8.cu",
                          "fd_split_mma_16bit.cu"),
                  "simt": ("fd_common.cuh", "fd_split_simt.cu")}


def source_digest(kernel_name: str = "mma") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "flash_decoding_attention_gb300", "csrc")
    for f in KERNEL_SOURCES.get(kernel_name, ()):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except (ValueError, OSError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(kernel_name: str, config: int):
    """DRAM bytes per launch of the split kernel from the committed ncu
    summary, if it was taken on the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except ValueError:
        return None
    e = d.get(f"{kernel_name}/config{config}")
    if not e or e.get("source_digest") != source_digest(kernel_name):
        return None
    return e.get("dram_bytes_per_launch")


SYNC_EVERY = 64   # timed steps between host waits (keeps the launch queue short)


def timed_steps(step, flush, stream, K, split_events: bool = False):
    """Times K steps, each after an L2 flush (outside the events), with CUDA
    events on the launching stream: around the whole step, or (split_events)
    around the split kernel's launch inside it.  The host waits for the GPU
    every SYNC_EVERY steps, between two timed steps, so the launch queue
    never fills (a host thread blocked on a full queue can wake up late and
    leave the GPU idle inside a timed step).  Returns milliseconds per step."""
    import torch
    import flash_decoding_attention_gb300 as fda
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    if split_events:
        for a, b in ev:           # torch creates the CUDA events on first record
            a.record(stream)
            b.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        flush()
        if split_events:
            fda.fd_set_split_events(*ev[i])
            step()
            fda.fd_set_split_events(None, None)
        else:
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        if (i + 1) % SYNC_EVERY == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def make_step(fda, w, t, out, lse, ws, stream, append: bool = False):
    """One decode step of workload w through the C ABI (the entry point its
    options call for)."""
    QH, KVH, D = w.num_q_heads, w.num_kv_heads, w.head_dim

    def step():
        if w.q_len > 1 and not append:
            fda.fd_decode_attention_multi(
                t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"], t["seq_len"],
                w.kv_rows, QH, KVH, D, w.page_size, float(w.softmax_scale), float(w.k_scale),
                float(w.v_scale), w.scale_kind, t["k_scales"], t["v_scales"], out, lse, ws, stream)
            return
        if append:
            fda.fd_decode_attention_append(
                t["q"], t["k_new"], t["v_new"], t["k"], t["v"], t["kv_start_idx"],
                t["block_table"], t["positions"], t["seq_len"], w.kv_rows, QH, KVH, D,
                w.page_size, float(w.softmax_scale), float(w.k_scale), float(w.v_scale),
                w.scale_kind, t["k_scales"], t["v_scales"], out, lse, ws, stream)
            return
        if w.scale_kind:
            fda.fd_decode_attention_scaled(
                t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"], t["seq_len"],
                w.kv_rows, QH, KVH, D, w.page_size, float(w.softmax_scale), float(w.k_scale),
                float(w.v_scale), w.scale_kind, t["k_scales"], t["v_scales"], out, lse, ws, stream)
            return
        fda.fd_decode_attention(t["q"], t["k"], t["v"], t["kv_start_idx"], t["block_table"],
                                t["seq_len"], w.kv_rows, QH, KVH, D, w.page_size,
                                float(w.softmax_scale), float(w.k_scale), float(w.v_scale), out,
                                lse, ws, stream)
    return step


def pct(xs, q):
    return round(float(np.percentile(xs, q)) * 1e3, 2)


# Workloads timed next to the headline one (same protocol): the other
# configurations, and the per-token-scale, INT8 and verify-step variants of
# the headline workloads.  name -> (config, kv format, scale kind, q_len)
# name: (workload, KV dtype, scale kind, query tokens, split kernel: 0 = the
# library's own choice, else an fd_kernel value timed for comparison)
PER_CONFIG = {
    "config1": (1, "e4m3", "tensor", 1, 0), "config2": (2, "e4m3", "tensor", 1, 0),
    "config3": (3, "e4m3", "tensor", 1, 0), "config4": (4, "e4m3", "tensor", 1, 0),
    "config5": (5, "e4m3", "tensor", 1, 0),
    "config4_token_scales": (4, "e4m3", "token", 1, 0), "config4_int8": (4, "i8", "tensor", 1, 0),
    "config5_q_len4": (5, "e4m3", "tensor", 4, 0),
    # the same steps on other split kernels: mma.sync for the 4-token MQA step
    # (the library takes tcgen05 there), CUDA-core FMAs for the FP8 paged one
    "config5_q_len4_mma_sync": (5, "e4m3", "tensor", 4, 2),
    "config4_cuda_core_fma": (4, "e4m3", "tensor", 1, 4),
}
KERNEL_IDS = {1: "simt", 2: "mma", 3: "tc", 4: "fma"}


def per_config_timings(args, dev, stream, flush, peak, kernel_name):
    """µs per step (mean, p10/p50/p90), effective GB/s and its fraction of the
    peak, and the split kernel's own µs, for every PER_CONFIG entry except
    the headline's own."""
    import torch
    import flash_decoding_attention_gb300 as fda
    K = max(100, min(args.steps, 400))
    res = {}
    for name, (cfg, kv, scales, q_len, kern) in PER_CONFIG.items():
        if (cfg, kv, scales, q_len, kern) == (args.config, args.kv, args.scales, args.q_len, 0):
            continue
        a = argparse.Namespace(**vars(args))
        a.config, a.kv, a.scales, a.q_len, a.shared_prefix = cfg, kv, scales, q_len, 0
        w = make_workload(a)
        t = fw.to_torch(w, dev)
        out = torch.empty_like(t["q"])
        lse = torch.empty(t["q"].shape[:-1], dtype=torch.float32, device=dev)
        ws = fda.alloc_workspace(w.batch, w.num_q_heads * w.q_len, w.num_kv_heads, w.head_dim,
                                 dev)
        step = make_step(fda, w, t, out, lse, ws, stream)
        fda.fd_set_kernel(kern if kern else {"auto": 0, "simt": 1, "mma": 2, "tc": 3,
                                             "fma": 4}[args.kernel])
        sel = fda.fd_selected_kernel(w.num_q_heads * w.q_len, w.num_kv_heads, w.head_dim,
                                     0 if w.q_dtype == "f16" else 1, fda.DTYPE_CODES[w.kv_dtype],
                                     w.paged, max(w.page_size, 1))
        for _ in range(5):
            flush()
            step()
        torch.cuda.synchronize()
        st, info = fda.fd_check_device_error(ws)
        if st != 0:
            raise RuntimeError(f"{name}: device error {fda.fd_status_string(st)} info={info}")
        ms = timed_steps(step, flush, stream, K)
        alg = w.algorithmic_bytes()
        mean_ms = sum(ms) / K
        e = {"workload": fw.WORKLOAD_NAMES[cfg], "steps": K, "us_per_step": round(mean_ms * 1e3, 2),
             "us_per_step_p10_p50_p90": [pct(ms, 10), pct(ms, 50), pct(ms, 90)],
             "kernel": KERNEL_IDS.get(sel, "none")}
        if kv != "e4m3":
            e["kv_dtype"] = kv
        if scales != "tensor":
            e["kv_scales"] = f"per {scales}"
        if q_len > 1:
            e["q_len"] = q_len
        if cfg == 1:
            e["note"] = "latency-bound (12 KB per step): time only"
        else:
            sms = timed_steps(step, flush, stream, K, split_events=True)
            split_ms = sum(sms) / K
            gbs = alg / (mean_ms * 1e-3) / 1e9
            e.update({"algorithmic_bytes_per_step": alg, "gbs": round(gbs, 1),
                      "frac": round(gbs / peak, 4), "split_us": round(split_ms * 1e3, 2),
                      "split_frac": round(alg / (split_ms * 1e-3) / 1e9 / peak, 4)})
        res[name] = e
        fda.fd_set_kernel({"auto": 0, "simt": 1, "mma": 2, "tc": 3, "fma": 4}[args.kernel])
        del t, out, lse, ws
        torch.cuda.empty_cache()
    return res


def run_gpu(args):
    import torch
    import flash_decoding_attention_gb300 as fda
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    fda.load_library()
    fda.fd_set_kernel({"auto": 0, "simt": 1, "mma": 2, "tc": 3, "fma": 4}[args.kernel])

    w = make_workload(args)
    t = fw.to_torch(w, dev)
    B, QH, KVH, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:-1], dtype=torch.float32, device=dev)
    ws = fda.alloc_workspace(B, QH * w.q_len, KVH, D, dev)
    stream = torch.cuda.current_stream(dev)
    sel = fda.fd_selected_kernel(QH * w.q_len, KVH, D, 0 if w.q_dtype == "f16" else 1,
                                 fda.DTYPE_CODES[w.kv_dtype], w.paged,
                                 max(w.page_size, 1))
    kname = {1: "simt", 2: "mma", 3: "tc", 4: "fma"}.get(sel, "none")

    if args.append:
        k_new, v_new = fw.new_tokens(w, 500 + args.config, n_new=w.q_len)
        qd, _ = fw.torch_dtypes(w)
        t["k_new"] = torch.from_numpy(k_new.view(np.int16)).view(qd).to(dev)
        t["v_new"] = torch.from_numpy(v_new.view(np.int16)).view(qd).to(dev)
        t["positions"] = torch.from_numpy(fw.last_positions(w, w.q_len)).to(dev)

    step = make_step(fda, w, t, out, lse, ws, stream, append=args.append)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(2 * l2 // 4, dtype=torch.int32, device=dev)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.int32, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.max()

    for _ in range(args.warmup):
        flush()   # also loads the flush kernels before anything is timed
        step()
    torch.cuda.synchronize()
    st, info = fda.fd_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error {fda.fd_status_string(st)} info={info}")

    K = args.steps
    clocks = ClockSampler(local, not args.no_clocks)
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    # headline: whole decode steps, L2 flushed before each
    step_ms = timed_steps(step, flush, stream, K)
    # roofline: the same steps again with events around the split kernel alone
    # (an event between two launches of a step stops them from overlapping,
    # so these steps are not used for the headline)
    split_ms = timed_steps(step, flush, stream, K, split_events=True)
    # diagnostic only: back-to-back steps without the L2 flush (inputs partly
    # L2-resident from the previous step), events around the whole run
    n_hot = min(K, 200)
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    h0.record(stream)
    for i in range(n_hot):
        step()
    h1.record(stream)
    torch.cuda.synchronize()
    hot_us = h0.elapsed_time(h1) / n_hot * 1e3
    if pg:
        pg.barrier()
    clk = clocks.stop()
    total_ms = sum(step_ms)
    if pg:
        total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / K
    alg = w.algorithmic_bytes() + (fw.append_bytes(w, w.q_len) if args.append else 0)
    value = whole_job_throughput(alg, world, ms_per_step * 1e-3) / 1e9

    # end to end through the public API: pinned host inputs in, result out
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else max(3, min(K, 50))
    e2e = None
    if e2e_steps > 0:
        h = fw.to_torch(w, "cpu", pin=True)
        if args.append:
            for key in ("k_new", "v_new", "positions"):
                h[key] = t[key].cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h_lse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        dev_in = {k: (torch.empty_like(v, device=dev) if v is not None else None) for k, v in h.items()}
        h2d = sum(v.numel() * v.element_size() for v in h.values() if v is not None)
        d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()

        def e2e_step():
            for k, v in h.items():
                if v is not None:
                    dev_in[k].copy_(v, non_blocking=True)
            fda.decode_attention(dev_in["q"], dev_in["k"], dev_in["v"], dev_in["seq_len"],
                                 kv_start_idx=dev_in["kv_start_idx"], block_table=dev_in["block_table"],
                                 softmax_scale=float(w.softmax_scale), k_scale=float(w.k_scale),
                                 v_scale=float(w.v_scale), workspace=ws, out=out, lse=lse,
                                 k_scales=dev_in.get("k_scales"), v_scales=dev_in.get("v_scales"),
                                 k_new=dev_in.get("k_new"), v_new=dev_in.get("v_new"),
                                 positions=dev_in.get("positions"))
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
        if pg:
            e2e_ms = max_over_ranks(e2e_ms, dev)
        e2e_val = whole_job_throughput(alg, world, e2e_ms * 1e-3) / 1e9
        e2e = {"value": round(e2e_val, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)}

    st, info = fda.fd_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error {fda.fd_status_string(st)} info={info}")

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    split_avg = sum(split_ms) / K
    achieved = alg / (split_avg * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    per_config = None
    if not args.no_per_config and world == 1:
        clocks2 = ClockSampler(local, not args.no_clocks)
        per_config = per_config_timings(args, dev, stream, flush, peak, kname)
        clk2 = clocks2.stop()
        if clk2:
            per_config["clocks"] = clk2
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "us_per_step_p10_p50_p90": [pct(step_ms, q) for q in (10, 50, 90)],
        "us_per_step_max": round(max(step_ms) * 1e3, 2),
        "slow_steps": int(sum(1 for x in step_ms if x > 1.5 * float(np.median(step_ms)))),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (f"{w.kv_dtype}->{w.q_dtype} {TENSOR_LABEL.get(kname, 'fma')}, f32 acc"
                  if w.kv_dtype in ("e4m3", "i8")
                  else f"{w.kv_dtype} {TENSOR_LABEL.get(kname, 'fma')}, f32 acc"),
        "data": "synthetic",
        "config": {**workload_config(args), "kernel": kname,
                   "algorithmic_bytes_per_step": alg, "sum_seq_len": int(w.seq_len.sum()),
                   "l2": "flushed between steps (write then read of 2x L2 buffers, outside the "
                         "timed events)",
                   "parallelism": f"replicas x{world}"},
        # split + combine (+ append) per step: the headline loop, the
        # roofline loop and the unflushed diagnostic
        "gpu_launches": (3 if args.append else 2) * (2 * K + n_hot),
        "diagnostic_unflushed_us_per_step": round(hot_us, 2),
        "env": device_env(dev),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None if (args.shared_prefix or args.scales != "tensor")
                     else recorded_traffic(kname, args.config),
                     "kernel": f"split ({kname})",
                     "split_us": round(split_avg * 1e3, 2)},
        "e2e": e2e,
        "clocks": clk,
    }
    if per_config is not None:
        line["per_config"] = per_config
    if not args.no_cpu_baseline and args.gpus == 1:
        gbs, threads, desc, _ = oracle_sample(w, budget_s=15.0)
        gbs1, _, desc1, _ = oracle_sample(w, budget_s=3.0, nthreads=1)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": desc,
                                "value_1thread": round(gbs1, 4), "sample_1thread": desc1}
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
