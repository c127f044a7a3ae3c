"""Throughput of zigzag context-parallel causal attention (forward + backward).

One step = one pass of the whole hot path over one batch of synthetic input:
cp_attn_fwd (zigzag index and gather, one persistent tensor-core launch over
all P ring steps whose online softmax is the log-sum-exp merge) followed by
cp_attn_bwd (preprocess, one tensor-core launch over all P ring steps that
sums dK / dV on chip, prefix gradient sum).  The other bf16 workloads of the method are measured the same way and
reported under "workloads".  Default workload: "long" -- 131072 text tokens, P = 8
simulated ranks, 32 heads, head_dim 128, bf16; inputs are ~1 GiB per tensor,
far larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on the host cores

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs an
independent replica (the path does not shard across GPUs); value is the sum
of all ranks' work over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from vlm_zigzag_head_gb300 import workloads as W  # noqa: E402

METRIC = "CP causal attention TFLOP/s fwd & fwd+bwd, % of GB300 BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# tensor-core backward on the named workload, from one ncu capture of this
# kernel (scaled from a smaller case where stated).  An entry is removed when
# the kernel changes, until it is captured again.
MEASURED_TRAFFIC = {"long": 26.99e9}
EX2_PER_CLK_SM = 32.0   # MUFU exp2 results per clock per SM (31.8 measured by a throughput loop)
# every bf16 forward + backward workload of the method; the default line's
# `value` is the 128K one, the others are reported under `workloads`
OTHER_WORKLOADS = ("long", "vlm_prefix", "packed_vlm", "text_llm")


def causal_pairs(w) -> int:
    """Visible (query, key) pairs per head: per sample n(n+1)/2 over [prefix, text]."""
    return sum((w.prefix_len + L) * (w.prefix_len + L + 1) // 2 for L in W.text_lengths(w))


def fwd_flops(w) -> float:
    """Algorithmic forward FLOPs: 4 d per visible pair and head (QK^T + PV)."""
    return 4.0 * w.d * w.H * causal_pairs(w)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", "cpattn_clocks_%d_%d.csv" % (os.getpid(), index))

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def oracle_sample(w, n_queries: int = 8192):
    """A bounded, exact piece of the workload for the CPU oracle: the first
    n_queries text tokens of sample 0, head 0 (causal: they see only keys
    before them), forward and backward.  Returns (seconds, algorithmic FLOPs,
    description)."""
    import numpy as np  # noqa: F401
    import oracle
    x = W.make_inputs(w)
    a = 0
    n = min(n_queries, x.cu_seqlens[1])
    q, k, v, do = (t[a:a + n, :1] for t in (x.q, x.k, x.v, x.dout))
    cu = [0, n]
    t0 = time.perf_counter()
    oracle.causal_attention_fwd(q, k, v, cu, x.scale)
    oracle.causal_attention_bwd(q, k, v, do, cu, x.scale)
    dt = time.perf_counter() - t0
    flops = 3.5 * 4.0 * w.d * (n * (n + 1) // 2)
    desc = ("first %d tokens of sample 0, head 0 of the '%s' workload (causal: a complete "
            "slice of its work), oracle forward + backward in fp64" % (n, w.name))
    return dt, flops, desc


def time_workload(cp, w, dev, steps: int, warmup: int) -> dict:
    """Forward, backward and forward+backward rates of one bf16 workload, inputs
    resident on the device, CUDA events on the launching stream."""
    x = W.make_inputs(w)
    stream = torch.cuda.current_stream(dev)
    qd, kd, vd, dod = (t.to(dev) for t in (x.q, x.k, x.v, x.dout))
    cu, P, N, scale = x.cu_seqlens, w.P, w.prefix_len, x.scale
    T, H, d = qd.shape
    Hkv = kd.shape[1]
    out, out_lo = torch.empty_like(qd), torch.empty_like(qd)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    grads = (torch.empty((T, H, d), dtype=torch.float32, device=dev),
             torch.empty((T, Hkv, d), dtype=torch.float32, device=dev),
             torch.empty((T, Hkv, d), dtype=torch.float32, device=dev))
    ws_f, ws_b = cp.Workspace(dev), cp.Workspace(dev)

    def fwd():
        cp.cp_attn_fwd(qd, kd, vd, cu, P, N, scale, out=out, lse=lse, workspace=ws_f,
                       residual=True, out_lo=out_lo)

    def bwd():
        cp.cp_attn_bwd(qd, kd, vd, out, lse, dod, cu, P, N, scale, workspace=ws_b, grads=grads,
                       out_lo=out_lo)

    def timed(fn, n):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a0.record(stream)
        for _ in range(n):
            fn()
        a1.record(stream)
        torch.cuda.synchronize(dev)
        return a0.elapsed_time(a1) / n

    for _ in range(warmup):
        fwd()
        bwd()
    torch.cuda.synchronize(dev)
    if cp.cp_workspace_status(ws_f) or cp.cp_workspace_status(ws_b):
        raise RuntimeError("a device wait timed out on workload %s" % w.name)
    f = fwd_flops(w)
    fwd_ms = timed(fwd, steps)
    bwd_ms = timed(bwd, steps)
    step_ms = timed(lambda: (fwd(), bwd()), steps)
    if cp.cp_workspace_status(ws_f) or cp.cp_workspace_status(ws_b):
        raise RuntimeError("a device wait timed out on workload %s" % w.name)
    return {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "ms_per_step": step_ms,
            "fwd_tflops": f / fwd_ms / 1e9, "bwd_tflops": 2.5 * f / bwd_ms / 1e9,
            "tflops": 3.5 * f / step_ms / 1e9, "flops_per_step": 3.5 * f,
            "softmax_scale": x.scale, "steps": steps, "warmup": warmup}


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time (the job finishes with its last replica)."""
    if dist is None:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_step: float, world: int, steps: int, ms: float) -> float:
    """TFLOP/s of the whole job: every replica runs the workload once per step."""
    return world * flops_per_step * steps / (ms / 1e3) / 1e12


def workload_config(w, world) -> dict:
    """The `config` object of both arms' JSON lines."""
    return {"workload": w.name, "text_len": W.text_lengths(w), "prefix_len": w.prefix_len,
            "P": w.P, "heads": w.H, "kv_heads": w.kv_heads, "head_dim": w.d,
            "n_seqs": w.n_seqs, "parallelism": "replicas" if world > 1 else "single",
            "l2": "inputs larger than L2 (no flush)"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return 0
    cores = os.cpu_count()
    times, flops = [], 0.0
    desc = ""
    n_q = args.oracle_queries
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample(w, n_q // 2)
    for _ in range(args.steps):
        dt, flops, desc = oracle_sample(w, n_q)
        times.append(dt)
    t = sum(times) / len(times)
    val = flops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(workload_config(w, world), sample=desc),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# CUDA leg
# ---------------------------------------------------------------------------
def run_cuda(args, w, rank, world, dist):
    import vlm_zigzag_head_gb300 as cp
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    x = W.make_inputs(w)
    stream = torch.cuda.current_stream(dev)
    qd, kd, vd, dod = (t.to(dev) for t in (x.q, x.k, x.v, x.dout))
    cu, P, N, scale = x.cu_seqlens, w.P, w.prefix_len, x.scale
    T, H, d = qd.shape
    out = torch.empty_like(qd)
    out_lo = torch.empty_like(qd)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    Hkv = kd.shape[1]
    grads = (torch.empty((T, H, d), dtype=torch.float32, device=dev),
             torch.empty((T, Hkv, d), dtype=torch.float32, device=dev),
             torch.empty((T, Hkv, d), dtype=torch.float32, device=dev))
    ws_f, ws_b = cp.Workspace(dev), cp.Workspace(dev)

    def step():
        cp.cp_attn_fwd(qd, kd, vd, cu, P, N, scale, out=out, lse=lse, workspace=ws_f,
                       residual=True, out_lo=out_lo)
        cp.cp_attn_bwd(qd, kd, vd, out, lse, dod, cu, P, N, scale, workspace=ws_b, grads=grads,
                       out_lo=out_lo)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if cp.cp_workspace_status(ws_f) or cp.cp_workspace_status(ws_b):
        raise RuntimeError("a device wait timed out during warm-up")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    f_flops = fwd_flops(w)
    total = 3.5 * f_flops
    # ---- timed region: K steps, CUDA events on the launching stream
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        cp.cp_profile_begin()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        barrier()
        prof = cp.cp_profile_end()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, dist, dev)
    if cp.cp_workspace_status(ws_f) or cp.cp_workspace_status(ws_b):
        raise RuntimeError("a device wait timed out in the timed region")
    ms_step = ms / args.steps
    value = whole_job_value(total, world, args.steps, ms)
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))

    # fwd-only and bwd-only timing (same workload, separate short loops)
    def timed(fn, n):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a0.record(stream)
        for _ in range(n):
            fn()
        a1.record(stream)
        torch.cuda.synchronize(dev)
        return a0.elapsed_time(a1) / n

    n_sub = max(1, min(args.steps, 3))
    fwd_ms = timed(lambda: cp.cp_attn_fwd(qd, kd, vd, cu, P, N, scale, out=out, lse=lse,
                                          workspace=ws_f, residual=True, out_lo=out_lo), n_sub)
    bwd_ms = timed(lambda: cp.cp_attn_bwd(qd, kd, vd, out, lse, dod, cu, P, N, scale,
                                          workspace=ws_b, grads=grads, out_lo=out_lo), n_sub)

    # dominant kernel: the tensor-core backward (algorithmic FLOPs: 10 d per
    # visible pair and head), one launch over every ring step of a call
    bwd_ms_k, bwd_launches = prof["tc_bwd_step"]
    fwd_ms_k, fwd_launches = prof["tc_fwd_step"]
    bwd_launch_flops = 2.5 * f_flops
    roof = None
    if bwd_launches:
        avg = bwd_ms_k / bwd_launches
        ach = bwd_launch_flops / (avg / 1e3) / 1e12
        roof = {"kernel": "tc_bwd_q128_kernel (all ring steps)", "bound": "tensor",
                "achieved": ach, "peak": peak_sus, "unit": "TFLOP/s", "frac": ach / peak_sus,
                "peak_source": "%s bf16_tflops_sustained" % peak_src,
                "traffic": (args.traffic if args.traffic is not None
                            else MEASURED_TRAFFIC.get(w.name) if w == W.get(w.name) else None),
                "launch_ms": avg,
                "flops_per_launch": bwd_launch_flops}
    kernels = {}
    for k, (kms, n) in prof.items():
        if n:
            kernels[k] = {"launches": n, "ms_total": kms, "share": kms / max(ms, 1e-9)}
    if fwd_launches:
        # one forward call is one all-steps launch (P ring-step launches under
        # CPATTN_FWD_PER_STEP=1): rate over the kernel time of a whole call
        avg = fwd_ms_k / args.steps
        kernels["tc_fwd_step"]["achieved_tflops"] = f_flops / (avg / 1e3) / 1e12
        # secondary bound: one exp2 per visible pair and head, against the MUFU
        # rate (32 exp2 per clock per SM on this part) at the maximum SM clock
        exps = causal_pairs(w) * H
        mufu = EX2_PER_CLK_SM * torch.cuda.get_device_properties(dev).multi_processor_count * \
            float(peaks.get("sm_max_mhz", 2070.0)) * 1e6
        kernels["tc_fwd_step"]["exp_per_s"] = exps / (avg / 1e3)
        kernels["tc_fwd_step"]["exp_frac"] = exps / (avg / 1e3) / mufu
    # memory kernels: algorithmic bytes per launch against the measured HBM copy rate
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    Hkv = kd.shape[1]
    text_rows = sum(W.text_lengths(w))
    mem_bytes = {
        "zigzag_gather": 2 * text_rows * (H + 2 * Hkv) * d * 2,          # q, k, v rows in and out
        "bwd_preprocess": T * H * d * 2 * 3 + T * H * 4 * 3,              # out, out_lo, dO; lse in, D, lse2 out
    }
    for k, nb in mem_bytes.items():
        if k in kernels:
            avg = kernels[k]["ms_total"] / kernels[k]["launches"]
            kernels[k]["achieved_gbs"] = nb / (avg / 1e3) / 1e9
            kernels[k]["hbm_frac"] = kernels[k]["achieved_gbs"] / hbm
    gpu_launches = sum(n for _, n in prof.values())

    # the standalone LSE merge (cp_lse_merge; inside the step the merge is the
    # forward's online softmax): P partial results of one rank's rows, fp32,
    # merged into bf16 out and fp32 lse, timed on its own
    R = max(1, T // P)
    parts_o = torch.randn((P, R, H, d), device=dev)
    parts_l = torch.randn((P, H, R), device=dev)
    m_out = torch.empty((R, H, d), dtype=torch.bfloat16, device=dev)
    m_lse = torch.empty((H, R), dtype=torch.float32, device=dev)
    merge_ms = timed(lambda: cp.cp_lse_merge(parts_o, parts_l, torch.bfloat16, out=m_out,
                                             lse=m_lse), 5)
    merge_bytes = P * R * H * (d + 1) * 4 + R * H * (d * 2 + 4)
    kernels["lse_merge"] = {"launches": 5, "ms_per_launch": merge_ms, "standalone": True,
                            "shape": [P, R, H, d], "bytes_per_launch": merge_bytes,
                            "achieved_gbs": merge_bytes / (merge_ms / 1e3) / 1e9,
                            "hbm_frac": merge_bytes / (merge_ms / 1e3) / 1e9 / hbm}
    del parts_o, parts_l

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (t.pin_memory() for t in (x.q, x.k, x.v, x.dout))
        host_out = None
        res = cp.attention_host(hq, hk, hv, hdo, cu, P, N, scale, device=dev)
        host_out = list(res)
        n_e2e = max(1, min(args.steps, 3))
        barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            cp.attention_host(hq, hk, hv, hdo, cu, P, N, scale, device=dev, host_out=host_out)
        barrier()
        e2e_s = (time.perf_counter() - t0) / n_e2e
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        # this box's pinned copy rates (one 1 GiB copy each way, outside the
        # timed steps): with every copy hidden behind the kernels the step is
        # bounded below by the slower direction's bytes at its rate
        buf_h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
        buf_d = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
        h2d_ms = timed(lambda: buf_d.copy_(buf_h, non_blocking=True), 2)
        d2h_ms = timed(lambda: buf_h.copy_(buf_d, non_blocking=True), 2)
        # the strided row copies of the head-chunk pipeline (one chunk of q)
        n_ch = cp.host_chunks(T, H, Hkv, d, 2)
        wid, pitch = (H // n_ch) * d * 2, H * d * 2
        rows = min(T, (1 << 30) // pitch)
        def rows_copy(up_):
            dst, src = (buf_d, buf_h) if up_ else (buf_h, buf_d)
            cp._copy_rows(dst, 0, pitch, src, 0, pitch, wid, rows, stream)
        h2d_rows_ms = timed(lambda: rows_copy(True), 2)
        d2h_rows_ms = timed(lambda: rows_copy(False), 2)
        del buf_h, buf_d
        rate = lambda nb, ms: nb / (ms / 1e3) / 1e9  # noqa: E731
        rate_h2d, rate_d2h = rate(1 << 30, h2d_ms), rate(1 << 30, d2h_ms)
        e2e = {"value": world * total / e2e_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_s * 1e3,
               "pinned_copy_gbs": {"h2d": rate_h2d, "d2h": rate_d2h,
                                   "h2d_rows": rate(wid * rows, h2d_rows_ms),
                                   "d2h_rows": rate(wid * rows, d2h_rows_ms),
                                   "row_bytes": wid, "pitch": pitch},
               "chunks": n_ch,
               "copy_floor_ms": max(h2d / rate_h2d, d2h / rate_d2h) / 1e6}

    # ---- the other bf16 workloads of the method (parity configs, measured the
    # same way at fewer steps): fwd, bwd and fwd+bwd rates, and the oracle's
    # wall time on a bounded slice of each
    workloads = {w.name: {"fwd_tflops": world * f_flops / (fwd_ms / 1e3) / 1e12,
                          "bwd_tflops": world * 2.5 * f_flops / (bwd_ms / 1e3) / 1e12,
                          "tflops": value / world, "ms_per_step": ms_step,
                          "pct_of_bf16_peak": 100.0 * (value / world) / peak_sus}}
    if not args.no_workloads:
        for name in OTHER_WORKLOADS:
            if name == w.name:
                continue
            wl = W.get(name, H_kv=args.kv_heads) if args.kv_heads else W.get(name)
            r = time_workload(cp, wl, dev, max(3, min(args.steps, 10)), max(3, args.warmup))
            r["pct_of_bf16_peak"] = 100.0 * r["tflops"] / peak_sus
            workloads[name] = r
    if not args.no_cpu_baseline and world == 1 and rank == 0:
        for name in workloads:
            wl = W.get(name)
            dt, fl, desc = oracle_sample(wl, args.workload_oracle_queries)
            workloads[name]["oracle"] = {"seconds": dt, "tflops": fl / dt / 1e12,
                                         "cores": os.cpu_count(), "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": workload_config(w, world),
            "pct_of_bf16_peak": 100.0 * (value / world) / peak_sus,
            "fwd_tflops": world * f_flops / (fwd_ms / 1e3) / 1e12, "fwd_ms": fwd_ms,
            "bwd_tflops": world * 2.5 * f_flops / (bwd_ms / 1e3) / 1e12, "bwd_ms": bwd_ms,
            "flops_per_step": total,
            "roofline": roof,
            "kernels": kernels,
            "workloads": workloads,
            "gpu_launches": gpu_launches,
            "clocks": clk.summary(),
            "e2e": e2e,
        }
        if not args.no_cpu_baseline and world == 1:
            dt, fl, desc = oracle_sample(w, args.oracle_queries)
            line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s",
                                    "cores": os.cpu_count(), "kind": "oracle", "sample": desc,
                                    "seconds": dt}
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--workload", default="long", choices=sorted(W.WORKLOADS))
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="KV heads for grouped-query attention (default: as many as query heads)")
    ap.add_argument("--text-len", type=int, default=0,
                    help="text tokens of a one-sample workload (smaller profiling cases)")
    ap.add_argument("--oracle-queries", type=int, default=32768)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other bf16 workloads (reported under 'workloads')")
    ap.add_argument("--workload-oracle-queries", type=int, default=8192,
                    help="queries of the oracle slice timed per workload")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args()
    over = {}
    if args.kv_heads:
        over["H_kv"] = args.kv_heads
    if args.text_len:
        if W.get(args.workload).n_seqs != 1:
            raise SystemExit("--text-len applies to one-sample workloads")
        over["text_lens"] = (args.text_len,)
    w = W.get(args.workload, **over)
    if w.dtype != "bf16" or not w.backward:
        raise SystemExit("bench workloads are the bf16 forward+backward ones")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        backend = "nccl" if torch.cuda.is_available() and args.impl == "cuda" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist_mod.init_process_group(backend)
        dist = dist_mod
    try:
        if args.impl == "reference":
            return run_reference(args, w, rank, world)
        return run_cuda(args, w, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
