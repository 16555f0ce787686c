#!/usr/bin/env python3
"""Benchmark of the jagged attention hot path: one step = forward + backward of one batch.

Default workload (``gdpa``): B=256 causal jagged self-attention with the non-softmax
activation P = SiLU(QK^T/sqrt(D))/L, lengths uniform in [256, 4096], H=8, D=128, bf16
inputs with fp32 accumulation -- the largest of the workloads and the one bound by the
tensor cores.  Metric: useful (unpadded) attention TFLOP/s of forward + backward; also
reported as a fraction of the measured dense BF16 peak.  Other workloads run with
``--workload``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent replica of
the workload on its own GPU (the path has no cross-sequence exchange), timing is the
maximum over ranks, and the value is the aggregate over all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "useful (unpadded) attention TFLOP/s fwd+bwd on 1 GB300; % of dense BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
# the sources each kernel is compiled from (its file and the headers it includes)
_TC_HEADERS = ("tc.h", "tc_host.h", "tc_ptx.cuh", "feed.cuh", "internal.h")
KERNEL_SOURCES = {"fwd": ("tc_fwd.cu",) + _TC_HEADERS, "bwd_dkdv": ("tc_bwd.cu",) + _TC_HEADERS,
                  "bwd_dq": ("tc_bwd.cu",) + _TC_HEADERS, "bwd_d": ("tc_bwd.cu",) + _TC_HEADERS,
                  "schedule": ("sched.cu", "internal.h")}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, world, device):
    """The largest x over all ranks: a job is as slow as its slowest replica."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(step_flops, world, seconds_per_step):
    """Whole-job throughput: every rank processes one batch of step_flops per step."""
    return world * step_flops / seconds_per_step / 1e12


def replica_seed(rank):
    """Each replica draws its own input values (same lengths, same shapes)."""
    return rank


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        out = {}
        for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            val = d.get(key)
            if isinstance(val, dict):
                val = val.get("value")
            out[key] = float(val)
        return out, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_flops_bytes(w, lq, lk, tq, tk):
    """Algorithmic FLOPs and bytes of one launch of each kernel kind.

    fwd:  QK^T and PV over the valid pairs; reads Q, K, V, writes O and lse.
    dkdv: S^T and dP^T recompute, dV and dK products; reads Q, K, V, dO, lse, D, writes dK, dV.
    dq:   S and dP recompute, dQ product; reads Q, K, V, dO, lse, D, writes dQ.
    d:    the row pass; reads O, dO and lse, writes the (lse, D) pairs.
    aux:  pooled attention's broadcast (writes the T_q query rows) or sum (reads the T_q
          per-sequence query-gradient rows); BlockAttention's block offsets.
    """
    P = workloads.valid_pairs(lq, lk, w.causal, w.block)
    H, dq, dv = w.heads, w.dim_qk, w.dim_v
    e = 2 if w.dtype == torch.bfloat16 else 4
    sm = w.act == workloads.ACT_SOFTMAX
    rowb = 8 * H * tq if sm else 0
    if w.pooled:
        aux = e * H * dq * tq
    elif w.block:
        n_blocks = int(sum(-(-int(n) // w.block) for n in lq))
        aux = 8 * (len(lq) + 1) + 8 * (n_blocks + 1)
    else:
        aux = 0
    return {
        "fwd": (2 * P * H * (dq + dv), e * H * (tq * dq + tk * dq + tk * dv + tq * dv) + (4 * H * tq if sm else 0)),
        "bwd_dkdv": (2 * P * H * (2 * dq + 2 * dv),
                     e * H * (tq * dq + tk * dq + tk * dv + tq * dv + tk * dq + tk * dv) + rowb),
        "bwd_dq": (2 * P * H * (2 * dq + dv),
                   e * H * (tq * dq + tk * dq + tk * dv + tq * dv + tq * dq) + rowb),
        "bwd_d": (2 * H * tq * dv, e * H * 2 * tq * dv + 12 * H * tq),
        "schedule": (0, 8 * (len(lq) + 1) * 2),
        "aux": (0, aux),
    }


def file_sha(names):
    """Hash of the named kernel sources, concatenated in order (None if one is missing)."""
    h = hashlib.sha256()
    for name in names:
        p = os.path.join(ROOT, "jagged_attention_recsys_gb300", "csrc", name)
        try:
            h.update(open(p, "rb").read())
        except OSError:
            return None
    return h.hexdigest()[:16]


def measured_traffic(kind, workload):
    """DRAM bytes per launch from a committed ncu capture, if the kernel source is unchanged."""
    try:
        d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
        ent = d[workload][kind]
    except Exception:
        return None
    if ent.get("source_sha") != file_sha(KERNEL_SOURCES.get(kind, ())):
        return None
    return ent.get("dram_bytes_per_launch")


class _Nvml:
    """Read-only NVML queries through ctypes (the driver's libnvidia-ml): SM clock, its
    maximum, and the active clock-event (throttle) reasons of one GPU."""
    # clock-event reason bits (nvml.h)
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}

    def __init__(self, cuda_index):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib, self.c = lib, ctypes
        self.h = ctypes.c_void_p()
        try:  # the CUDA device's PCI address, so that the NVML and CUDA numberings may differ
            pr = torch.cuda.get_device_properties(cuda_index)
            bus = b"%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            rc = lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h))
        except Exception:
            rc = -1
        if rc != 0 and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index),
                                                          ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        self.max_mhz = self._clock(lib.nvmlDeviceGetMaxClockInfo)

    def _clock(self, fn):
        v = self.c.c_uint()
        if fn(self.h, self.c.c_uint(1), self.c.byref(v)) != 0:  # NVML_CLOCK_SM
            raise RuntimeError("clock query failed")
        return float(v.value)

    def sample(self):
        r = self.c.c_ulonglong()
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        if fn is None:  # the older name of the same query
            fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(self.h, self.c.byref(r)) != 0:
            raise RuntimeError("reason query failed")
        flags = ["Active" if r.value & b else "Not Active" for b in
                 (self.BITS["hw_slowdown"], self.BITS["hw_thermal_slowdown"],
                  self.BITS["sw_thermal_slowdown"], self.BITS["sw_power_cap"])]
        return "%s, %s, %s" % (self._clock(self.lib.nvmlDeviceGetClockInfo), self.max_mhz,
                               ", ".join(flags))


class ClockSampler:
    """SM clocks and throttle reasons, sampled in the background: through NVML every
    10 ms where the driver's library loads, else from nvidia-smi every 50 ms.

    Each sample is stamped with the host time it was taken; the summary covers the
    samples inside the marked window (``mark_start`` / ``mark_end``), or, when the window
    is shorter than the sampling period, the nearest sample on each side.
    """
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index):
        self.proc = None
        self.nvml = None
        self.stop = False
        self.dev = device_index
        self.stamped = []
        self.t0 = self.t1 = None
        self.source = None

    def _reader(self):
        for line in self.proc.stdout:
            if line.strip():
                self.stamped.append((time.time(), line))

    def _poller(self):
        while not self.stop:
            try:
                self.stamped.append((time.time(), self.nvml.sample()))
            except Exception:
                return
            time.sleep(0.01)

    def __enter__(self):
        import threading
        try:
            self.nvml = _Nvml(self.dev)
            self.nvml.sample()
            self.thread = threading.Thread(target=self._poller, daemon=True)
            self.thread.start()
            self.source = "NVML every 10 ms"
            return self
        except Exception:
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
            deadline = time.time() + 3.0  # let the sampler come up before the timed region
            while not self.stamped and time.time() < deadline:
                time.sleep(0.01)
            self.source = "nvidia-smi every 50 ms"
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        if self.proc is not None or self.nvml is not None:  # one more sample after the window
            n = len(self.stamped)
            deadline = time.time() + 0.5
            while len(self.stamped) == n and time.time() < deadline:
                time.sleep(0.01)

    def __exit__(self, *exc):
        self.stop = True
        if self.nvml is not None:
            self.thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        rows = []
        for t, l in self.stamped:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 6:
                continue
            try:
                rows.append((t, float(parts[0]), float(parts[1]), parts[2:6]))
            except ValueError:
                continue
        if not rows:
            return None
        t0 = self.t0 if self.t0 is not None else rows[0][0]
        t1 = self.t1 if self.t1 is not None else rows[-1][0]
        inside = [r for r in rows if t0 <= r[0] <= t1]
        where = "during the timed region"
        if not inside:  # region shorter than the sampling period: nearest on each side
            before = [r for r in rows if r[0] < t0][-1:]
            after = [r for r in rows if r[0] > t1][:1]
            inside = before + after
            where = "nearest samples around a %.0f ms timed region" % ((t1 - t0) * 1e3)
        reasons = set()
        for r in inside:
            for n, val in zip(self.NAMES, r[3]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "samples": len(inside),
                "window": where, "reasons": sorted(reasons), "source": self.source}


# ----------------------------------------------------------------------------- our arm
def config_of(w, lq, lk, world):
    """The workload as both arms report it (identical keys and values in both lines)."""
    tq, tk = int(np.sum(lq)), int(np.sum(lk))
    if w.pooled:
        tq_in = w.pooled
    else:
        tq_in = tq
    fwd_f, bwd_f = workloads.useful_flops(w, lq, lk)
    e = 2 if w.dtype == torch.bfloat16 else 4
    in_bytes = e * w.heads * (tq_in * w.dim_qk + tk * (w.dim_qk + w.dim_v) + tq * w.dim_v)
    return {"workload": w.name, "batch": w.batch, "heads": w.heads, "dim_qk": w.dim_qk,
            "dim_v": w.dim_v, "causal": w.causal,
            "activation": "softmax" if w.act == workloads.ACT_SOFTMAX else "silu_over_len",
            "cross": w.cross, "pooled_queries": w.pooled or None, "block": w.block or None,
            "rope": w.rope or None,
            "total_q": tq, "total_k": tk,
            "useful_gflop_fwd": round(fwd_f / 1e9, 3), "useful_gflop_bwd": round(bwd_f / 1e9, 3),
            "l2": "inputs %.2f GB (L2 is 0.13 GB); the GPU arm also writes 256 MiB between "
                  "timed steps" % (in_bytes / 1e9),
            "parallelism": "replicas" if world > 1 else "single"}


def gpu_step_fn(jfa, w, d, ws):
    """One step as a training loop issues it: the batch's work lists built once (the plan),
    then the forward and backward calls on them.  The pooled calls schedule for themselves
    (they take no plan)."""
    q, k, v, do, oq, ok = d["q"], d["k"], d["v"], d["do"], d["oq"], d["ok"]
    o, lse, dq, dk, dv = d["o"], d["lse"], d["dq"], d["dk"], d["dv"]
    sc = w.scale
    if w.block:
        def step():
            jfa.jfa_block_plan(q, k, v, oq, scale=sc, causal=w.causal, ws=ws)
            jfa.jfa_block_fwd(q, k, v, oq, scale=sc, causal=w.causal, o=o, lse=lse, ws=ws,
                              rope=w.rope, planned=True)
            jfa.jfa_block_bwd(q, k, v, o, lse, do, oq, scale=sc, causal=w.causal, dq=dq, dk=dk,
                              dv=dv, ws=ws, rope=w.rope, planned=True)
    elif w.pooled:
        def step():
            jfa.jfa_pooled_fwd(q, k, v, ok, scale=sc, o=o, lse=lse, ws=ws)
            jfa.jfa_pooled_bwd(q, k, v, o, lse, do, ok, scale=sc, dq=dq, dk=dk, dv=dv, ws=ws)
    elif w.act == workloads.ACT_SILU_OVER_LEN:
        def step():
            jfa.jfa_plan(q, k, v, oq, ok, scale=sc, causal=w.causal, ws=ws)
            jfa.jfa_gdpa_fwd(q, k, v, oq, ok, scale=sc, causal=w.causal, o=o, ws=ws, planned=True)
            jfa.jfa_gdpa_bwd(q, k, v, do, oq, ok, scale=sc, causal=w.causal, dq=dq, dk=dk, dv=dv,
                             ws=ws, planned=True)
    elif w.cross:
        def step():
            jfa.jfa_plan(q, k, v, oq, ok, scale=sc, ws=ws)
            jfa.jfa_cross_fwd(q, k, v, oq, ok, scale=sc, o=o, lse=lse, ws=ws, planned=True)
            jfa.jfa_cross_bwd(q, k, v, o, lse, do, oq, ok, scale=sc, dq=dq, dk=dk, dv=dv, ws=ws,
                              planned=True)
    else:
        def step():
            jfa.jfa_plan(q, k, v, oq, scale=sc, causal=w.causal, ws=ws)
            jfa.jfa_fwd(q, k, v, oq, scale=sc, causal=w.causal, o=o, lse=lse, ws=ws,
                        planned=True)
            jfa.jfa_bwd(q, k, v, o, lse, do, oq, scale=sc, causal=w.causal, dq=dq, dk=dk, dv=dv,
                        ws=ws, planned=True)
    return step


def cpu_baseline(w, lq, lk, budget_s=12.0, seed=0):
    """The fp64 oracle, as it stands, on a bounded seeded sample of the workload's sequences."""
    import oracle

    cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    rng = np.random.default_rng(seed + 7)
    order = rng.permutation(len(lq))
    per_flop = 1.0 / (3.0e9 * cores)  # plain fp64 loops run at roughly 3-4 GFLOP/s per core
    chosen, est = [], 0.0
    for b in order:
        f, g = workloads.useful_flops(w, [lq[b]], [lk[b]])
        chosen.append(int(b))
        est += (f + g) * per_flop
        if est >= budget_s:
            break
    slq = [int(lq[b]) for b in chosen]
    slk = [int(lk[b]) for b in chosen]
    oq, ok = workloads.offsets(slq), workloads.offsets(slk)
    q, k, v, do = workloads.values(int(oq[-1]), int(ok[-1]), w.heads, w.dim_qk, w.dim_v,
                                   w.dtype, seed=seed)
    f64 = lambda t: t.to(torch.float64).numpy()
    q, k, v, do = f64(q), f64(k), f64(v), f64(do)
    oracle.build()
    t0 = time.perf_counter()
    if w.pooled:
        oracle.pooled_fwd(q[:w.pooled], k, v, ok, scale=w.scale)
        oracle.pooled_bwd(q[:w.pooled], k, v, do, ok, scale=w.scale)
    elif w.block and w.rope:
        oracle.block_rope_fwd(q, k, v, oq, scale=w.scale, causal=w.causal)
        oracle.block_rope_bwd(q, k, v, do, oq, scale=w.scale, causal=w.causal)
    elif w.block:
        oracle.block_fwd(q, k, v, oq, scale=w.scale, causal=w.causal)
        oracle.block_bwd(q, k, v, do, oq, scale=w.scale, causal=w.causal)
    else:
        oracle.fwd(q, k, v, oq, ok, scale=w.scale, causal=w.causal, act=w.act)
        oracle.bwd(q, k, v, do, oq, ok, scale=w.scale, causal=w.causal, act=w.act)
    dt = time.perf_counter() - t0
    f, g = workloads.useful_flops(w, slq, slk)
    return {"value": (f + g) / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "seconds": dt,
            "sample": "%d of %d sequences (seeded), fp64 forward+backward, %.3g useful GFLOP"
                      % (len(chosen), len(lq), (f + g) / 1e9)}


def run_ours(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import jagged_attention_recsys_gb300 as jfa

    jfa.lib()
    w = workloads.WORKLOADS[args.workload]
    lq, lk = workloads.lengths(w.name, seed=0)
    if args.max_seqs:
        # profiling aid: the first N sequences of the workload (not a benchmark line)
        lq, lk = lq[:args.max_seqs], lk[:args.max_seqs]
    batch = workloads.make_batch(w, lq, lk, seed=replica_seed(rank), device=dev)
    d = dict(q=batch["q"], k=batch["k"], v=batch["v"], do=batch["do"],
             oq=torch.as_tensor(batch["offs_q"], device=dev),
             ok=torch.as_tensor(batch["offs_k"], device=dev))
    tq, tk = int(batch["offs_q"][-1]), d["k"].shape[0]
    d["o"] = torch.empty(tq, w.heads, w.dim_v, dtype=w.dtype, device=dev)
    d["lse"] = torch.empty(tq, w.heads, dtype=torch.float32, device=dev)
    d["dq"] = torch.empty_like(d["q"])
    d["dk"] = torch.empty_like(d["k"])
    d["dv"] = torch.empty_like(d["v"])
    if w.pooled:
        p, m = jfa.pooled_params(d["q"], d["k"], d["v"], d["ok"], w.scale)
        ws = jfa.pooled_workspace(p, m, dev)
    elif w.block:
        p = jfa.params_for(d["q"], d["k"], d["v"], d["oq"], w.scale, w.causal)
        ws = jfa.block_workspace(p, dev)
    else:
        p = jfa.params_for(d["q"], d["k"], d["v"], d["oq"], w.scale, w.causal)
        ws = jfa.workspace(p, dev)
    step = gpu_step_fn(jfa, w, d, ws)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    fwd_f, bwd_f = workloads.useful_flops(w, lq, lk)
    step_flops = fwd_f + bwd_f

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = jfa.jfa_status_check(ws)
    if st != 0:
        raise RuntimeError("device status after warm-up: %s" % jfa.status_string(st))
    run, launch = capture_graph(jfa, step, ws) if not args.no_graph else (step, "eager")

    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark_start()
        for i in range(args.steps):
            flush.fill_(float(i))  # evicts the inputs from L2 between timed steps
            starts[i].record(stream)
            run()
            ends[i].record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    ms_total = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)), world, dev)
    if world > 1:
        torch.distributed.barrier()
    # per-kernel times: the same steps launched one call at a time with event timing (the
    # graph replays exactly these kernels)
    jfa.jfa_profile_reset()
    jfa.jfa_profile_enable(True)
    for i in range(args.steps):
        flush.fill_(float(i))
        step()
    torch.cuda.synchronize()
    jfa.jfa_profile_enable(False)
    prof = {k: jfa.jfa_profile_read(k) for k in jfa.KERNEL_KINDS}
    launches = sum(n for n, _ in prof.values())
    ms_per_step = ms_total / args.steps
    value = job_tflops(step_flops, world, ms_per_step * 1e-3)

    # roofline of the dominant kernel
    pk, peak_src = peaks()
    per_kernel = kernel_flops_bytes(w, lq, lk, tq, tk)
    kind = max(prof, key=lambda k: prof[k][1])
    n_launch, kms = prof[kind]
    avg_s = kms / max(n_launch, 1) * 1e-3
    kf, kb = per_kernel[kind]
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    bound = "tensor" if kb == 0 or kf / kb >= ridge else "hbm"
    if bound == "tensor":
        achieved, peak, unit = kf / avg_s / 1e12, pk["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = kb / avg_s / 1e9, pk["hbm_gbs"], "GB/s"
    roof = {"kernel": kind, "bound": bound, "achieved": round(achieved, 2), "peak": peak,
            "unit": unit, "frac": round(achieved / peak, 4), "peak_source": peak_src,
            "traffic": measured_traffic(kind, w.name),
            "algorithmic_flops_per_launch": kf, "algorithmic_bytes_per_launch": kb,
            "avg_launch_ms": round(kms / max(n_launch, 1), 5)}
    kernels = {k: {"launches": n, "ms_per_launch": round(ms / max(n, 1), 5),
                   "share": round(ms / max(sum(x for _, x in prof.values()), 1e-12), 4)}
               for k, (n, ms) in prof.items() if n}

    # end to end through the public API with pinned host buffers
    e2e = None if args.no_e2e else e2e_measure(jfa, w, batch, d, ws, p, args, dev, step_flops,
                                                 world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, lq, lk)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if w.dtype == torch.bfloat16 else "f32", "data": "synthetic (seeded, no padding)",
        "frac_of_bf16_peak": round(value / world / pk["bf16_tflops"], 4),
        "config": config_of(w, lq, lk, world),
        "timing": {"l2_flush": "256 MiB written between timed steps", "launch": launch,
                   "schedule": "pooled: each call builds its lists" if w.pooled else
                               "one plan per step, used by the forward and backward calls",
                   "max_seqs": args.max_seqs or None},
        "roofline": roof, "kernels": kernels, "gpu_launches": launches,
        "e2e": e2e, "cpu_baseline": cpu, "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def capture_graph(jfa, step, ws):
    """One step (the library's forward and backward calls, as a training loop issues them)
    captured in a CUDA graph; returns (replay function, launch description).  Steps whose
    capture fails run as separate calls."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm the library's own streams and events off-capture
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        g.replay()
        torch.cuda.synchronize()
        st = jfa.jfa_status_check(ws)
        if st != 0:
            raise RuntimeError(jfa.status_string(st))
        return g.replay, "one CUDA graph per step (the library's calls captured)"
    except Exception as e:  # noqa: BLE001 - report and time the calls instead
        return step, "separate calls (graph capture failed: %s)" % str(e).splitlines()[0][:100]


def e2e_measure(jfa, w, batch, d, ws, p, args, dev, step_flops, world):
    """The metric end to end through the public API: every step copies its inputs from
    pinned host memory to the device, runs forward and backward, and copies its results
    (O, dQ, dK, dV) back to pinned host memory, all inside the timed region.  Steps are
    pipelined as a serving loop would run them: two device buffer sets, the copies on
    their own streams, so that step i+1's inputs arrive and step i-1's results leave while
    step i computes."""
    names_in = ["q", "k", "v", "do"]
    host = {n: batch[n].to("cpu").pin_memory() for n in names_in}
    host["oq"] = torch.as_tensor(batch["offs_q"]).pin_memory()
    host["ok"] = torch.as_tensor(batch["offs_k"]).pin_memory()
    outs = ["o", "dq", "dk", "dv"]
    host_out = {n: torch.empty(d[n].shape, dtype=d[n].dtype).pin_memory() for n in outs}
    sets = [dict(d), {n: torch.empty_like(t) for n, t in d.items()}]
    steps = [gpu_step_fn(jfa, w, st, ws) for st in sets]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(d[n].numel() * d[n].element_size() for n in outs)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}

    def run(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:  # set b's inputs are free once step i-2 has run
                    s_in.wait_event(ev["comp"][b])
                for name, t in host.items():
                    sets[b][name].copy_(t, non_blocking=True)
                ev["in"][b].record(s_in)
            comp.wait_event(ev["in"][b])
            if i >= 2:  # set b's outputs are free once step i-2's results have left
                comp.wait_event(ev["out"][b])
            steps[b]()
            ev["comp"][b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["comp"][b])
                for name in outs:
                    host_out[name].copy_(sets[b][name], non_blocking=True)
                ev["out"][b].record(s_out)
        torch.cuda.synchronize()

    run(max(2, args.warmup))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(args.steps)
    dt = max_over_ranks(time.perf_counter() - t0, world, dev)
    return {"value": round(job_tflops(step_flops, world, dt / args.steps), 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(dt / args.steps * 1e3, 4),
            "pipelined": "two device buffer sets; host-to-device and device-to-host copies on "
                         "their own streams overlap the neighbouring steps' kernels"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    lq, lk = workloads.lengths(w.name, seed=0)
    budget = max(2.0, 150.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        cpu_baseline(w, lq, lk, budget_s=budget)
    vals, secs = [], 0.0
    res = None
    for _ in range(args.steps):
        res = cpu_baseline(w, lq, lk, budget_s=budget)
        vals.append(res["value"])
        secs += res["seconds"]
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / max(args.steps, 1) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": config_of(w, lq, lk, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": res["cores"],
                         "kind": "oracle", "sample": res["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="gdpa", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step as separate API calls instead of one CUDA graph")
    ap.add_argument("--no-e2e", action="store_true",
                    help="profiling aid: skip the end-to-end measurement (and its buffers)")
    ap.add_argument("--max-seqs", type=int, default=0,
                    help="profiling aid: only the first N sequences of the workload")
    args = ap.parse_args()
    if args.warmup < 3:
        log("note: warm-up raised to 3 steps (minimum)")
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
