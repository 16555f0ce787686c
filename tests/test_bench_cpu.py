"""bench.py's reference arm (the fp64 oracle on the host cores) and its JSON line, on CPU.

The GPU arm needs a GB300; the reference arm runs anywhere, so its output contract is
checked here: one JSON line with the shared keys, an `e2e` object with no copies, and,
under torchrun, a single line from rank 0 while the other ranks exit without work.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"]


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_line(d, n_gpus):
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == n_gpus and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "4 of 4 sequences" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable] + ARGS, cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


def test_reference_arm_warmup_floor():
    r = subprocess.run([sys.executable] + ARGS[:-1] + ["1"], cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert _json_lines(r.stdout)[0]["warmup"] == 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + ARGS + ["--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1  # rank 0 alone
    _check_line(lines[0], 2)


def test_roofline_counts_hand_worked():
    """Per-launch algorithmic FLOPs and bytes behind the roofline object, on one causal
    sequence of 3 rows (6 valid pairs), H=2, Dqk=4, Dv=2, bf16."""
    import torch

    import bench
    import workloads

    w = workloads.Workload("t", 1, 2, 4, 2, True, workloads.ACT_SOFTMAX, torch.bfloat16, False)
    r = bench.kernel_flops_bytes(w, [3], [3], 3, 3)
    P, H, dq, dv, T = 6, 2, 4, 2, 3
    assert r["fwd"] == (2 * P * H * (dq + dv), 2 * H * T * (2 * dq + 2 * dv) + 4 * H * T)
    # dK/dV: reads Q, K, V, dO and the (lse, D) pairs; writes dK, dV
    assert r["bwd_dkdv"] == (2 * P * H * (2 * dq + 2 * dv),
                             2 * H * T * (dq + dq + dv + dv + dq + dv) + 8 * H * T)
    # dQ: reads Q, K, V, dO and the pairs; writes dQ
    assert r["bwd_dq"] == (2 * P * H * (2 * dq + dv),
                           2 * H * T * (dq + dq + dv + dv + dq) + 8 * H * T)
    # row pass: reads O, dO, lse; writes the pairs
    assert r["bwd_d"] == (2 * H * T * dv, 2 * H * T * 2 * dv + 12 * H * T)
    assert r["aux"] == (0, 0)


def test_roofline_counts_d64_workload():
    """The default line's dominant kernel, dK/dV on the d64 workload."""
    import bench
    import workloads

    w = workloads.WORKLOADS["d64"]
    lq, lk = workloads.lengths("d64")
    r = bench.kernel_flops_bytes(w, lq, lk, int(lq.sum()), int(lk.sum()))
    assert r["bwd_dkdv"] == (49681547264.0, 212475008)


def test_roofline_counts_auxiliary_kernels():
    import torch

    import bench
    import workloads

    w = workloads.WORKLOADS["pooled"]
    lq, lk = workloads.lengths("pooled")
    tq = int(lq.sum())
    assert bench.kernel_flops_bytes(w, lq, lk, tq, int(lk.sum()))["aux"] == (0, 2 * 4 * 128 * tq)
    w = workloads.Workload("b", 2, 1, 64, 64, True, workloads.ACT_SOFTMAX, torch.bfloat16, False,
                           block=64)
    # lengths 65 and 64: 2 + 1 blocks; reads 3 offsets, writes 4
    assert bench.kernel_flops_bytes(w, [65, 64], [65, 64], 129, 129)["aux"] == (0, 8 * 3 + 8 * 4)


def test_reference_arm_config_is_the_gpu_arms():
    """Both arms describe the workload with the same config dict (config_of)."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads

    r = subprocess.run([sys.executable] + ARGS, cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = _json_lines(r.stdout)[0]
    lq, lk = workloads.lengths("tiny")
    assert line["config"] == json.loads(json.dumps(bench.config_of(
        workloads.WORKLOADS["tiny"], lq, lk, 1)))
    assert line["config"]["activation"] == "softmax" and line["config"]["total_q"] == 105


def test_default_workload_is_gdpa():
    sys.path.insert(0, ROOT)
    import argparse
    import bench

    src = open(os.path.join(ROOT, "bench.py")).read()
    assert 'ap.add_argument("--workload", default="gdpa"' in src


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traffic_is_reported_only_while_the_kernel_sources_are_unchanged(monkeypatch):
    b = _bench_module()
    stored = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["gdpa"]["bwd_dkdv"]
    # the capture names the hash of every source the dK/dV kernel is built from: the figure
    # is reported while that hash matches the sources, and not once they have changed
    monkeypatch.setattr(b, "file_sha", lambda names: stored["source_sha"])
    assert b.measured_traffic("bwd_dkdv", "gdpa") == stored["dram_bytes_per_launch"]
    monkeypatch.setattr(b, "file_sha", lambda names: "0" * 16)
    assert b.measured_traffic("bwd_dkdv", "gdpa") is None
    monkeypatch.undo()
    h = b.file_sha(b.KERNEL_SOURCES["bwd_dkdv"])
    assert h is not None and h != b.file_sha(b.KERNEL_SOURCES["bwd_dkdv"] + ("sched.cu",))
    assert b.measured_traffic("fwd", "no_such_workload") is None
    assert b.file_sha(("no_such_file.cu",)) is None


def test_clock_summary_inside_and_around_the_window():
    b = _bench_module()
    c = b.ClockSampler(0)
    na, ac = "Not Active", "Active"
    c.stamped = [(0.9, "2070, 2070, %s, %s, %s, %s" % (na, na, na, na)),
                 (1.1, "1900, 2070, %s, %s, %s, %s" % (na, na, na, ac)),
                 (1.2, "1950, 2070, %s, %s, %s, %s" % (na, na, na, na)),
                 (1.3, "2000, 2070, %s, %s, %s, %s" % (na, na, na, na)),
                 (1.6, "2070, 2070, %s, %s, %s, %s" % (na, na, na, na))]
    c.t0, c.t1, c.source = 1.0, 1.5, "test"
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1950 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "during the timed region"
    c.t0, c.t1 = 1.31, 1.35  # shorter than the sampling period: the nearest sample each side
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == (2000 + 2070) / 2
    assert s["window"].startswith("nearest samples around")


class _Recorder:
    """Stands in for the binding: records the calls a step makes, in order."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*a, **kw):
            self.calls.append((name, kw.get("planned", False)))
        return call


def test_bench_step_is_one_plan_then_planned_calls():
    import workloads

    b = _bench_module()
    d = {n: None for n in ("q", "k", "v", "do", "oq", "ok", "o", "lse", "dq", "dk", "dv")}
    for name, plan, calls in (("gdpa", "jfa_plan", ("jfa_gdpa_fwd", "jfa_gdpa_bwd")),
                              ("d64", "jfa_plan", ("jfa_fwd", "jfa_bwd")),
                              ("cross", "jfa_plan", ("jfa_cross_fwd", "jfa_cross_bwd")),
                              ("block", "jfa_block_plan", ("jfa_block_fwd", "jfa_block_bwd")),
                              ("block_rope", "jfa_block_plan", ("jfa_block_fwd", "jfa_block_bwd"))):
        rec = _Recorder()
        b.gpu_step_fn(rec, workloads.WORKLOADS[name], d, ws=None)()
        assert rec.calls == [(plan, False), (calls[0], True), (calls[1], True)], name
    rec = _Recorder()  # the pooled calls take no plan
    b.gpu_step_fn(rec, workloads.WORKLOADS["pooled"], d, ws=None)()
    assert rec.calls == [("jfa_pooled_fwd", False), ("jfa_pooled_bwd", False)]
