"""bench.py's reference arm (the fp64 oracle timed on the host cores) keeps the JSON-line
contract: one line from rank 0 with the metric, unit and config of the GPU arm, a
cpu_baseline describing the run and an e2e object with no host-device bytes; ranks
other than 0 exit 0 without output."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny_stream_f32",
       "--steps", "2", "--warmup", "1"]


def _run(env_extra):
    env = dict(os.environ)
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        env.pop(k, None)
    env.update(env_extra)
    return subprocess.run(CMD, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    import bench
    r = _run({})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["config"]["workload"] == "tiny_stream_f32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_secondary_runs_report_each_workload_and_survive_a_failure(monkeypatch):
    """The default run's secondary list: one entry per (workload, variant) with the
    throughput and roofline of its run, an e2e object only where the step has one, and a
    workload that raises reported with its error instead of ending the headline line."""
    import argparse
    import bench

    seen = []

    def fake_line(sub, w, e2e=True):
        seen.append((sub.workload, sub.f32, sub.rope, sub.query_frames, sub.steps, sub.warmup,
                     sub.no_cpu_baseline, w.dtype))
        d = {"metric": "m", "value": 1.0, "unit": "u", "ms_per_step": 2.0, "steps": sub.steps,
             "warmup": sub.warmup, "dtype": w.dtype,
             "roofline": {"bound": "hbm", "achieved": 3.0, "peak": 4.0, "unit": "GB/s", "frac": 0.75,
                          "avg_launch_us": 5.0, "traffic": 7, "kernel": "k"},
             "gpu_launches": 6, "clocks": {"sm_mhz": 1.0}, "device_status": 0}
        if e2e:
            d["e2e"] = {"value": 0.9, "unit": "u", "outputs_match_device_path": True}
        return d

    def fake_gpu(sub, w):
        if sub.workload == "high_res_999":
            raise RuntimeError("out of memory")
        return fake_line(sub, w)

    monkeypatch.setattr(bench, "run_gpu", fake_gpu)
    monkeypatch.setattr(bench, "run_prefill", lambda sub, w: fake_line(sub, w, e2e=False))
    args = argparse.Namespace(workload="steady_state_10k", steps=100, warmup=5, no_cpu_baseline=False,
                              rope=False, f32=False, query_frames=1, splits=0, blocks=0, no_secondary=False)
    out = bench.run_secondary(args)
    assert [(e["workload"], e["variant"]) for e in out] == [(n, v) for n, v, _ in bench.SECONDARY]
    by = {(e["workload"], e["variant"]): e for e in out}
    assert by[("high_res_999", "")]["error"] == "RuntimeError: out of memory"
    assert by[("lingbot_like_200", "f32")]["dtype"] == "f32"
    assert "e2e" not in by[("steady_state_10k", "prefill8")]
    assert by[("batched4_d128", "")]["roofline"] == {"bound": "hbm", "achieved": 3.0, "peak": 4.0, "unit": "GB/s",
                                                      "frac": 0.75, "avg_launch_us": 5.0}
    assert by[("batched4_d128", "")]["e2e"] == {"value": 0.9, "outputs_match_device_path": True}
    # every secondary run skips the oracle baseline and uses its own step counts
    assert all(s[6] for s in seen)
    assert ("lingbot_like_200", True, False, 1, 5, 3, True, "f32") in seen
    assert ("steady_state_10k", False, False, 8, 20, 5, True, "bf16") in seen
    assert ("steady_state_10k", False, True, 1, 20, 5, True, "bf16") in seen
    assert args.workload == "steady_state_10k" and args.steps == 100  # the headline args are untouched
