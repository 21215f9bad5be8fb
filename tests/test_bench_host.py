"""CPU checks of bench.py's host-side contract (no GPU): argument rules, the
reference arm's rank handling, the traffic lookup keyed by the kernel sources,
and the end-to-end arm's host copies of product operands."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def run_bench(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_warmup_below_three_is_refused():
    r = run_bench(["--warmup", "1", "--steps", "1"])
    assert r.returncode == 2 and "--warmup must be >= 3" in r.stderr


def test_reference_arm_runs_on_rank_zero_only():
    r = run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3"], env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_on_a_small_workload():
    r = run_bench(["--impl", "reference", "--workload", "nvfp4_gemv_1x256x256", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    # the same configuration object as this arm's line
    assert line["config"] == bench.workload_config("nvfp4_gemv_1x256x256", 32)


def test_default_workload_is_the_largest_configuration():
    """The headline line is the nvfp4 prefill GEMM 8192^3 (the largest
    single-GPU configuration); the others are reported under 'configs'."""
    assert bench.HEADLINE == "nvfp4_prefill_gemm_8192" == bench.WORKLOADS[0]
    from block_scaled_precision_packed_gb300 import synthetic as S
    flops = {w: 2 * S.WORKLOADS[w]["M"] * S.WORKLOADS[w]["N"] * S.WORKLOADS[w]["K"]
             for w in S.WORKLOADS if "M" in S.WORKLOADS[w]}
    assert max(flops, key=flops.get) == bench.HEADLINE


def test_oracle_sample_one_core_and_all_cores_share_the_product():
    """The cpu_baseline legs and the reference arm time the same product on
    the oracle's own quantization of the workload's inputs; the all-core sample
    is the larger one."""
    one = bench.OracleSample("nvfp4_gemv_1x256x256", 1)
    every = bench.OracleSample("nvfp4_gemv_1x256x256", 0)
    assert one.desc == every.desc and one.step_seconds() > 0 and every.step_seconds() > 0
    assert bench.ORACLE_SAMPLE[0][0] * bench.ORACLE_SAMPLE[0][1] > bench.ORACLE_SAMPLE[1][0] * bench.ORACLE_SAMPLE[1][1]


def test_traffic_counts_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    entries = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    key = next(k for k in entries if not k.startswith("_"))
    kernel, workload = key.split("@")[:2]
    m = int(key.split("@M")[1]) if "@M" in key else None
    sha = bench.src_sha()
    monkeypatch.setattr(bench, "src_sha", lambda: entries[key]["src_sha"])
    assert bench.traffic_for(kernel, workload, m) == entries[key]["bytes_per_launch"]
    monkeypatch.setattr(bench, "src_sha", lambda: "0" * 16 if sha != "0" * 16 else "1" * 16)
    assert bench.traffic_for(kernel, workload, m) is None


def test_operand_host_copies_are_raw_bytes():
    torch = pytest.importorskip("torch")

    class W:
        pass
    w = W()
    w.codes = torch.arange(12, dtype=torch.int32).reshape(3, 4)
    w.scale = torch.tensor([0.25], dtype=torch.float32)
    out = bench.operand_host_copies(w, ("codes", "scale"))
    assert out["codes"].dtype == np.uint8 and out["codes"].size == 48
    assert np.array_equal(out["codes"].view(np.int32), np.arange(12, dtype=np.int32))
    assert out["scale"].view(np.float32)[0] == np.float32(0.25)
