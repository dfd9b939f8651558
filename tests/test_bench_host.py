"""Host logic of bench.py, on the CPU: the reference arm's JSON line, the
choice of the roofline op, and the rule that a DRAM-traffic record counts
only while its kernel source is unchanged."""
import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run(["--impl", "reference", "--config", "c1", "--steps", "1", "--warmup", "0"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == "TFLOP/s"
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["steps"] == 1 and j["warmup"] == 0 and j["n_gpus"] == 1
    assert j["higher_is_better"] is True and j["scaling"] == "weak" and j["vs_baseline"] is None
    assert j["config"]["workload"] == "c1_block_d256"
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    r = _run(["--impl", "reference", "--config", "c1", "--steps", "1", "--warmup", "0"],
             {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


PEAKS = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0, "source": "test"}


def test_roofline_takes_the_op_with_the_largest_share_against_its_own_roof(monkeypatch):
    monkeypatch.setattr(bench, "measured_traffic", lambda cfg, op: None)
    # (ms a launch, flops, bytes, launches a forward, bound)
    kern = {"gemm_gu": (0.5, 1.0e12, 1.0e8, 10, "tensor"),      # 5 ms a forward
            "attn_w0": (0.6, 4.0e11, 5.0e7, 6, "tensor"),       # 3.6 ms
            "add_norm": (0.1, 0, 6.0e8, 20, "hbm")}             # 2 ms
    r = bench.roofline_for(kern, "c5", PEAKS)
    assert r["kernel"] == "gemm_gu" and r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(2000.0) and r["frac"] == pytest.approx(1.0)
    kern["add_norm"] = (0.1, 0, 6.0e8, 60, "hbm")                # now 6 ms a forward
    r = bench.roofline_for(kern, "c5", PEAKS)
    assert r["kernel"] == "add_norm" and r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(6000.0) and r["frac"] == pytest.approx(0.75)
    assert r["algorithmic_per_launch"] == 6.0e8


def test_traffic_record_counts_only_while_its_source_is_unchanged(tmp_path, monkeypatch):
    csrc = tmp_path / "transformer_encoder_forward_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = csrc / "q8_linear.cu"
    src.write_bytes(b"// kernel v1\n")
    (tmp_path / "profiles").mkdir()
    rec = {"kernel": "k", "source": "q8_linear.cu", "dram_bytes_per_launch": 12345,
           "source_sha256": hashlib.sha256(b"// kernel v1\n").hexdigest()}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({"gemm_gu@c5": rec}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("c5", "gemm_gu") == 12345
    assert bench.measured_traffic("c2", "gemm_gu") is None           # no record for that workload
    src.write_bytes(b"// kernel v2\n")
    assert bench.measured_traffic("c5", "gemm_gu") is None           # the kernel changed since


def test_committed_traffic_records_name_their_ops_source():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        recs = json.load(f)
    n = 0
    for key, rec in recs.items():
        if key.startswith("_"):
            continue
        op, cfg = key.split("@")
        prefix = next(k for k in bench.OP_SOURCE if op.startswith(k))
        assert rec["source"] == bench.OP_SOURCE[prefix], key
        assert cfg in bench.synth.CONFIGS, key
        assert rec["dram_bytes_per_launch"] > 0 and len(rec["source_sha256"]) == 64
        n += 1
    assert n > 0
