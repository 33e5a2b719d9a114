"""Host-side logic of bench.py (CPU only).

* DRAM traffic from the committed ncu capture is reported only while the kernel sources
  still hash the same; any change makes it null.
* The reference arm (`--impl reference`) prints one JSON line with the contract's keys,
  timing the oracle on the host cores.
* The FLOP convention: 4*B*H*Nq*Nk*D for the forward, halved when causal; backward 2.5x.
"""
import json
import os
import subprocess
import sys

import pytest

import bench
from tiled_attention_11_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_is_null_once_a_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    record = {"demo": {"dram_bytes_per_launch": 1234, "source_sha": bench.sources_sha(["k.cu"])}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(record))
    assert bench.traffic_for("demo", ["k.cu"]) == 1234.0
    assert bench.traffic_for("other", ["k.cu"]) is None
    src.write_text("kernel v2\n")
    assert bench.traffic_for("demo", ["k.cu"]) is None


def test_flop_convention():
    p = I.Problem(2, 3, 100, 70, 64, False)
    assert I.flops_fwd(p) == 4.0 * 2 * 3 * 100 * 70 * 64
    assert I.flops_fwd(I.Problem(2, 3, 100, 70, 64, True)) == I.flops_fwd(p) / 2
    assert I.flops_bwd(p) == 2.5 * I.flops_fwd(p)
    assert I.flops_fwd(I.LAYER) == pytest.approx(5.4976e11, rel=1e-4)


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["warmup"] >= 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert isinstance(line["cpu_baseline"]["cpu_model"], str) and line["cpu_baseline"]["cpu_model"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("multi-head LLM-shaped attention layer")


def test_reference_arm_prints_on_rank_zero_only():
    # under torchrun every rank runs the arm; ranks other than 0 exit 0 without work or output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
