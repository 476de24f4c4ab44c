"""Host-side logic of the benchmark, on the CPU: the roofline's traffic
record is used only while the kernel's source is unchanged, the peak comes
from the measured file when present, and both arms describe the workload
with the same config object; the oracle arm's launch at N = 2."""
import hashlib
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traffic_record_follows_the_kernel_source(tmp_path):
    b = _bench()
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "hybrid_draft_tree_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1\n")
    rec = {"k_x": {"source": "k.cu", "source_sha256": hashlib.sha256(b"kernel v1\n").hexdigest(),
                   "bytes_per_launch": 123}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    b.ROOT = str(tmp_path)
    assert b.traffic_record("k_x")["bytes_per_launch"] == 123
    assert b.traffic_record("k_other") is None
    (csrc / "k.cu").write_text("kernel v2\n")                 # the kernel changed since the capture
    assert b.traffic_record("k_x") is None
    (csrc / "k.cu").unlink()
    assert b.traffic_record("k_x") is None


def test_peak_prefers_the_measured_file(tmp_path):
    b = _bench()
    b.ROOT = str(tmp_path)
    assert b.measured_peak_gbs() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6763.6}))
    assert b.measured_peak_gbs() == (6763.6, "measured")


def test_both_arms_share_the_workload_config():
    import workloads as W
    b = _bench()
    w = W.WORKLOADS[2]
    cfg = b.workload_config(w, 1)
    assert cfg["workload"] == w.name and cfg["vocab"] == 151936 and cfg["batch"] == 16
    assert cfg["slots_per_request"] == 61 and cfg["logits_bytes_per_step"] == 16 * 61 * 151936 * 2
    assert b.workload_config(w, 4)["parallelism"] == "replicas"


def test_reference_arm_under_torchrun_world_size_2():
    """The oracle arm launched like the GPU arm at N = 2 (torchrun, gloo on
    the host): rank 0 alone prints one JSON line, every rank exits 0."""
    import socket
    import subprocess
    import sys
    pytest.importorskip("torch")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
                        "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["steps"] == 1
    assert out["value"] > 0 and out["cpu_baseline"]["kind"] == "oracle"
    assert out["cpu_baseline"]["value"] == out["value"] == out["e2e"]["value"]
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["d2h_bytes_per_step"] == 0
