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
                   "bytes_per_launch": 123, "workload": "w-big, 976 valid rows"}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    b.ROOT = str(tmp_path)
    assert b.traffic_record("k_x", "w-big")["bytes_per_launch"] == 123
    assert b.traffic_record("k_x", "w-small") is None       # captured on another workload
    assert b.traffic_record("k_other", "w-big") is None
    (csrc / "k.cu").write_text("kernel v2\n")                 # the kernel changed since the capture
    assert b.traffic_record("k_x", "w-big") is None
    (csrc / "k.cu").unlink()
    assert b.traffic_record("k_x", "w-big") is None


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


@pytest.mark.parametrize("wid,sigma", [(0, 0.75), (4, None)])
def test_winner_slot_and_retrieval_hits(wid, sigma):
    """The bench recovers each request's deepest accepted node from the
    step's outputs alone; on oracle-verified trees of a closed loop it equals
    the winner found by brute force from the rows' argmaxes (deepest accepted
    node, lower slot on ties), and retrieved winners occur."""
    import numpy as np

    import oracle
    import workloads as W
    b_ = _bench()
    kw = {} if sigma is None else {"draft_sigma": sigma}
    w = W.WORKLOADS[wid].scaled(V=400, B=2, **kw)
    h = W.Harness(w)
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode)
    C = oracle.new_matrix(w.V)
    root, prev, ctx = h.init_state()
    hits_seen = 0
    for step in range(25):
        tok, par, aux = h.draft(step, root, prev)
        trees = [oracle.assemble(P, root[b], tok[b], aux[b], C, None if par is None else par[b]) for b in range(w.B)]
        tt = np.stack([t.tok for t in trees])
        pp = np.stack([t.par for t in trees]).astype(np.int8)
        lg = h.tree_logits(tt, pp, ctx, prev)
        accs, outs = [], []
        for b in range(w.B):
            acc, out, topk = oracle.verify(trees[b], lg[b], w.dtype)
            y = topk[:, 0]
            best_d, best_i = 0, 0
            for i in range(1, w.S):
                if tt[b][i] < 0:
                    continue
                ok, d, j = True, 0, i
                while j != 0:
                    p = int(pp[b][j])
                    ok &= bool(tt[b][j] == y[p])
                    d += 1
                    j = p
                if ok and d > best_d:
                    best_d, best_i = d, i
            assert best_d == acc
            assert b_.winner_slot(tt[b], pp[b], acc, out) == best_i, (step, b)
            oracle.update(C, trees[b], topk)
            accs.append(acc)
            outs.append(out)
        acc_a, out_a = np.array(accs, np.int32), np.stack(outs)
        # slot provenance of checkpoint / tail trees: the kept draft slots follow
        # the root, the retrieved ones follow them (info[1] kept draft slots)
        src = np.where(tt >= 0, 1, -1).astype(np.int8)
        src[:, 0] = np.where(tt[:, 0] >= 0, 0, -1)
        for b in range(w.B):
            r0 = 1 + int(trees[b].info[1])
            src[b, r0:][tt[b, r0:] >= 0] = 2
        hits = b_.retrieval_hits(src, tt, pp, acc_a, out_a)
        assert all(hv in (0, 1) for hv in hits)
        for b in range(w.B):
            wsl = b_.winner_slot(tt[b], pp[b], acc_a[b], out_a[b])
            assert hits[b] == int(acc_a[b] > 0 and wsl >= 1 + int(trees[b].info[1]))
        hits_seen += sum(hits)
        h.advance(root, prev, ctx, out_a, acc_a)
    assert hits_seen > 0


def test_hit_rate_and_populated_rows():
    import numpy as np
    b_ = _bench()
    assert b_.hit_rate_of([[0, 1], [1, 1]]) == 0.75
    assert b_.hit_rate_of([[0, 1], None]) is None and b_.hit_rate_of([]) is None
    C = np.full((5, 8), -1, np.int32)
    C[[1, 3], :] = 7
    assert b_.populated_rows(C) == 2


def test_prune_histogram_and_cpu_baseline_entry():
    """The prune-depth histogram counts each request-step's info[0] (fired
    checkpoint layer, or the kept block prefix in tail mode; none in static
    mode), and the CPU-baseline object reports the all-cores figure with the
    one-core figure beside it."""
    import numpy as np

    import workloads as W
    b_ = _bench()
    infos = [np.array([[-1, 60, 0, 61], [1, 24, 30, 55]], np.int32), np.array([[-1, 60, 0, 61], [5, 40, 12, 53]])]
    h = b_.prune_histogram(W.MODE_CHECKPOINT, infos)
    assert h == {"key": "fired_layer", "counts": {"-1": 2, "1": 1, "5": 1}}
    assert b_.prune_histogram(W.MODE_TAIL, infos)["key"] == "kept_prefix"
    assert b_.prune_histogram(W.MODE_STATIC, infos) is None
    det = {"steps": 4, "requests": 16, "threads": 8, "one_core": 2.0, "all_cores": 12.5, "one_core_s": 2.0,
           "all_cores_s": 0.32, "warm_s": None, "warm_rows": 0}
    e = b_.cpu_baseline_entry(det, W.WORKLOADS[2])
    assert e["value"] == 12.5 and e["cores"] == 8 and e["kind"] == "oracle"
    assert e["one_core"] == {"value": 2.0, "unit": "steps/s", "cores": 1, "timed_s": 2.0}
    assert "warm_start" not in e
    det.update(warm_s=1.25, warm_rows=1280)
    assert b_.cpu_baseline_entry(det, W.WORKLOADS[1])["warm_start"]["rows"] == 1280
