"""Benchmark of the Graft hot path on GB300.

One step = graft_assemble + graft_verify_update (checkpoint / static / tail
selection, template retrieval, flattening, greedy verification, online top-8
update) for one batch, on the synthetic static-tree workload at batch 16,
V = 151936, bf16 logits [16, 61, 151936] (296.6 MB per step).

Timed region: CUDA events on the library's stream around the two graft calls
of each step; the synthetic target's logits are generated between them
(untimed) and L2 is flushed (256 MB write) before each graft call, so the
logits are read from HBM.  ``e2e`` repeats the step through the C ABI from
pinned HOST buffers (draft inputs and logits copied in, accept lengths and
emitted tokens copied out) inside the timed region.

``--impl reference`` times the CPU oracle (plain C, one thread) on a bounded
sample of the same workload.  With several GPUs (torchrun) every rank runs an
independent replica.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "Graft steps/s (assemble+verify+update) and logits HBM GB/s vs GB300 peak"
UNIT = "steps/s"
L2_FLUSH_BYTES = 256 << 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["graft", "reference"], default="graft")
    p.add_argument("--workload", type=int, default=2, help="synthetic workload id (0-4); 2 is the headline")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time budget for cpu_baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--scan-kernel", type=int, default=0, help="verify scan (graft_config.scan_kernel); 0 = automatic")
    p.add_argument("--next-rows", action="store_true",
                   help="also time the stochastic step and the confidence / coverage calls (JSON key next_rows)")
    p.add_argument("--sample-temperature", type=float, default=1.0)
    p.add_argument("--no-workloads", action="store_true", help="skip the other workloads and the warm start")
    p.add_argument("--oracle-warm", action="store_true", help="reference arm: also time the oracle's warm-up load")
    p.add_argument("--workload-steps", type=int, default=60, help="timed steps of each other workload")
    p.add_argument("--draft-sigma", type=float, default=None,
                   help="sibling-logit scale of the synthetic drafter (default: the workload's)")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


# --------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(w: W.Workload, budget_s: float, max_steps: int | None = None, threads: int | None = None,
                  warm: bool = False):
    """Closed-loop oracle decode of the whole batch.  Per step: the oracle
    assembles every request (one thread), verifies every request on one
    thread, verifies them again over a pool of `threads` threads
    (independent requests; the C calls release the GIL; the results must
    agree), then applies the updates in (request, slot) order on one thread.
    The synthetic logits are generated outside the timed parts (host
    generator, all threads).  Runs until the one-thread time reaches
    `budget_s`, or for `max_steps` steps.  With `warm`, the workload's warm-up
    rows are first loaded in order by the oracle (one thread; rows generated
    in chunks outside the timed part).  Returns a dict with both rates."""
    import concurrent.futures as cf

    import oracle
    threads = threads or W.host_threads()
    h = W.Harness(w)
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode)
    C = oracle.new_matrix(w.V)
    root, prev, ctx = h.init_state()
    oracle.lib()
    warm_s, warm_rows = None, 0
    if warm and w.warm != "none":
        toks, rk, pl, bi = h.warm_rowparams()
        warm_s, warm_rows = 0.0, len(toks)
        for r0 in range(0, warm_rows, 2048):
            r1 = min(warm_rows, r0 + 2048)
            rows = W.fill_rows(rk[r0:r1], pl[r0:r1], bi[r0:r1], w.V, w.dtype, threads=threads)
            t0 = time.perf_counter()
            oracle.warmup(C, toks[r0:r1], rows, w.dtype)
            warm_s += time.perf_counter() - t0
    t_asm = t_one = t_all = t_upd = 0.0
    steps = 0
    pool = cf.ThreadPoolExecutor(threads)
    try:
        while (max_steps is None and t_asm + t_one + t_upd < budget_s) or (max_steps is not None and steps < max_steps):
            tok, par, aux = h.draft(steps, root, prev)
            t0 = time.perf_counter()
            trees = [oracle.assemble(P, root[b], tok[b], aux[b], C, None if par is None else par[b])
                     for b in range(w.B)]
            t_asm += time.perf_counter() - t0
            lg = h.tree_logits(np.stack([t.tok for t in trees]), np.stack([t.par for t in trees]).astype(np.int8),
                               ctx, prev, threads=threads)
            t0 = time.perf_counter()
            one = [oracle.verify(trees[b], lg[b], w.dtype) for b in range(w.B)]
            t_one += time.perf_counter() - t0
            t0 = time.perf_counter()
            res = list(pool.map(lambda b: oracle.verify(trees[b], lg[b], w.dtype), range(w.B)))
            t_all += time.perf_counter() - t0
            for (a1, o1, k1), (a2, o2, k2) in zip(one, res):
                if a1 != a2 or not np.array_equal(o1, o2) or not np.array_equal(k1, k2):
                    raise RuntimeError("oracle results differ between one thread and the pool")
            t0 = time.perf_counter()
            for b in range(w.B):
                oracle.update(C, trees[b], res[b][2])
            t_upd += time.perf_counter() - t0
            h.advance(root, prev, ctx, np.stack([r[1] for r in res]), np.array([r[0] for r in res], np.int32))
            steps += 1
    finally:
        pool.shutdown()
    return {"steps": steps, "requests": w.B, "threads": threads, "warm_s": warm_s, "warm_rows": warm_rows,
            "one_core": steps / (t_asm + t_one + t_upd), "all_cores": steps / (t_asm + t_all + t_upd),
            "one_core_s": t_asm + t_one + t_upd, "all_cores_s": t_asm + t_all + t_upd}


def cpu_baseline_entry(det, w):
    """The `cpu_baseline` object: the oracle over all host cores (value,
    cores) with its one-core figure beside it."""
    sample = (f"{det['steps']} closed-loop oracle steps of the full batch ({det['requests']} requests): assemble and "
              f"update on one thread, verification over {det['threads']} threads (one request per task) and again "
              f"on one thread; logits generation excluded")
    return {"value": round(det["all_cores"], 5), "unit": UNIT, "cores": det["threads"], "kind": "oracle",
            "sample": sample, "cpu": cpu_model(), "timed_s": round(det["all_cores_s"], 3),
            "one_core": {"value": round(det["one_core"], 5), "unit": UNIT, "cores": 1,
                         "timed_s": round(det["one_core_s"], 3)},
            "note": "one request per pool task, so the pool uses at most min(cores, batch) threads at once"
            if w.B < det["threads"] else "one request per pool task",
            **({"warm_start": {"rows": det["warm_rows"], "s": round(det["warm_s"], 3), "cores": 1,
                               "note": "the oracle's in-order load of every warm-up row (one thread)"}}
               if det.get("warm_s") is not None else {})}


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        # raw samples go to $GRAFT_CLOCKS_DIR (kept) or the temp directory
        d = os.environ.get("GRAFT_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(sms)}


# --------------------------------------------------------------------------- GPU arm
def measured_peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_record(kernel, workload):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, valid
    only for the workload it was captured on (the name before the record's
    first comma) and while that kernel's source file is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("workload", "").split(",")[0].strip() != workload:
        return None
    path = os.path.join(ROOT, "hybrid_draft_tree_gb300", "csrc", rec["source"])
    if not os.path.exists(path):
        return None
    with open(path, "rb") as f:
        src = f.read()
    if rec.get("source_sha256") != hashlib.sha256(src).hexdigest():
        return None
    return rec


def workload_config(w, ws):
    """The `config` object of both arms' JSON lines: what the workload is."""
    return {"workload": w.name, "vocab": w.V, "batch": w.B, "slots_per_request": w.S, "draft_sigma": w.draft_sigma,
            "mode": ["checkpoint", "static", "tail"][w.mode], "logits_bytes_per_step": w.logits_bytes_per_step(),
            "parallelism": "replicas" if ws > 1 else "single",
            "l2_between_steps": "flushed before each graft call (256 MB written, then read back)"}


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def winner_slot(tok, par, accept_len, out_tokens) -> int:
    """Slot of a request's deepest accepted node, recovered from the step's
    outputs: the lowest slot at depth accept_len whose root path carries the
    emitted tokens (verification breaks depth ties toward the lower slot).
    Parents precede children in the flattened tree.  -1 for an empty tree."""
    S = len(tok)
    if S == 0 or tok[0] < 0:
        return -1
    depth = np.full(S, -1, np.int64)
    depth[0] = 0
    for i in range(1, S):
        p = int(par[i])
        if tok[i] < 0 or p < 0 or p >= i or depth[p] < 0:
            continue
        d = depth[p] + 1
        if d <= accept_len and tok[i] == out_tokens[d - 1]:
            depth[i] = d
    hits = np.flatnonzero(depth == accept_len)
    return int(hits[0]) if len(hits) else -1


def retrieval_hits(src, tok, par, accept_len, out_tokens):
    """Per request: 1 when the deepest accepted node came from the matrix
    (slot provenance 2, as graft_assemble_src reports it: a retrieval node,
    or an in-place replacement in static mode), else 0."""
    hits = []
    for b in range(len(accept_len)):
        ws_ = winner_slot(tok[b], par[b], int(accept_len[b]), out_tokens[b])
        hits.append(int(accept_len[b] > 0 and ws_ >= 0 and src[b][ws_] == 2))
    return hits


def hit_rate_of(hits):
    """Mean of the per-step retrieval hits (lists of 0/1 per request); None
    when any step has none (static mode, or a statistic that failed)."""
    if not hits or any(h is None for h in hits):
        return None
    return float(np.mean(np.concatenate([np.asarray(h, np.float64) for h in hits])))


def populated_rows(matrix) -> int:
    """Rows of the continuation matrix that hold at least one successor."""
    return int((np.asarray(matrix)[:, 0] >= 0).sum())


def make_flush(dev):
    """L2 flush on the current stream: write a buffer larger than L2, then
    read it back, so L2 ends up holding clean lines and the next kernel pays
    no write-backs of the flush."""
    import torch
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    sink = torch.empty(1, dtype=torch.int32, device=dev)

    def flush_l2():
        flush.zero_()
        torch.amax(flush, dim=0, keepdim=True, out=sink)
    return flush_l2


def make_engine(w, scan_kernel=0):
    import hybrid_draft_tree_gb300 as g
    return g.Graft(g.graft_default_config(w.V, w.B, w.mode, w.dtype, budget=w.budget, max_draft_nodes=w.draft_nodes,
                                          scan_kernel=scan_kernel))


class DecodeTimer:
    """Timed decode steps of one workload: per step, L2 flushed, then
    graft_assemble between CUDA events; the target's logits (untimed); L2
    flushed, then graft_verify_update between events.  With tracing on, the
    library's per-kernel event pairs are collected instead."""

    def __init__(self, w, eng, loop, stream, flush_l2):
        self.w, self.eng, self.loop, self.stream, self.flush_l2 = w, eng, loop, stream, flush_l2
        self.kernel_ms = {}

    def step(self, ev=None, tracing=False):
        import torch
        loop, eng, stream = self.loop, self.eng, self.stream
        loop.draft()
        with torch.cuda.stream(stream):
            self.flush_l2()
        if ev:
            ev[0].record(stream)
        loop.assemble()
        n = eng.last_launch_count()
        if ev:
            ev[1].record(stream)
        loop.make_logits()
        with torch.cuda.stream(stream):
            self.flush_l2()
        if ev:
            ev[2].record(stream)
        loop.verify_update()
        n += eng.last_launch_count()
        if ev:
            ev[3].record(stream)
        loop.advance(read_back=False)
        stream.synchronize()                             # the next draft needs the state
        valid = int((loop.tok >= 0).sum().item())
        acc = loop.accept_len.cpu().numpy()
        info = loop.info.cpu().numpy()
        try:
            hit = retrieval_hits(loop.src.cpu().numpy(), loop.tok.cpu().numpy(), loop.par.cpu().numpy(), acc,
                                 loop.out_tokens.cpu().numpy())
        except Exception:                                # a statistic only: never costs the measurement
            hit = None
        loop.pull_state()
        if tracing:
            for name, ms in eng.profile_read():
                self.kernel_ms.setdefault(name, []).append(ms)
        return n, valid, acc, info, hit

    def run(self, steps, tracing=False):
        """`steps` timed steps; returns their records and event pairs."""
        import torch
        if tracing:
            self.eng.profile_enable(True)
            self.eng.profile_read()
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        recs = [self.step(events[k], tracing) for k in range(steps)]
        torch.cuda.synchronize()
        if tracing:
            self.eng.profile_enable(False)
        t_asm = [e[0].elapsed_time(e[1]) for e in events]
        t_ver = [e[2].elapsed_time(e[3]) for e in events]
        return recs, t_asm, t_ver


def run_graft(args, ws, rank, local):
    import torch
    from hybrid_draft_tree_gb300 import _build
    from workloads.device_loop import DeviceLoop

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        _build.build()  # a no-op when the library is current; one rank only, so no two compile the same objects
    if ws > 1:
        torch.distributed.barrier()
    w = W.WORKLOADS[args.workload]
    if args.draft_sigma is not None:
        w = w.scaled(draft_sigma=args.draft_sigma)
    if rank:
        w = w.scaled(seed=w.seed + 1000 * rank)
    eng = make_engine(w, args.scan_kernel)
    stream = torch.cuda.Stream(dev)
    loop = DeviceLoop(w, eng, device=dev, stream=stream, track_src=True)
    flush_l2 = make_flush(dev)
    if w.warm != "none":
        toks_d, logits_d, _ = loop.warm_inputs_device()
        eng.warmup(toks_d, logits_d, stream=stream)
        stream.synchronize()
        del logits_d, toks_d
        torch.cuda.empty_cache()

    timer = DecodeTimer(w, eng, loop, stream, flush_l2)
    for _ in range(args.warmup):
        timer.step()
    clocks = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.perf_counter()
    recs, t_asm, t_ver = timer.run(args.steps)
    wall = time.perf_counter() - wall0
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    launches = sum(r[0] for r in recs)
    valid_rows = [r[1] for r in recs]
    accs = [r[2] for r in recs]
    hits = [r[4] for r in recs]
    # a second timed region of the same length with kernel tracing on (event
    # pairs around every kernel), for the per-kernel durations; the headline
    # value above is taken without the tracing events
    timer.run(args.steps, tracing=True)
    kernel_ms = timer.kernel_ms
    total_ms = max_over_ranks(sum(t_asm) + sum(t_ver), dev)
    value = ws * args.steps / (total_ms / 1e3)

    # roofline of the dominant kernel (largest share of the timed kernel time):
    # algorithmic bytes = the logits rows it streams (valid rows x V x element size)
    esize = w.esize
    algo_bytes = statistics.mean([v * w.V * esize for v in valid_rows])
    kern = {k: statistics.mean(v) for k, v in kernel_ms.items()}
    dominant = max(kernel_ms, key=lambda k: sum(kernel_ms[k]))
    dom_s = kern[dominant] / 1e3
    achieved = algo_bytes / dom_s / 1e9
    peak, peak_kind = measured_peak_gbs()
    tr = traffic_record(dominant, w.name)
    mat = float(np.mean(np.concatenate(accs))) + 1.0

    # incremental drafting (checkpoint mode): the critical-path assembly when
    # the checkpoints are evaluated as the layers are drafted and the
    # retrieval is gathered beside the drafter
    incremental = run_incremental(w, eng, loop, stream, flush_l2) if w.mode == W.MODE_CHECKPOINT else None
    next_rows = run_next_rows(args, w, eng, loop, stream, flush_l2) if args.next_rows else None

    # e2e through the C ABI from pinned host buffers
    e2e = run_e2e(args, w, eng, loop, stream, dev)

    # the continuation matrix's populated rows (the pages quote its size as the
    # bytes of the rows that hold successors) and the retrieval hit rate
    try:
        populated = populated_rows(eng.get_matrix(stream=stream))
    except Exception:
        populated = None
    try:
        hit_rate = hit_rate_of(hits)
    except Exception:
        hit_rate = None

    out = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == W.BF16 else "f32",
        "data": "synthetic",
        "config": workload_config(w, ws),
        "timing": {"l2": "flushed before each graft call (256 MB written, then read back); logits "
                         f"{w.logits_bytes_per_step() / 1e6:.1f} MB per step",
                   "timed": "assemble + verify_update per step (CUDA events on the library stream)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": tr["bytes_per_launch"] if tr else None,
                     "peak_source": f"{peak_kind} hbm_gbs (of measured)", "kernel": dominant,
                     "algorithmic_bytes_per_launch": round(algo_bytes),
                     "ms_per_launch": round(kern[dominant], 5),
                     "verify_update_GBps": round(algo_bytes / (statistics.mean(t_ver) / 1e3) / 1e9, 1),
                     "step_GBps": round(algo_bytes / (total_ms / args.steps / 1e3) / 1e9, 1),
                     "step_frac": round(algo_bytes / (total_ms / args.steps / 1e3) / 1e9 / peak, 4)},
        "kernels_us": {k: round(v * 1e3, 2) for k, v in sorted(kern.items())},
        "kernels_note": "per-kernel CUDA-event durations from a second timed region with kernel tracing on",
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches,
        "breakdown_ms": {"assemble": round(statistics.mean(t_asm), 5), "verify_update": round(statistics.mean(t_ver), 5)},
        "incremental": incremental,
        "next_rows": next_rows,
        "stats": {"mean_accepted_tokens_per_step": round(mat, 4), "valid_rows_per_step": statistics.mean(valid_rows),
                  "retrieval_hit_rate": None if hit_rate is None else round(hit_rate, 4),
                  "retrieval_hit_note": "share of request-steps whose deepest accepted node came from the matrix "
                                        "(slot provenance from graft_assemble_src; in static mode an in-place "
                                        "replacement)",
                  "prune_depth_histogram": prune_histogram(w.mode, [r[3] for r in recs]),
                  "matrix_populated_rows": populated,
                  "matrix_populated_bytes": None if populated is None else populated * 32,
                  "wall_s": round(wall, 2)},
    }
    if ws == 1 and not args.no_workloads:
        # the other synthetic workloads and the warm start, each on a fresh
        # handle (the headline's handle is released first)
        eng.close()
        del loop, timer
        torch.cuda.empty_cache()
        out["workloads"] = {}
        for wid in (0, 1, 3, 4):
            if wid == args.workload:
                continue
            out["workloads"][str(wid)] = run_other_workload(wid, dev, args.workload_steps, flush_l2, peak)
            torch.cuda.empty_cache()
    return out


def prune_histogram(mode, infos):
    """How often each checkpoint fired (info[b][0]: -1 none, else the draft
    layer), over all request-steps; in tail mode the kept block prefix length."""
    ev = np.concatenate([np.asarray(i)[:, 0] for i in infos]) if infos else np.zeros(0, np.int32)
    if mode == W.MODE_STATIC:
        return None
    keys, counts = np.unique(ev, return_counts=True)
    name = "kept_prefix" if mode == W.MODE_TAIL else "fired_layer"
    return {"key": name, "counts": {str(int(k)): int(c) for k, c in zip(keys, counts)}}


def run_other_workload(wid, dev, steps, flush_l2, peak, warm_reps=3):
    """One of the other synthetic workloads at its stated size: its warm-up
    (timed, with the matrix's populated rows right after it), then `steps`
    timed decode steps and as many traced ones."""
    import torch
    from workloads.device_loop import DeviceLoop
    w = W.WORKLOADS[wid]
    eng = make_engine(w)
    stream = torch.cuda.Stream(dev)
    loop = DeviceLoop(w, eng, device=dev, stream=stream, track_src=True)
    res = {"workload": w.name, "vocab": w.V, "batch": w.B, "slots_per_request": w.S,
           "mode": ["checkpoint", "static", "tail"][w.mode], "dtype": "bf16" if w.dtype == W.BF16 else "f32"}
    if w.warm != "none":
        toks_d, logits_d, (toks, _, _, _) = loop.warm_inputs_device()
        stream.synchronize()
        distinct = len(set(toks.tolist()))
        algo = distinct * w.V * w.esize
        times, kern = [], {}
        for r in range(warm_reps):
            if r == 1:
                populated = populated_rows(eng.get_matrix(stream=stream))
            eng.profile_enable(r == warm_reps - 1)
            eng.profile_read()
            with torch.cuda.stream(stream):
                flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            eng.warmup(toks_d, logits_d, stream=stream)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
            for name, ms in eng.profile_read():
                kern[name] = ms
        eng.profile_enable(False)
        ms = statistics.mean(times[1:]) if len(times) > 1 else times[0]
        res["warm_start"] = {
            "rows": len(toks), "distinct_rows": distinct, "naive_bytes": len(toks) * w.V * w.esize,
            "algorithmic_bytes": algo, "ms": round(ms, 4), "GBps": round(algo / (ms / 1e3) / 1e9, 1),
            "frac": round(algo / (ms / 1e3) / 1e9 / peak, 4), "calls_timed": len(times) - 1,
            "matrix_populated_rows": populated, "matrix_populated_bytes": populated * 32,
            "note": "graft_warmup (mark last occurrences, list them, top-8 of those rows, reset), CUDA events, L2 "
                    "flushed before each call; algorithmic bytes = distinct last-occurrence rows x V x element size"}
        del logits_d, toks_d
        torch.cuda.empty_cache()
    timer = DecodeTimer(w, eng, loop, stream, flush_l2)
    for _ in range(5):
        timer.step()
    recs, t_asm, t_ver = timer.run(steps)
    timer.run(steps, tracing=True)
    step_ms = statistics.mean(t_asm) + statistics.mean(t_ver)
    algo = statistics.mean([r[1] * w.V * w.esize for r in recs])
    kern = {k: statistics.mean(v) for k, v in timer.kernel_ms.items()}
    # the kernel that reads the logits: pass 1 of the two-pass scan, or the
    # cluster-per-row verify (small steps)
    scan_k = next((k for k in ("k_umax", "k_cluster_select") if k in kern), None)
    scan_ms = kern.get(scan_k) if scan_k else None
    try:
        hit_rate = hit_rate_of([r[4] for r in recs])
    except Exception:
        hit_rate = None
    res.update({
        "steps": steps, "steps_per_s": round(1e3 / step_ms, 1), "ms_per_step": round(step_ms, 5),
        "breakdown_ms": {"assemble": round(statistics.mean(t_asm), 5), "verify_update": round(statistics.mean(t_ver), 5)},
        "logits_bytes_per_step": round(algo), "step_GBps": round(algo / (step_ms / 1e3) / 1e9, 1),
        "scan_kernel": scan_k,
        "scan_GBps": round(algo / (scan_ms / 1e3) / 1e9, 1) if scan_ms else None,
        "scan_frac": round(algo / (scan_ms / 1e3) / 1e9 / peak, 4) if scan_ms else None,
        "kernels_us": {k: round(v * 1e3, 2) for k, v in sorted(kern.items())},
        "mean_accepted_tokens_per_step": round(float(np.mean(np.concatenate([r[2] for r in recs]))) + 1.0, 4),
        "prune_depth_histogram": prune_histogram(w.mode, [r[3] for r in recs]),
        "retrieval_hit_rate": None if hit_rate is None else round(hit_rate, 4),
    })
    eng.close()
    return res


def run_next_rows(args, w, eng, loop, stream, flush_l2, steps=50):
    """Timings of the calls beyond the greedy step, on this workload: the
    stochastic step (assemble + verify_update_sample, events around the two
    calls, L2 flushed before each) with its per-kernel times, and the traced
    kernels of the confidence (tree modes) and coverage (checkpoint and tail
    modes) calls."""
    import torch
    dev = stream.device
    B, S = w.B, w.S
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    u = torch.empty((B, S), dtype=torch.float32, device=dev)
    ur = torch.empty((B,), dtype=torch.float32, device=dev)
    best = torch.empty((B, 3), dtype=torch.float32, device=dev)
    gain = torch.empty((B,), dtype=torch.float32, device=dev)
    temp = args.sample_temperature
    ms_asm, ms_ver, acc = [], [], []
    kern = {}
    for k in range(steps + 3):
        trace = k >= 3 and k % 2 == 1                   # alternate traced and untimed-by-events steps
        eng.profile_enable(trace)
        eng.profile_read()
        loop.draft()
        with torch.cuda.stream(stream):
            u.uniform_(generator=gen)
            ur.uniform_(generator=gen)
            flush_l2()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        loop.assemble()
        e[1].record(stream)
        if w.mode != W.MODE_TAIL:
            eng.confidence(B, loop.d_par, loop.d_aux, best, stream=stream)
        loop.make_logits()
        if w.mode != W.MODE_STATIC:
            eng.coverage(B, loop.tok, loop.par, loop.info, loop.logits, gain, stream=stream)
        with torch.cuda.stream(stream):
            flush_l2()
        e[2].record(stream)
        eng.verify_update_sample(B, loop.tok, loop.par, loop.pos, loop.mask, loop.logits, temp, u, ur,
                                 loop.accept_len, loop.out_tokens, stream=stream)
        e[3].record(stream)
        loop.advance()
        if k >= 3:
            if trace:
                for name, ms in eng.profile_read():
                    kern.setdefault(name, []).append(ms)
            else:
                ms_asm.append(e[0].elapsed_time(e[1]))
                ms_ver.append(e[2].elapsed_time(e[3]))
                acc.append(float(loop.accept_len.float().mean().item()))
    eng.profile_enable(False)
    step_ms = statistics.mean(ms_asm) + statistics.mean(ms_ver)
    return {"stochastic_step": {"steps_per_s": round(1e3 / step_ms, 1), "ms_per_step": round(step_ms, 5),
                                "temperature": temp, "mean_accept_len": round(statistics.mean(acc), 3)},
            "kernels_us": {k: round(statistics.mean(v) * 1e3, 2) for k, v in sorted(kern.items())},
            "note": "stochastic step = assemble + verify_update_sample (CUDA events, L2 flushed before each); "
                    "kernels from alternate steps with tracing on; k_check here is graft_confidence"}


def run_incremental(w, eng, loop, stream, flush_l2, steps=30):
    """Mean per-step kernel times (us) of the incremental-drafting calls next to
    graft_assemble on the same drafts, L2 flushed before each: graft_check's
    launches (made while the drafter works), graft_retrieve (beside it), and
    graft_assemble_staged (what stays on the critical path)."""
    import torch
    side = torch.cuda.Stream(stream.device)
    eng.profile_enable(True)
    eng.profile_read()
    acc = {"assemble": [], "check_total": [], "retrieve": [], "assemble_staged": []}
    fired = 0
    for _ in range(steps):
        loop.draft()
        with torch.cuda.stream(stream):
            flush_l2()
        loop.assemble()
        with torch.cuda.stream(stream):
            flush_l2()
        loop.assemble_incremental(side)
        loop.make_logits()
        loop.verify_update()
        loop.advance()
        names = eng.profile_read()
        asm = [ms for n, ms in names if n == "k_assemble"]
        acc["assemble"].append(asm[0])
        acc["assemble_staged"].append(asm[1])
        acc["check_total"].append(sum(ms for n, ms in names if n == "k_check"))
        acc["retrieve"].append(sum(ms for n, ms in names if n == "k_retrieve"))
        fired += int((loop.event >= 0).sum().item())
    eng.profile_enable(False)
    out = {k: round(statistics.mean(v) * 1e3, 2) for k, v in acc.items()}
    out["fired_fraction"] = round(fired / (steps * w.B), 3)
    out["note"] = "us per step; the side stream's retrieve overlaps the drafter, assemble_staged replaces assemble"
    return out


def pinned_copy(t):
    """A copy of device tensor t in page-locked host memory."""
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def run_e2e(args, w, eng, loop, stream, dev):
    """Same step through the C ABI with host buffers: the inputs of recorded
    steps are replayed from pinned memory (H2D inside the timed region, one
    cudaMemcpyAsync per buffer), the accept lengths and emitted tokens copied
    back (D2H inside).  Two device input sets: step k + 1's inputs are copied
    on a copy stream while step k's kernels run (events order a set's copy
    after the kernels that last read it).  The pinned-to-device copy rate of
    the logits alone is measured beside it."""
    import torch
    n_rec = 2
    B, S, n = w.B, w.S, w.draft_nodes
    rec = []
    for _ in range(n_rec):
        loop.draft()
        loop.assemble()
        loop.make_logits()
        with torch.cuda.stream(stream):
            # The replayed trees change as the matrix does, so a slot that was a
            # pad when the step was recorded may be verified in a replay: give
            # every pad row (NaN, so that reading one is flagged) its request's
            # root row, so the replay verifies ordinary rows.
            lg = loop.logits.view(B, S, -1)
            pad = torch.isnan(lg[:, :, 0].float())
            lg.copy_(torch.where(pad[:, :, None], lg[:, :1, :], lg))
        stream.synchronize()
        rec.append({k: pinned_copy(t) for k, t in (("root", loop.root), ("tok", loop.d_tok), ("par", loop.d_par),
                                                    ("aux", loop.d_aux), ("logits", loop.logits))})
        loop.verify_update()
        loop.advance()
    tail = w.mode == W.MODE_TAIL
    sets = [dict(root=torch.empty(B, dtype=torch.int32, device=dev), tok=torch.empty_like(loop.d_tok),
                 par=None if tail else torch.empty_like(loop.d_par), aux=torch.empty_like(loop.d_aux),
                 logits=torch.empty_like(loop.logits)) for _ in range(2)]
    h_acc = torch.empty(B, dtype=torch.int32).pin_memory()
    h_out = torch.empty((B, S), dtype=torch.int32).pin_memory()
    h2d = sum(rec[0][k].numel() * rec[0][k].element_size() for k in ("root", "tok", "aux", "logits"))
    if not tail:
        h2d += rec[0]["par"].numel() * rec[0]["par"].element_size()
    d2h = B * 4 + B * S * 4
    steps = max(args.e2e_steps, 1)
    cs = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def copy_in(k):
        d, r = sets[k % 2], rec[k % n_rec]
        cs.wait_event(free[k % 2])                   # the kernels that last read this set are done
        with torch.cuda.stream(cs):
            for key in ("root", "tok", "par", "aux", "logits"):
                if d[key] is not None:
                    d[key].copy_(r[key], non_blocking=True)
        ready[k % 2].record(cs)

    def compute(k):
        d = sets[k % 2]
        stream.wait_event(ready[k % 2])
        eng.assemble(B, d["root"], d["tok"], d["par"], d["aux"], loop.tok, loop.par, loop.pos, loop.mask, loop.info,
                     stream=stream)
        eng.verify_update(B, loop.tok, loop.par, loop.pos, loop.mask, d["logits"], loop.accept_len, loop.out_tokens,
                          stream=stream)
        free[k % 2].record(stream)
        with torch.cuda.stream(stream):
            h_acc.copy_(loop.accept_len, non_blocking=True)
            h_out.copy_(loop.out_tokens, non_blocking=True)

    def run(nsteps):
        copy_in(0)
        for k in range(nsteps):
            if k + 1 < nsteps:
                copy_in(k + 1)
            compute(k)

    run(3)
    torch.cuda.synchronize()
    reps = []
    for _ in range(2):  # two timed repetitions, both reported; the value is their mean
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cs.wait_event(e0)
        run(steps)
        e1.record(stream)
        e1.synchronize()
        reps.append(e0.elapsed_time(e1))
    ms = statistics.mean(reps)
    # the link alone: each recorded step's logits copied from pinned memory on the copy stream
    lbytes = rec[0]["logits"].numel() * rec[0]["logits"].element_size()
    links = []
    for r in rec:
        lms = []
        for _ in range(3):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(cs)
            with torch.cuda.stream(cs):
                sets[0]["logits"].copy_(r["logits"], non_blocking=True)
            c1.record(cs)
            c1.synchronize()
            lms.append(c0.elapsed_time(c1))
        links.append(lbytes / (min(lms) / 1e3) / 1e9)
    link = statistics.mean(links)
    return {"value": round(steps / (ms / 1e3), 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "h2d_link_GBps": round(link, 1),
            "h2d_link_GBps_per_buffer": [round(x, 1) for x in links],
            "repetitions_steps_per_s": [round(steps / (m / 1e3), 3) for m in reps],
            "h2d_GBps_achieved": round(h2d * steps / (ms / 1e3) / 1e9, 1),
            "note": "inputs copied from pinned host memory each step (copy stream, double-buffered: step k + 1's "
                    "copy overlaps step k's kernels); h2d_link_GBps = a lone pinned-to-device copy of the logits"}


def main():
    args = parse()
    ws, rank, local = dist_env()
    if ws > 1:
        import torch
        backend = "nccl" if args.impl == "graft" else "gloo"
        if args.impl == "graft":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    w = W.WORKLOADS[args.workload]
    if args.draft_sigma is not None:
        w = w.scaled(draft_sigma=args.draft_sigma)
    if args.impl == "reference":
        if rank != 0:
            return
        # the CPU oracle on the whole batch, every host core
        if args.warmup > 0:
            oracle_sample(w, 0.0, max_steps=args.warmup)
        det = oracle_sample(w, 0.0, max_steps=args.steps, warm=args.oracle_warm)
        v = det["all_cores"]
        out = {"metric": METRIC, "value": round(v, 5), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": round(1e3 / v, 3), "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == W.BF16 else "f32",
               "data": "synthetic", "impl": "reference",
               "config": workload_config(w, ws),
               "cpu_baseline": cpu_baseline_entry(det, w),
               "e2e": {"value": round(v, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(out))
        return
    out = run_graft(args, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and ws == 1:
            out["cpu_baseline"] = cpu_baseline_entry(oracle_sample(w, args.cpu_seconds), w)
        print(json.dumps(out))
    if ws > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
