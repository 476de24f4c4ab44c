"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle,
element by element on the same seeded inputs — trees, positions, masks,
acceptance, emitted tokens and the continuation matrix after every step.

Covers the five workloads (checkpoint / static / tail modes, fp32 and bf16),
ragged and unaligned rows (vector and scalar load paths, tail elements),
rows that overflow the candidate list (all-equal values), warm-up, the
device-side error flags, and full-size cases in the benchmark's launch
configuration.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def G():
    import hybrid_draft_tree_gb300 as g
    return g


def engine_for(w, **kw):
    g = G()
    cfg = g.graft_default_config(w.V, w.B, w.mode, w.dtype, budget=w.budget, max_draft_nodes=w.draft_nodes, **kw)
    return g.Graft(cfg)


def u16_to_bf16_tensor(u16, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).to(device).view(torch.bfloat16)


def assert_trees_equal(loop, trees, step):
    B = loop.w.B
    gt = loop.tok.cpu().numpy()
    gp = loop.par.cpu().numpy().astype(np.int32)
    gpos = loop.pos.cpu().numpy()
    gm = loop.mask.cpu().numpy().view(np.uint64)
    gi = loop.info.cpu().numpy()
    for b in range(B):
        tr = trees[b]
        assert np.array_equal(gt[b], tr.tok), (step, b, "tok")
        assert np.array_equal(gp[b], tr.par), (step, b, "parent")
        assert np.array_equal(gpos[b], tr.pos), (step, b, "pos")
        assert np.array_equal(gm[b], tr.mask), (step, b, "mask")
        assert np.array_equal(gi[b], tr.info), (step, b, "info", gi[b], tr.info)


def lockstep(w, steps, warm=False, check_rows=0, stats=None, **cfg):
    """Run the GPU closed loop and the oracle side by side; compare all."""
    from workloads.device_loop import DeviceLoop
    g = engine_for(w, **cfg)
    loop = DeviceLoop(w, g)
    shared = {k: v for k, v in cfg.items() if k in ("tpl_depth", "tpl_width", "ablation", "fixed_draft")}
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode, **shared)
    C = oracle.new_matrix(w.V)
    if warm:
        toks_d, logits_d, (toks, rk, pl, bi) = loop.warm_inputs_device()
        g.warmup(toks_d, logits_d)
        rows = W.fill_rows(rk, pl, bi, w.V, w.dtype)
        oracle.warmup(C, toks, rows, w.dtype)
        assert np.array_equal(g.get_matrix(), C), "matrix after warm-up"
        del logits_d
    for step in range(steps):
        tok, par, aux = loop.draft()
        loop.assemble()
        trees = [oracle.assemble(P, loop.root_h[b], tok[b], aux[b], C, None if par is None else par[b])
                 for b in range(w.B)]
        assert_trees_equal(loop, trees, step)
        loop.make_logits()
        tt = np.stack([t.tok for t in trees])
        pp = np.stack([t.par for t in trees]).astype(np.int8)
        lg = loop.h.tree_logits(tt, pp, loop.ctx_h, loop.prev_h)
        if check_rows:
            dev = loop.logits.view(torch.int16 if w.dtype else torch.int32).cpu().numpy()
            flat = lg.reshape(w.B * w.S, -1)
            for r in np.random.default_rng(step).choice(w.B * w.S, check_rows, replace=False):
                if tt.reshape(-1)[r] >= 0:
                    assert np.array_equal(dev[r].view(flat.dtype), flat[r]), ("logits row", step, r)
        loop.verify_update()
        acc_g = loop.accept_len.cpu().numpy()
        out_g = loop.out_tokens.cpu().numpy()
        for b in range(w.B):
            acc, out, topk = oracle.verify(trees[b], lg[b], w.dtype)
            oracle.update(C, trees[b], topk)
            assert acc_g[b] == acc, (step, b, "accept_len", acc_g[b], acc)
            assert np.array_equal(out_g[b], out), (step, b, "out_tokens", out_g[b], out)
            if stats is not None:
                stats.append((int(trees[b].info[0]), acc))
        assert np.array_equal(g.get_matrix(), C), (step, "matrix")
        loop.advance()
    assert g.sync() == 0
    g.close()


# ------------------------------------------------------------------------------ generator
def test_generator_device_matches_host():
    rng = np.random.default_rng(0)
    for dtype in (W.F32, W.BF16):
        h = W.Harness(W.WORKLOADS[1].scaled(V=1037, dtype=dtype))
        ds = W.DeviceSynth(h, torch.device("cuda"))
        n = 7
        rk = rng.integers(0, 2**64, n, dtype=np.uint64)
        pl = np.array([5, -1, -2, 1036, 0, 77, -1], np.int32)
        bi = np.full(n, 5.0, np.float32)
        host = W.fill_rows(rk, pl, bi, 1037, dtype)
        out = torch.empty((n, 1037), dtype=torch.float32 if dtype == W.F32 else torch.bfloat16, device="cuda")
        ds.fill_rows(torch.from_numpy(rk.view(np.int64)).cuda(), torch.from_numpy(pl).cuda(),
                     torch.from_numpy(bi).cuda(), out, torch.cuda.current_stream().cuda_stream)
        bits = np.uint32 if dtype == W.F32 else np.uint16                 # NaN pad rows compare by bits
        dev = out.view(torch.int32 if dtype == W.F32 else torch.int16).cpu().numpy().view(bits)
        assert np.array_equal(dev, host.view(bits))
    # tree row parameters
    B, S = 3, 61
    tok = rng.integers(0, 1037, (B, S)).astype(np.int32)
    par = np.full((B, S), -1, np.int8)
    for i in range(1, S):
        par[:, i] = rng.integers(0, i, B)
    tok[1, 40:] = -1
    prev = rng.integers(0, 1037, B).astype(np.int32)
    ctx = rng.integers(0, 2**64, B, dtype=np.uint64)
    hk, hp, hb = h.tree_rowparams(tok, par, ctx, prev)
    dk, dp, db = ds.tree_rowparams(torch.from_numpy(tok).cuda(), torch.from_numpy(par).cuda(),
                                   torch.from_numpy(ctx.view(np.int64)).cuda(), torch.from_numpy(prev).cuda(),
                                   torch.cuda.current_stream().cuda_stream)
    assert np.array_equal(dk.cpu().numpy().view(np.uint64), hk)
    assert np.array_equal(dp.cpu().numpy(), hp)
    assert np.array_equal(db.cpu().numpy(), hb)


# ------------------------------------------------------------------------------ closed loops
@pytest.mark.parametrize("wid,V,B,sigma,steps", [
    (0, 3001, 1, 2.0, 25),      # checkpoint, fp32, ragged V
    (0, 4000, 1, 0.75, 40),     # checkpoint, all checkpoints fire
    (0, 4000, 4, 0.5, 20),      # batched checkpoint mode
    (1, 5003, 1, 0.75, 30),     # bf16 trigram target, ragged V
    (2, 6000, 16, 2.0, 20),     # static mode, shared matrix across 16 requests
    (2, 777, 16, 0.75, 20),     # static mode, heavy duplicate tokens (last-writer races)
    (4, 6007, 64, 2.0, 15),     # tail mode, 64 requests
    (4, 500, 64, 2.0, 15),      # tail mode, small vocab: many duplicate writers
])
def test_lockstep_small(wid, V, B, sigma, steps):
    w = W.WORKLOADS[wid].scaled(V=V, B=B, draft_sigma=sigma)
    stats = []
    lockstep(w, steps, check_rows=8, stats=stats)
    assert any(a > 0 for _, a in stats)


@pytest.mark.parametrize("seed", range(40))
def test_lockstep_random_configurations(seed):
    """Seeded random configurations (mode, logits type, vocabulary, batch,
    draft spread and verify path drawn together), four closed-loop steps
    each against the oracle: combinations the hand-picked cases above leave
    out (e.g. fp32 static trees on the cluster verify, small tail batches on
    the unit-record scan)."""
    rng = np.random.default_rng(1000 + seed)
    wid = int(rng.choice([0, 1, 2, 4]))
    V = int(rng.integers(300, 50001))
    dtype = int(rng.choice([W.F32, W.BF16]))
    B = int(rng.integers(1, 9)) if wid != 4 else int(rng.integers(1, 65))
    sigma = float(rng.choice([0.5, 0.75, 2.0]))
    scan_kernel = int(rng.choice([0, 1, 2, 3, 4, 5]))
    w = W.WORKLOADS[wid].scaled(V=V, B=B, draft_sigma=sigma, dtype=dtype)
    lockstep(w, 4, check_rows=2, scan_kernel=scan_kernel)


@pytest.mark.parametrize("wid,V,B,sigma", [(0, 3000, 3, 0.75), (2, 777, 16, 0.75), (4, 6007, 64, 2.0)])
def test_slot_provenance(wid, V, B, sigma):
    """graft_assemble_src writes the same trees as graft_assemble (compared
    with the oracle) plus each slot's provenance: the root, the kept draft
    nodes (info[1] of them), the matrix (info[2]: retrieval nodes after the
    kept draft slots, or in-place replacements in static mode), pads."""
    from workloads.device_loop import DeviceLoop
    w = W.WORKLOADS[wid].scaled(V=V, B=B, draft_sigma=sigma)
    g = engine_for(w)
    loop = DeviceLoop(w, g, track_src=True)
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode)
    C = oracle.new_matrix(w.V)
    retrieved = 0
    for step in range(12):
        tok, par, aux = loop.draft()
        loop.assemble()
        trees = [oracle.assemble(P, loop.root_h[b], tok[b], aux[b], C, None if par is None else par[b])
                 for b in range(w.B)]
        assert_trees_equal(loop, trees, step)
        src = loop.src.cpu().numpy()
        for b, tr in enumerate(trees):
            valid = tr.tok >= 0
            assert np.array_equal(src[b] == -1, ~valid), (step, b)
            assert src[b][0] == (0 if valid[0] else -1)
            assert int((src[b] == 1).sum()) == tr.info[1] and int((src[b] == 2).sum()) == tr.info[2], (step, b)
            if w.mode != W.MODE_STATIC:
                r0 = 1 + int(tr.info[1])
                assert (src[b][1:r0][valid[1:r0]] == 1).all() and (src[b][r0:][valid[r0:]] == 2).all()
            retrieved += int(tr.info[2])
        loop.make_logits()
        tt = np.stack([t.tok for t in trees])
        pp = np.stack([t.par for t in trees]).astype(np.int8)
        lg = loop.h.tree_logits(tt, pp, loop.ctx_h, loop.prev_h)
        loop.verify_update()
        for b in range(w.B):
            acc, out, topk = oracle.verify(trees[b], lg[b], w.dtype)
            oracle.update(C, trees[b], topk)
        loop.advance()
    assert retrieved > 0
    assert g.sync() == 0
    g.close()


@pytest.mark.parametrize("scan_kernel", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("wid,V,B,sigma,steps", [
    (2, 40000, 16, 2.0, 8),     # static, 80 KB rows: 3 chunks per row, rows split over CTAs
    (4, 24576, 64, 2.0, 6),     # tail, 64 requests x 17 slots
    (0, 16384, 1, 0.75, 20),    # fp32 checkpoint, 64 KB rows, few rows per step
])
def test_lockstep_both_scan_kernels(scan_kernel, wid, V, B, sigma, steps):
    """The single-pass, TMA-pipelined, two-pass (unit maxima only, and unit
    records) and cluster-per-row verify scans on rows of >= 32 KB, closed loop
    against the oracle (the cluster path takes the 61-row case; the others
    fall back to the two-pass scan)."""
    w = W.WORKLOADS[wid].scaled(V=V, B=B, draft_sigma=sigma)
    lockstep(w, steps, check_rows=4, scan_kernel=scan_kernel)


@pytest.mark.parametrize("scan_kernel", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("V,pad,fn", [(40000, 0, "normal"), (40003, 5, "normal"), (65536, 0, "ties"),
                                      (33000, 0, "constant")])
def test_verify_scan_kernels(scan_kernel, dtype, V, pad, fn):
    """Every scan on aligned rows: ragged tails (V % 8 != 0 with a padded
    stride), heavy ties, all-equal rows (candidate overflow)."""
    fns = {"normal": _normal, "ties": _ties, "constant": _constant}
    _verify_case(V, dtype, 61, 3, fns[fn], stride_pad=pad, seed=V + pad, scan_kernel=scan_kernel)


@pytest.mark.parametrize("cfg", [dict(ablation=1), dict(ablation=2, fixed_draft=40), dict(ablation=2, fixed_draft=0),
                                 dict(ablation=2, fixed_draft=60), dict(tpl_depth=2), dict(tpl_depth=12),
                                 dict(tpl_width=4), dict(tpl_width=16), dict(tpl_depth=10, tpl_width=16)])
def test_lockstep_ablations_and_templates(cfg):
    """The section 五 ablations (no retrieval, fixed split) and other
    template depths and widths, closed loop against the oracle."""
    w = W.WORKLOADS[0].scaled(V=3000, B=3, draft_sigma=0.75)
    stats = []
    lockstep(w, 12, stats=stats, **cfg)
    if cfg.get("fixed_draft", 1) > 0:    # with no draft slots and a cold matrix nothing is accepted
        assert any(a > 0 for _, a in stats)


@pytest.mark.parametrize("cfg", [{}, dict(ablation=1), dict(ablation=2, fixed_draft=40), dict(tpl_depth=12)])
def test_incremental_drafting_matches_assemble_and_oracle(cfg):
    """Checkpoints evaluated layer by layer, the retrieval gathered on a
    second stream, then the staged assembly: the same trees as graft_assemble
    and as the oracle, closed loop (the matrix fills as the loop runs)."""
    _incremental_case(W.WORKLOADS[0].scaled(V=3000, B=4, draft_sigma=0.75), cfg, 12)


@pytest.mark.slow
def test_incremental_drafting_full_size():
    """The same at full size (V = 151936, bf16), the matrix filling as the loop runs."""
    _incremental_case(W.WORKLOADS[3].scaled(draft_sigma=0.75), {}, 6)


def _incremental_case(w, cfg, steps):
    from workloads.device_loop import DeviceLoop
    g = engine_for(w, **cfg)
    loop = DeviceLoop(w, g)
    shared = {k: v for k, v in cfg.items() if k in ("tpl_depth", "tpl_width", "ablation", "fixed_draft")}
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode, **shared)
    C = oracle.new_matrix(w.V)
    side = torch.cuda.Stream()
    fired = 0
    for step in range(steps):
        tok, par, aux = loop.draft()
        loop.assemble()
        ref = [t.clone() for t in (loop.tok, loop.par, loop.pos, loop.mask, loop.info)]
        loop.assemble_incremental(side)
        for x, y in zip((loop.tok, loop.par, loop.pos, loop.mask, loop.info), ref):
            assert torch.equal(x, y), step
        ev_g = loop.event.cpu().numpy()
        rt_g = loop.retrieved.cpu().numpy()
        depth = np.zeros(w.draft_nodes, np.int32)
        for i in range(w.draft_nodes):
            depth[i] = 0 if par[0][i] < 0 else depth[par[0][i]] + 1
        for b in range(w.B):
            ev = -1
            for L in range(int(depth.max()) + 1):
                m = int((depth <= L).sum())
                ev = oracle.check_layer(P, par[b][:m], aux[b][:m], L, ev)
            assert ev_g[b] == ev, (step, b)
            assert np.array_equal(rt_g[b], oracle.retrieve(P, loop.root_h[b], ev, C)), (step, b)
            fired += ev >= 0
        trees = [oracle.assemble(P, loop.root_h[b], tok[b], aux[b], C, par[b]) for b in range(w.B)]
        assert_trees_equal(loop, trees, step)
        loop.make_logits()
        tt = np.stack([t.tok for t in trees])
        pp = np.stack([t.par for t in trees]).astype(np.int8)
        lg = loop.h.tree_logits(tt, pp, loop.ctx_h, loop.prev_h)
        loop.verify_update()
        for b in range(w.B):
            acc, out, topk = oracle.verify(trees[b], lg[b], w.dtype)
            oracle.update(C, trees[b], topk)
        assert np.array_equal(g.get_matrix(), C), step
        loop.advance()
    assert g.sync() == 0
    if cfg.get("ablation", 0) != 2:
        assert fired > 0
    g.close()


def _oracle_layer_best(par, prob):
    """Best fp32 path confidence of checkpoint layers 0, 1, 5 from the
    oracle's path confidences and depths (-1 for an empty layer)."""
    conf, depth = oracle.path_conf(par, prob)
    return np.array([conf[depth == d].max() if (depth == d).any() else -1.0 for d in (0, 1, 5)], np.float32)


def test_confidence_and_calibrated_thresholds():
    """graft_confidence returns each checkpoint layer's best fp32 path
    confidence, equal to the maximum of the oracle's path confidences over
    that layer; thresholds calibrated from those over warm-up steps then
    drive the checkpoints exactly as in the oracle with the same thresholds.
    The oracle runs the whole closed loop on its own matrix."""
    from workloads.device_loop import DeviceLoop
    w = W.WORKLOADS[0].scaled(V=3000, B=4, draft_sigma=0.75)
    g_ = G()
    eng = engine_for(w)
    loop = DeviceLoop(w, eng)
    best = torch.empty((w.B, 3), dtype=torch.float32, device="cuda")
    C = oracle.new_matrix(w.V)

    def closed_step(P, step):
        tok, par, aux = loop.draft()
        eng.confidence(w.B, loop.d_par, loop.d_aux, best)
        got = best.cpu().numpy()
        for b in range(w.B):
            assert np.array_equal(got[b], _oracle_layer_best(par[b], aux[b])), (step, b)
        loop.assemble()
        trees = [oracle.assemble(P, loop.root_h[b], tok[b], aux[b], C, par[b]) for b in range(w.B)]
        assert_trees_equal(loop, trees, step)
        loop.make_logits()
        tt = np.stack([t.tok for t in trees])
        pp = np.stack([t.par for t in trees]).astype(np.int8)
        lg = loop.h.tree_logits(tt, pp, loop.ctx_h, loop.prev_h)
        loop.verify_update()
        acc_g = loop.accept_len.cpu().numpy()
        out_g = loop.out_tokens.cpu().numpy()
        for b in range(w.B):
            acc, out, topk = oracle.verify(trees[b], lg[b], w.dtype)
            oracle.update(C, trees[b], topk)
            assert acc_g[b] == acc and np.array_equal(out_g[b], out), (step, b)
        assert np.array_equal(eng.get_matrix(), C), step
        loop.advance()
        return got, sum(int(t.info[0] >= 0) for t in trees)

    P0 = oracle.make_params(w.V)
    samples = [closed_step(P0, step)[0] for step in range(6)]
    thr = g_.calibrate_thresholds(np.concatenate(samples), 0.4)
    eng.set_thresholds(thr)
    P = oracle.make_params(w.V, ckpt_thr=tuple(float(x) for x in thr))
    fired = sum(closed_step(P, 6 + step)[1] for step in range(8))
    assert fired > 0
    assert eng.sync() == 0
    with pytest.raises(g_.GraftError):
        eng.set_thresholds([0.5, 1.5, 0.1])
    eng.close()


@pytest.mark.parametrize("wid,B", [(0, 3), (4, 8)])
def test_coverage_gain_matches_oracle(wid, B):
    """The coverage diagnostic against the oracle's fp64 value (fp32 softmax
    over one row: relative 1e-4, absolute 1e-7)."""
    _coverage_case(W.WORKLOADS[wid].scaled(V=5000, B=B, draft_sigma=0.75), 10)


@pytest.mark.parametrize("seed", range(10))
def test_coverage_gain_random_configurations(seed):
    """The coverage diagnostic on seeded random configurations (checkpoint
    or tail mode, logits type, vocabulary with ragged tails, batch, draft
    spread) against the oracle's fp64 value."""
    rng = np.random.default_rng(5000 + seed)
    wid = int(rng.choice([0, 1, 4]))
    V = int(rng.integers(300, 60001))
    dtype = int(rng.choice([W.F32, W.BF16]))
    B = int(rng.integers(1, 7)) if wid != 4 else int(rng.integers(1, 65))
    sigma = float(rng.choice([0.5, 0.75, 2.0]))
    _coverage_case(W.WORKLOADS[wid].scaled(V=V, B=B, draft_sigma=sigma, dtype=dtype), 8, need_gain=False)


@pytest.mark.slow
def test_coverage_gain_full_size_tail():
    """The same on the tail workload at full size (64 requests, V = 151936)."""
    _coverage_case(W.WORKLOADS[4], 2)


def _coverage_case(w, steps, need_gain=True):
    from workloads.device_loop import DeviceLoop
    B = w.B
    eng = engine_for(w)
    loop = DeviceLoop(w, eng)
    gain = torch.empty((B,), dtype=torch.float32, device="cuda")
    seen = 0
    for step in range(steps):
        loop.draft()
        loop.assemble()
        loop.make_logits()
        eng.coverage(B, loop.tok, loop.par, loop.info, loop.logits, gain)
        got = gain.cpu().numpy()
        toks, pars, info = loop.tok.cpu().numpy(), loop.par.cpu().numpy(), loop.info.cpu().numpy()
        rows = loop.logits.view(torch.int16 if w.dtype else torch.int32).cpu().numpy().reshape(B, w.S, -1)
        for b in range(B):
            t = oracle.Tree(w.S)
            t.tok[:], t.par[:] = toks[b], pars[b].astype(np.int32)
            exp = oracle.coverage(t, info[b], rows[b].view(np.uint16) if w.dtype else rows[b].view(np.float32), w.dtype)
            assert abs(got[b] - exp) <= 1e-4 * exp + 1e-7, (step, b, got[b], exp)
            seen += exp > 0
        loop.verify_update()
        loop.advance()
    assert seen > 0 or not need_gain
    eng.close()
    return seen


@pytest.mark.parametrize("wid,B,temp", [(0, 4, 1.0), (0, 4, 0.7), (2, 4, 1.0), (4, 8, 1.5)])
def test_stochastic_verification_matches_oracle(wid, B, temp):
    """Sampling acceptance against the oracle's fp64 walk on the same
    uniforms, closed loop.  Where a decision of the oracle lies within 2e-5
    (relative) of its threshold, fp32 and fp64 may take either side (the
    kernel's sums of exp over a row carry ~1e-6 relative error), so only
    requests whose every decision is clear are compared; the matrix update
    is the greedy one and is compared always."""
    w = W.WORKLOADS[wid].scaled(V=5000, B=B, draft_sigma=0.75, bias=12.0)   # a confident target: paths get accepted
    _stochastic_case(w, temp, 10, wid * 10 + int(temp * 10))


@pytest.mark.parametrize("wid,B,temp,dtype", [(4, 64, 1.0, W.BF16), (4, 48, 0.5, W.F32), (2, 40, 0.5, W.BF16),
                                               (2, 32, 1.0, W.F32)])
def test_stochastic_verification_many_requests(wid, B, temp, dtype):
    """Batches of 32 requests and more: more clusters than fit beside pass 2's
    CTAs at once, so the walk's CTAs start in several waves."""
    w = W.WORKLOADS[wid].scaled(V=6007 if wid == 4 else 7001, B=B, draft_sigma=0.75, dtype=dtype)
    _stochastic_case(w, temp, 5, 60 + B, min_fraction=0.4)


@pytest.mark.parametrize("V,B", [(100003, 2), (330007, 1)])
def test_stochastic_verification_long_fp32_rows(V, B):
    """fp32 rows whose eighth per cluster CTA needs more than the default 48 KB
    of shared memory (the kernel opts in) and more than the 160 KB it stages
    (the draw then re-reads its chunk from global memory)."""
    w = W.WORKLOADS[0].scaled(V=V, B=B, draft_sigma=0.75, bias=16.0)   # the planted token dominates each draw
    _stochastic_case(w, 1.0, 4, V % 97)


@pytest.mark.parametrize("wid,B", [(0, 2), (2, 1)])
def test_stochastic_verification_after_the_cluster_verify(wid, B):
    """Sampling acceptance when the greedy pass is the cluster-per-row verify
    (it writes the staged top-8s and the matrix, the walk follows it)."""
    w = W.WORKLOADS[wid].scaled(V=5000, B=B, draft_sigma=0.75, bias=12.0)
    _stochastic_case(w, 1.0, 8, 40 + wid, scan_kernel=5)


@pytest.mark.slow
def test_stochastic_verification_full_size_static():
    """The same on the static workload at full size (16 x 61 rows of 151936).
    Every context gets a planted successor with a large boost so that the
    draws land on wide intervals: a draw among 150K near-equal tokens is an
    fp32 tie."""
    _stochastic_case(W.WORKLOADS[2].scaled(bias=20.0, hit_rate=1.0), 1.0, 2, 99)


def _stochastic_case(w, temp, steps, seed, min_fraction=0.5, need_accept=True, **cfg):
    from workloads.device_loop import DeviceLoop
    eng = engine_for(w, **cfg)
    loop = DeviceLoop(w, eng)
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode)
    C = oracle.new_matrix(w.V)
    rng = np.random.default_rng(seed)
    compared = total = accepted = 0
    for step in range(steps):
        tok, par, aux = loop.draft()
        loop.assemble()
        trees = [oracle.assemble(P, loop.root_h[b], tok[b], aux[b], C, None if par is None else par[b])
                 for b in range(w.B)]
        assert_trees_equal(loop, trees, step)
        loop.make_logits()
        tt = np.stack([t.tok for t in trees])
        pp = np.stack([t.par for t in trees]).astype(np.int8)
        lg = loop.h.tree_logits(tt, pp, loop.ctx_h, loop.prev_h)
        u = rng.random((w.B, w.S)).astype(np.float32)
        ur = rng.random(w.B).astype(np.float32)
        eng.verify_update_sample(w.B, loop.tok, loop.par, loop.pos, loop.mask, loop.logits, temp,
                                 torch.from_numpy(u).cuda(), torch.from_numpy(ur).cuda(), loop.accept_len,
                                 loop.out_tokens)
        acc_g = loop.accept_len.cpu().numpy()
        out_g = loop.out_tokens.cpu().numpy()
        for b in range(w.B):
            acc, out, margin = oracle.verify_sample(trees[b], lg[b], w.dtype, 1.0 / temp, u[b].astype(np.float64),
                                                    float(ur[b]))
            total += 1
            if margin > 2e-5:
                compared += 1
                assert acc_g[b] == acc and np.array_equal(out_g[b], out), (step, b, acc_g[b], acc, out_g[b], out)
                accepted += acc
            _, _, topk = oracle.verify(trees[b], lg[b], w.dtype)
            oracle.update(C, trees[b], topk)
        assert np.array_equal(eng.get_matrix(), C), step
        loop.advance()
    assert eng.sync() == 0
    assert compared >= min_fraction * total and (accepted > 0 or not need_accept), (compared, total, accepted)
    eng.close()


@pytest.mark.parametrize("seed", range(16))
def test_stochastic_random_configurations(seed):
    """Seeded random configurations of the stochastic walk (mode, logits
    type, vocabulary, batch, temperature, verify path) in closed loop against
    the oracle's fp64 walk on the same uniforms."""
    rng = np.random.default_rng(2000 + seed)
    wid = int(rng.choice([0, 1, 2, 4]))
    # the draw is compared only where the target lies more than 2e-5 of the
    # mass from a token boundary: vocabularies and temperatures that keep
    # most draws comparable
    V = int(rng.integers(300, 12001))
    dtype = int(rng.choice([W.F32, W.BF16]))
    B = int(rng.integers(1, 7)) if wid != 4 else int(rng.integers(1, 33))
    temp = float(rng.choice([0.25, 0.5, 1.0]))
    scan_kernel = int(rng.choice([0, 3, 5]))
    w = W.WORKLOADS[wid].scaled(V=V, B=B, draft_sigma=0.75, dtype=dtype)
    _stochastic_case(w, temp, 4, 3000 + seed, min_fraction=0.3, need_accept=False, scan_kernel=scan_kernel)


@pytest.mark.parametrize("dtype,V,n,distinct,pad", [
    (W.BF16, 12000, 5000, 4500, 0),   # more last occurrences than the two-pass warm-up takes: the rest single-pass
    (W.F32, 9001, 3000, 800, 0),      # fp32, a vocabulary tail
    (W.BF16, 7001, 2000, 1500, 1),    # rows off 16-byte boundaries: single-pass only
])
def test_warmup_paths_match_oracle(dtype, V, n, distinct, pad):
    """graft_warmup against the oracle's row-by-row load: the two-pass scan
    over the listed last occurrences, its single-pass remainder, unaligned
    rows, tie-heavy rows (the exact rescan)."""
    g_ = G()
    rng = np.random.default_rng(V + n)
    pool = rng.choice(V, distinct, replace=False).astype(np.int32)
    toks = pool[rng.integers(0, distinct, n)]
    vals = rng.normal(size=(n, V)).astype(np.float32)
    ties = rng.random(n) < 0.1
    vals[ties] = rng.integers(-2, 3, (int(ties.sum()), V)).astype(np.float32)
    host_rows = (vals.view(np.uint32) >> 16).astype(np.uint16) if dtype == W.BF16 else vals
    stride = V + pad
    buf = np.zeros((n, stride), host_rows.dtype)
    buf[:, :V] = host_rows
    dev = u16_to_bf16_tensor(buf) if dtype == W.BF16 else torch.from_numpy(buf).cuda()
    eng = g_.Graft(g_.graft_default_config(V, 1, 0, dtype))
    for call in range(2):                         # the second call reuses the handle's warm-up scratch
        eng.warmup(torch.from_numpy(toks).cuda(), dev[:, :V])
        C = oracle.new_matrix(V)
        oracle.warmup(C, toks, host_rows, dtype)
        assert np.array_equal(eng.get_matrix(), C), call
    assert eng.sync() == 0
    eng.close()


@pytest.mark.parametrize("seed", range(12))
def test_warmup_random_configurations(seed):
    """Seeded random warm-up loads (logits type, vocabulary, row count,
    distinct tokens, row padding) against the oracle's row-by-row load."""
    g_ = G()
    rng = np.random.default_rng(4000 + seed)
    dtype = int(rng.choice([W.F32, W.BF16]))
    V = int(rng.integers(100, 40001))
    n = int(rng.integers(1, max(2, min(6000, 40_000_000 // V))))
    distinct = int(rng.integers(1, min(V, n) + 1))
    pad = int(rng.choice([0, 0, 1, 3]))
    pool = rng.choice(V, distinct, replace=False).astype(np.int32)
    toks = pool[rng.integers(0, distinct, n)]
    vals = rng.normal(size=(n, V)).astype(np.float32)
    host_rows = (vals.view(np.uint32) >> 16).astype(np.uint16) if dtype == W.BF16 else vals
    buf = np.zeros((n, V + pad), host_rows.dtype)
    buf[:, :V] = host_rows
    dev = u16_to_bf16_tensor(buf) if dtype == W.BF16 else torch.from_numpy(buf).cuda()
    eng = g_.Graft(g_.graft_default_config(V, 1, 0, dtype))
    eng.warmup(torch.from_numpy(toks).cuda(), dev[:, :V])
    C = oracle.new_matrix(V)
    oracle.warmup(C, toks, host_rows, dtype)
    assert np.array_equal(eng.get_matrix(), C), (dtype, V, n, distinct, pad)
    assert eng.sync() == 0
    eng.close()


@pytest.mark.parametrize("wid", [1, 3])
def test_lockstep_warmup_small(wid):
    base = W.WORKLOADS[wid]
    kw = dict(V=2048, draft_sigma=0.75)
    if base.warm == "history":
        kw.update(hist_len=3000, hist_active=300)
    lockstep(base.scaled(**kw), 15, warm=True)


# ------------------------------------------------------------------------------ assemble edge cases
def _assemble_case(mode, tok, par, prob, C, root, V, budget=60):
    """One request through graft_assemble vs the oracle."""
    g_ = G()
    n = len(tok)
    cfg = g_.graft_default_config(V, 1, mode, W.BF16, budget=budget, max_draft_nodes=max(n, 1))
    eng = g_.Graft(cfg)
    eng.set_matrix(C)
    S = budget + 1
    d = lambda a_, dt: torch.from_numpy(np.ascontiguousarray(a_, dt)[None]).cuda()
    t_tok, t_par, t_pos = (torch.empty((1, S), dtype=x, device="cuda") for x in (torch.int32, torch.int8, torch.int32))
    t_mask = torch.empty((1, S), dtype=torch.int64, device="cuda")
    info = torch.empty((1, 4), dtype=torch.int32, device="cuda")
    eng.assemble(1, torch.tensor([root], dtype=torch.int32, device="cuda"), d(tok, np.int32),
                 None if par is None else d(par, np.int16), d(prob, np.float32), t_tok, t_par, t_pos, t_mask, info)
    P = oracle.make_params(V, budget=budget, mode=mode)
    tr = oracle.assemble(P, root, tok, prob, C, par)
    assert np.array_equal(t_tok.cpu().numpy()[0], tr.tok)
    assert np.array_equal(t_par.cpu().numpy()[0].astype(np.int32), tr.par)
    assert np.array_equal(t_pos.cpu().numpy()[0], tr.pos)
    assert np.array_equal(t_mask.cpu().numpy()[0].view(np.uint64), tr.mask)
    assert np.array_equal(info.cpu().numpy()[0], tr.info), (info.cpu().numpy()[0], tr.info)
    assert eng.sync() == 0
    eng.close()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("seed", range(4))
def test_assemble_degenerate_probabilities(mode, seed):
    """Signed zeros, exact confidence ties, probability-1 chains and an empty
    matrix row: kept set, checkpoint firing and replacement match the oracle."""
    rng = np.random.default_rng(seed)
    V = 500
    h = W.Harness(W.WORKLOADS[0].scaled(V=V))
    root, prev, ctx = h.init_state()
    tok, par, prob = h.draft(seed, root, prev)
    tok, par, prob = tok[0], par[0], prob[0].copy()
    choice = rng.integers(0, 4, len(prob))
    prob[choice == 0] = 0.0
    prob[choice == 1] = -0.0
    prob[choice == 2] = 0.25                      # many exact ties
    prob[:4] = [0.25, 0.25, -0.0, 0.25]
    C = rng.integers(-1, V, (V, 8)).astype(np.int32)
    C[int(root[0])] = -1
    _assemble_case(mode, tok, par, prob, C, int(root[0]), V)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", ["chain8", "chain9", "chain40", "deep_random"])
def test_assemble_deep_trees(mode, shape):
    """Trees whose depth reaches and passes the eight ancestors a node walks
    for its path confidence (deeper ones take the layer-by-layer passes)."""
    rng = np.random.default_rng(len(shape) + 10 * mode)
    V = 400
    if shape.startswith("chain"):
        n = int(shape[5:])
        par = np.arange(-1, n - 1, dtype=np.int16)
    else:
        n = 120
        par = np.array([-1] + [int(rng.integers(max(0, i - 3), i)) for i in range(1, n)], np.int16)
    tok = rng.integers(0, V, n).astype(np.int32)
    prob = rng.choice(np.array([1.0, 0.97, 0.9, 0.5, 0.25], np.float32), n)
    C = rng.integers(-1, V, (V, 8)).astype(np.int32)
    _assemble_case(mode, tok, par, prob, C, 3, V)


def test_assemble_tail_degenerate():
    V = 300
    rng = np.random.default_rng(5)
    C = rng.integers(-1, V, (V, 8)).astype(np.int32)
    btok = rng.integers(0, V, 16).astype(np.int32)
    for conf in ([0.4] * 16, [0.39] + [0.9] * 15, [0.9] * 15 + [-0.0], [0.0] * 16):
        _assemble_case(2, btok, None, np.array(conf, np.float32), C, 7, V, budget=16)
    _assemble_case(2, btok[:0], None, np.zeros(0, np.float32), C, 7, V, budget=16)   # empty block


# ------------------------------------------------------------------------------ verify edge cases
def _tree_from_parents(tok, par):
    S = len(tok)
    t = oracle.Tree(S)
    t.tok[:] = tok
    t.par[:] = par
    for i in range(S):
        if tok[i] < 0:
            t.par[i], t.pos[i], t.mask[i] = -1, -1, 0
        elif i == 0:
            t.pos[0], t.mask[0] = 0, 1
        else:
            t.pos[i] = t.pos[par[i]] + 1
            t.mask[i] = np.uint64(int(t.mask[par[i]]) | (1 << i))
    return t


def _verify_case(V, dtype, S, B, rows_fn, stride_pad=0, seed=0, offset_elems=0, scan_kernel=0):
    """Random trees over rows_fn(rng, n, V) logits, each node following its
    parent's argmax with probability 1/2; GPU verify_update vs the oracle."""
    g_ = G()
    rng = np.random.default_rng(seed)
    vals = rows_fn(rng, B * S, V)                       # float32 [B*S, V]
    if dtype == W.BF16:
        host_rows = (vals.view(np.uint32) >> 16).astype(np.uint16)
    else:
        host_rows = vals
    hr = host_rows.reshape(B, S, V)
    trees = []
    for b in range(B):
        n = int(rng.integers(1, S + 1))
        tok = np.full(S, -1, np.int32)
        par = np.full(S, -1, np.int32)
        tok[:n] = rng.integers(0, V, n)
        for i in range(1, n):
            par[i] = rng.integers(0, i)
            if rng.random() < 0.5:
                tok[i] = oracle.topk8_row(hr[b, par[i]], dtype)[0]
        trees.append(_tree_from_parents(tok, par))
    stride = V + stride_pad
    buf = np.zeros(B * S * stride + offset_elems, host_rows.dtype)
    buf[offset_elems:].reshape(B * S, stride)[:, :V] = host_rows
    dev = u16_to_bf16_tensor(buf) if dtype == W.BF16 else torch.from_numpy(buf).cuda()
    logits = dev[offset_elems:].view(B * S, stride)
    cfg = g_.graft_default_config(V, B, 0, dtype, budget=S - 1, scan_kernel=scan_kernel,
                                  ckpt_draft=(min(8, S - 1), min(24, S - 1), min(40, S - 1)))
    eng = g_.Graft(cfg)
    tt = torch.from_numpy(np.stack([t.tok for t in trees])).cuda()
    tp = torch.from_numpy(np.stack([t.par for t in trees]).astype(np.int8)).cuda()
    tpos = torch.from_numpy(np.stack([t.pos for t in trees])).cuda()
    tm = torch.from_numpy(np.stack([t.mask for t in trees]).view(np.int64)).cuda()
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, S), dtype=torch.int32, device="cuda")
    C0 = rng.integers(-1, V, (V, 8)).astype(np.int32)
    eng.set_matrix(C0)
    eng.verify_update(B, tt, tp, tpos, tm, logits, acc, out)
    C = C0.copy()
    accepted = 0
    for b in range(B):
        a, o, topk = oracle.verify(trees[b], hr[b], dtype)
        oracle.update(C, trees[b], topk)
        assert acc.cpu().numpy()[b] == a
        assert np.array_equal(out.cpu().numpy()[b], o)
        accepted += a
    assert np.array_equal(eng.get_matrix(), C)
    assert eng.sync() == 0
    eng.close()
    return accepted


def _normal(rng, n, V):
    return rng.normal(size=(n, V)).astype(np.float32)


def _ties(rng, n, V):
    v = rng.integers(-2, 3, (n, V)).astype(np.float32)
    v[rng.random((n, V)) < 0.3] = -0.0
    return v


def _constant(rng, n, V):
    return np.full((n, V), 1.5, np.float32)


@pytest.mark.parametrize("V", [1, 7, 8, 37, 1000, 4099, 40000])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_verify_ragged_vocab(V, dtype):
    _verify_case(V, dtype, 61, 2, _normal, seed=V)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("pad,off", [(1, 0), (3, 1), (8, 0)])
def test_verify_unaligned_rows(dtype, pad, off):
    """Row starts off 16-byte boundaries take the scalar-load path."""
    _verify_case(3001, dtype, 17, 3, _normal, stride_pad=pad, offset_elems=off, seed=pad)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_verify_beyond_the_two_pass_row_limit(dtype):
    """More verified rows than the two-pass scan takes (4096): the automatic
    choice falls back to the single-pass scan; same results."""
    _verify_case(1024, dtype, 61, 72, _normal, seed=5)          # 72 x 61 = 4392 rows


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("fn", [_ties, _constant])
def test_verify_ties_and_candidate_overflow(dtype, fn):
    """Heavy ties and all-equal rows (more candidates than the list holds:
    the exact fallback selection)."""
    _verify_case(20000, dtype, 33, 2, fn, seed=11)


def _sparse(rng, n, V):
    """Rows of -inf but for a few finite values: most threads and CTAs see
    no finite element (fewer than 8 finite maxima: the exact pass)."""
    v = np.full((n, V), -np.inf, np.float32)
    k = min(5, V)
    for r in range(n):
        v[r, rng.choice(V, k, replace=False)] = rng.normal(size=k)
    return v


@pytest.mark.parametrize("V", [1, 7, 8, 37, 1000, 4099, 40000])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_cluster_verify_ragged_vocab(V, dtype):
    """The cluster-per-row verify on tiny and ragged rows: CTAs with empty or
    partial ranges, a scalar rest after the last whole vector."""
    _verify_case(V, dtype, 61, 2, _normal, seed=V + 1, scan_kernel=5)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("fn", [_ties, _constant, _sparse])
def test_cluster_verify_ties_overflow_and_sparse_rows(dtype, fn):
    """Heavy ties and all-equal rows (a CTA's list overflows: its exact pass)
    and rows of -inf with a few finite values (no threshold: the exact pass)."""
    _verify_case(20000, dtype, 33, 2, fn, seed=12, scan_kernel=5)


@pytest.mark.parametrize("V,dtype", [(300000, W.F32), (300007, W.F32), (500000, W.BF16), (420000, W.F32)])
def test_cluster_verify_wide_rows(V, dtype):
    """Rows whose eighth needs more than the default 48 KB of shared memory
    (the kernel opts in per launch): 16-byte aligned rows take several 32 KB
    bulk copies per CTA, V = 300007 fp32 rows (not aligned) the plain-load
    staging; past 200 KB per CTA (420000 fp32) the call takes the two-pass
    scan."""
    _verify_case(V, dtype, 9, 2, _normal, seed=V % 1000, scan_kernel=5)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("pad,off", [(1, 0), (3, 1)])
def test_cluster_verify_unaligned_rows(dtype, pad, off):
    """Row starts off 16-byte boundaries: scalar staging."""
    _verify_case(3001, dtype, 17, 3, _normal, stride_pad=pad, offset_elems=off, seed=pad + 7, scan_kernel=5)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("scan_kernel", [0, 1, 3, 5])
def test_verify_request_without_valid_slots(scan_kernel, mode):
    """A request whose slots are all pads (token -1) has no row to finish it:
    the verify still writes its acceptance (nothing accepted, nothing
    emitted; the oracle takes only trees with a valid root), and the other
    requests match the oracle.  A static-mode handle expects every slot
    filled (pass 1 prefetches by that guess): with pads the guess is wrong
    and the results must not change."""
    g_ = G()
    rng = np.random.default_rng(31)
    V, B, S = 3000, 3, 61
    vals = rng.normal(size=(B * S, V)).astype(np.float32)
    trees = []
    for b in range(B):
        n = 0 if b == 1 else int(rng.integers(1, S + 1))
        tok = np.full(S, -1, np.int32)
        par = np.full(S, -1, np.int32)
        tok[:n] = rng.integers(0, V, n)
        for i in range(1, n):
            par[i] = rng.integers(0, i)
        trees.append(_tree_from_parents(tok, par))
    eng = g_.Graft(g_.graft_default_config(V, B, mode, W.F32, scan_kernel=scan_kernel))
    tt = torch.from_numpy(np.stack([t.tok for t in trees])).cuda()
    tp = torch.from_numpy(np.stack([t.par for t in trees]).astype(np.int8)).cuda()
    tpos = torch.from_numpy(np.stack([t.pos for t in trees])).cuda()
    tm = torch.from_numpy(np.stack([t.mask for t in trees]).view(np.int64)).cuda()
    acc = torch.full((B,), 77, dtype=torch.int32, device="cuda")
    out = torch.full((B, S), 77, dtype=torch.int32, device="cuda")
    eng.verify_update(B, tt, tp, tpos, tm, torch.from_numpy(vals).cuda(), acc, out)
    C = oracle.new_matrix(V)
    hr = vals.reshape(B, S, V)
    for b in (0, 2):
        a, o, topk = oracle.verify(trees[b], hr[b], W.F32)
        oracle.update(C, trees[b], topk)
        assert acc.cpu().numpy()[b] == a
        assert np.array_equal(out.cpu().numpy()[b], o)
    assert acc.cpu().numpy()[1] == 0 and (out.cpu().numpy()[1] == -1).all()
    assert np.array_equal(eng.get_matrix(), C)
    assert eng.sync() == 0
    eng.close()


@pytest.mark.parametrize("dtype,pad", [(W.BF16, 0), (W.F32, 0), (W.BF16, 3)])
def test_stochastic_request_without_valid_slots(dtype, pad):
    """Stochastic verification with an all-pad request beside valid ones, on
    the walk's bulk-staged rows (aligned) and its thread-loaded rows (a padded
    stride): the empty request's cluster leaves at once (nothing accepted,
    nothing emitted), and every other request matches the oracle's fp64 walk
    on the same uniforms."""
    g_ = G()
    rng = np.random.default_rng(41 + pad)
    V, B, S = 5003, 4, 61
    vals = (rng.normal(size=(B * S, V)) * 2.0).astype(np.float32)
    host = (vals.view(np.uint32) >> 16).astype(np.uint16) if dtype == W.BF16 else vals
    hb = host.reshape(B, S, V)  # the oracle's input: float32, or bf16 as uint16 bit patterns
    hr = (host.astype(np.uint32) << 16).view(np.float32).reshape(B, S, V) if dtype == W.BF16 else hb
    trees = []
    for b in range(B):
        n = 0 if b == 2 else int(rng.integers(1, S + 1))
        tok = np.full(S, -1, np.int32)
        par = np.full(S, -1, np.int32)
        tok[:n] = rng.integers(0, V, n)
        for i in range(1, n):
            par[i] = rng.integers(0, i)
            if rng.random() < 0.6:
                tok[i] = int(np.argmax(hr[b, par[i]]))
        trees.append(_tree_from_parents(tok, par))
    stride = V + pad
    buf = np.zeros((B * S, stride), host.dtype)
    buf[:, :V] = host
    logits = u16_to_bf16_tensor(buf.reshape(-1)).view(B * S, stride) if dtype == W.BF16 else torch.from_numpy(buf).cuda()
    eng = g_.Graft(g_.graft_default_config(V, B, 0, dtype))
    tt = torch.from_numpy(np.stack([t.tok for t in trees])).cuda()
    tp = torch.from_numpy(np.stack([t.par for t in trees]).astype(np.int8)).cuda()
    tpos = torch.from_numpy(np.stack([t.pos for t in trees])).cuda()
    tm = torch.from_numpy(np.stack([t.mask for t in trees]).view(np.int64)).cuda()
    u = rng.random((B, S)).astype(np.float32)
    ur = rng.random(B).astype(np.float32)
    acc = torch.full((B,), 77, dtype=torch.int32, device="cuda")
    out = torch.full((B, S), 77, dtype=torch.int32, device="cuda")
    eng.verify_update_sample(B, tt, tp, tpos, tm, logits, 1.0, torch.from_numpy(u).cuda(), torch.from_numpy(ur).cuda(),
                             acc, out)
    acc_g, out_g = acc.cpu().numpy(), out.cpu().numpy()
    assert acc_g[2] == 0 and (out_g[2] == -1).all()
    C = oracle.new_matrix(V)
    compared = 0
    for b in (0, 1, 3):
        a, o, margin = oracle.verify_sample(trees[b], hb[b], dtype, 1.0, u[b].astype(np.float64), float(ur[b]))
        if margin > 2e-5:
            compared += 1
            assert acc_g[b] == a and np.array_equal(out_g[b], o), (b, acc_g[b], a, out_g[b], o)
        _, _, topk = oracle.verify(trees[b], hb[b], dtype)
        oracle.update(C, trees[b], topk)
    assert compared >= 2
    assert np.array_equal(eng.get_matrix(), C)
    assert eng.sync() == 0
    eng.close()


def test_stochastic_walk_wait_limit_expires_and_the_handle_recovers():
    """The stochastic walk's staging wait (bulk copies on an mbarrier) gets a
    limit of one poll: the kernel flags GRAFT_ERR_TIMEOUT, lets its copies
    land and finishes.  With the default limit restored, the next call on the
    same handle is clean and gives the same acceptance as a fresh handle."""
    g_ = G()
    rng = np.random.default_rng(23)
    V, B, S = 40000, 4, 61
    vals = rng.normal(size=(B * S, V)).astype(np.float32)
    logits = u16_to_bf16_tensor((vals.view(np.uint32) >> 16).astype(np.uint16))
    trees = []
    for b in range(B):
        tok = rng.integers(0, V, S).astype(np.int32)
        par = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, S)], np.int32)
        trees.append(_tree_from_parents(tok, par))
    tt = torch.from_numpy(np.stack([t.tok for t in trees])).cuda()
    tp = torch.from_numpy(np.stack([t.par for t in trees]).astype(np.int8)).cuda()
    tpos = torch.from_numpy(np.stack([t.pos for t in trees])).cuda()
    tm = torch.from_numpy(np.stack([t.mask for t in trees]).view(np.int64)).cuda()
    u = torch.from_numpy(rng.random((B, S)).astype(np.float32)).cuda()
    ur = torch.from_numpy(rng.random(B).astype(np.float32)).cuda()

    def call(eng):
        acc = torch.empty(B, dtype=torch.int32, device="cuda")
        out = torch.empty((B, S), dtype=torch.int32, device="cuda")
        eng.verify_update_sample(B, tt, tp, tpos, tm, logits, 1.0, u, ur, acc, out)
        return acc, out

    eng = g_.Graft(g_.graft_default_config(V, B, 0, W.BF16))
    eng.set_wait_limit(1)
    call(eng)
    assert eng.sync(raise_on_error=False) & g_.graft.GRAFT_ERR_TIMEOUT
    eng.set_wait_limit(0)
    acc, out = call(eng)
    assert eng.sync() == 0
    fresh = g_.Graft(g_.graft_default_config(V, B, 0, W.BF16))
    acc2, out2 = call(fresh)
    assert fresh.sync() == 0
    assert torch.equal(acc, acc2) and torch.equal(out, out2)
    eng.close()
    fresh.close()


def test_batch_zero_is_a_noop():
    g_ = G()
    eng = g_.Graft(g_.graft_default_config(100, 4, 0, W.BF16))
    eng.verify_update(0, None, None, None, None, torch.empty((1, 100), dtype=torch.bfloat16, device="cuda"),
                      None, None)
    assert eng.sync() == 0
    assert (eng.get_matrix() == -1).all()


def test_error_flags_and_recovery():
    """NaN logits and out-of-range tokens raise device flags (no fault); the
    handle stays usable."""
    g_ = G()
    V, S = 500, 61
    eng = g_.Graft(g_.graft_default_config(V, 1, 0, W.F32))
    tok = np.array([3, 4] + [-1] * (S - 2), np.int32)
    par = np.array([-1, 0] + [-1] * (S - 2), np.int32)
    tr = _tree_from_parents(tok, par)
    tt = torch.from_numpy(tr.tok[None]).cuda()
    tp = torch.from_numpy(tr.par[None].astype(np.int8)).cuda()
    tpos = torch.from_numpy(tr.pos[None]).cuda()
    tm = torch.from_numpy(tr.mask[None].view(np.int64)).cuda()
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, S), dtype=torch.int32, device="cuda")
    logits = torch.zeros((S, V), dtype=torch.float32, device="cuda")
    logits[1, 17] = float("nan")
    eng.verify_update(1, tt, tp, tpos, tm, logits, acc, out)
    assert eng.sync(raise_on_error=False) & g_.graft.GRAFT_ERR_NAN
    assert eng.sync() == 0                               # cleared
    tt[0, 1] = V + 9
    logits[1, 17] = 0.0
    eng.verify_update(1, tt, tp, tpos, tm, logits, acc, out)
    assert eng.sync(raise_on_error=False) & g_.graft.GRAFT_ERR_TOKEN
    tt[0, 1] = 4
    eng.verify_update(1, tt, tp, tpos, tm, logits, acc, out)
    assert eng.sync() == 0
    assert acc.item() == 0 and out[0, 0].item() == 0     # argmax of a zero row is id 0


@pytest.mark.parametrize("scan_kernel,B", [(2, 8), (5, 4)])
def test_bulk_copy_wait_limit_expires_and_the_handle_recovers(scan_kernel, B):
    """Failure detection on the GPU without a fault: the waits for the bulk
    copies (the TMA scan's ring, the cluster verify's staging) get a limit of
    one poll, so they run out while the copies are in flight; the kernel
    flags GRAFT_ERR_TIMEOUT, lets its copies land and finishes.  With the
    default limit restored the next call on the same handle is clean and
    matches the oracle."""
    g_ = G()
    rng = np.random.default_rng(21)
    V, S = 40000, 61
    vals = rng.normal(size=(B * S, V)).astype(np.float32)
    host_rows = (vals.view(np.uint32) >> 16).astype(np.uint16)
    logits = u16_to_bf16_tensor(host_rows)
    trees = []
    for b in range(B):
        tok = rng.integers(0, V, S).astype(np.int32)
        par = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, S)], np.int32)
        trees.append(_tree_from_parents(tok, par))
    eng = g_.Graft(g_.graft_default_config(V, B, 0, W.BF16, scan_kernel=scan_kernel))
    tt = torch.from_numpy(np.stack([t.tok for t in trees])).cuda()
    tp = torch.from_numpy(np.stack([t.par for t in trees]).astype(np.int8)).cuda()
    tpos = torch.from_numpy(np.stack([t.pos for t in trees])).cuda()
    tm = torch.from_numpy(np.stack([t.mask for t in trees]).view(np.int64)).cuda()
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, S), dtype=torch.int32, device="cuda")
    eng.set_wait_limit(1)
    eng.verify_update(B, tt, tp, tpos, tm, logits, acc, out)
    assert eng.sync(raise_on_error=False) & g_.graft.GRAFT_ERR_TIMEOUT
    eng.set_wait_limit(0)
    C0 = rng.integers(-1, V, (V, 8)).astype(np.int32)
    eng.set_matrix(C0)
    eng.verify_update(B, tt, tp, tpos, tm, logits, acc, out)
    assert eng.sync() == 0
    C = C0.copy()
    for b in range(B):
        a, o, topk = oracle.verify(trees[b], host_rows.reshape(B, S, V)[b], W.BF16)
        oracle.update(C, trees[b], topk)
        assert acc.cpu().numpy()[b] == a and np.array_equal(out.cpu().numpy()[b], o)
    assert np.array_equal(eng.get_matrix(), C)
    eng.close()


def test_invalid_arguments_are_rejected():
    g_ = G()
    eng = g_.Graft(g_.graft_default_config(100, 2, 0, W.BF16))
    with pytest.raises(g_.GraftError):
        eng.verify_update(3, None, None, None, None, torch.empty((1, 100), device="cuda"), None, None)  # batch > max
    static = g_.Graft(g_.graft_default_config(100, 2, 1, W.BF16))
    ev = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(g_.GraftError):            # incremental drafting is for checkpoint mode
        static.check(2, torch.zeros((2, 4), dtype=torch.int16, device="cuda"),
                     torch.ones((2, 4), device="cuda"), 0, ev)
    with pytest.raises(g_.GraftError):
        eng.check(2, torch.zeros((2, 4), dtype=torch.int16, device="cuda"), torch.ones((2, 4), device="cuda"), -1, ev)
    tok = torch.full((2, eng.S), -1, dtype=torch.int32, device="cuda")    # a root (token 0) and pads
    tok[:, 0] = 0
    par = torch.full((2, eng.S), -1, dtype=torch.int8, device="cuda")
    pos = torch.full((2, eng.S), -1, dtype=torch.int32, device="cuda")
    pos[:, 0] = 0
    mask = torch.zeros((2, eng.S), dtype=torch.int64, device="cuda")
    mask[:, 0] = 1
    lg = torch.zeros((2 * eng.S, 100), dtype=torch.bfloat16, device="cuda")
    u, ur = torch.full((2, eng.S), 0.5, device="cuda"), torch.full((2,), 0.5, device="cuda")
    acc = torch.empty(2, dtype=torch.int32, device="cuda")
    out = torch.empty((2, eng.S), dtype=torch.int32, device="cuda")
    for temp in (0.0, -1.0, float("inf"), float("nan"), 1e-39):   # the last: a subnormal with an infinite inverse
        with pytest.raises(g_.GraftError):
            eng.verify_update_sample(2, tok, par, pos, mask, lg, temp, u, ur, acc, out)
    eng.verify_update_sample(2, tok, par, pos, mask, lg, 1e-30, u, ur, acc, out)     # tiny but invertible
    assert eng.sync() == 0
    # raw calls past the binding: buffers off their element alignment are refused before anything is queued
    from hybrid_draft_tree_gb300 import graft as gb
    L = g_.load()
    p = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    args = [p(tok), p(par), p(pos), p(mask), p(lg), ctypes.c_int64(100), p(acc), p(out), ctypes.c_void_p(0)]
    assert L.graft_verify_update(eng.h, 2, *args) == gb.GRAFT_OK
    for i, off in ((0, 2), (2, 2), (3, 4), (4, 1), (6, 2), (7, 2)):
        bad = list(args)
        bad[i] = p([tok, par, pos, mask, lg, None, acc, out][i], off)
        assert L.graft_verify_update(eng.h, 2, *bad) == gb.GRAFT_EINVAL, (i, off)
    assert eng.sync() == 0
    for mode, kw in ((0, dict(topk=4)), (1, dict(ablation=1)), (2, dict(ablation=2)), (0, dict(ablation=3)),
                     (0, dict(ablation=2, fixed_draft=61)), (0, dict(tpl_width=65)), (0, dict(tpl_depth=17)),
                     (0, dict(scan_kernel=6)), (0, dict(scan_kernel=-1))):
        with pytest.raises(g_.GraftError):
            g_.Graft(g_.graft_default_config(100, 2, mode, W.BF16, **kw))


@pytest.mark.parametrize("B,sample", [(4, False), (1, False), (4, True), (1, True)])
def test_step_replays_from_a_cuda_graph(B, sample):
    """assemble + verify_update (or verify_update_sample, on fixed uniforms)
    are captured into a CUDA graph and replayed: the same trees, acceptance
    and matrix as the same calls made directly on an identical handle.  Four
    requests take the two-pass scan (with the dependent launch of pass 2, and
    the walk's clusters as its dependent), one request the cluster-per-row
    verify."""
    from workloads.device_loop import DeviceLoop
    w = W.WORKLOADS[2].scaled(V=40000, B=B)
    eager = engine_for(w)
    graphed = engine_for(w)
    loop = DeviceLoop(w, eager)
    for _ in range(3):                                 # fill the matrix a little
        loop.step()
    graphed.set_matrix(eager.get_matrix())
    loop.draft()
    side = torch.cuda.Stream()
    outs = {}
    for name, eng in (("eager", eager), ("graph", graphed)):
        bufs = [torch.empty_like(t) for t in (loop.tok, loop.par, loop.pos, loop.mask, loop.info)]
        acc = torch.empty_like(loop.accept_len)
        out = torch.empty_like(loop.out_tokens)
        par = loop.d_par

        u = torch.linspace(0.05, 0.95, w.B * w.S, device="cuda").view(w.B, w.S)
        ur = torch.linspace(0.1, 0.9, w.B, device="cuda")

        def step():
            eng.assemble(w.B, loop.root, loop.d_tok, par, loop.d_aux, *bufs, stream=torch.cuda.current_stream())
            if sample:
                eng.verify_update_sample(w.B, bufs[0], bufs[1], bufs[2], bufs[3], loop.logits, 1.0, u, ur, acc, out,
                                         stream=torch.cuda.current_stream())
            else:
                eng.verify_update(w.B, bufs[0], bufs[1], bufs[2], bufs[3], loop.logits, acc, out,
                                  stream=torch.cuda.current_stream())
        if name == "graph":
            with torch.cuda.stream(side):
                step()                                 # first call on the stream: nothing new is set up in capture
            side.synchronize()
            graphed.set_matrix(eager_matrix_before)
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_, stream=side):
                step()
            g_.replay()
        else:
            eager_matrix_before = eager.get_matrix()
            loop.assemble()                            # logits of this step's tree (same tree as both will build)
            loop.make_logits()
            step()
        torch.cuda.synchronize()
        outs[name] = [t.clone() for t in bufs] + [acc.clone(), out.clone(), torch.from_numpy(eng.get_matrix())]
    for x, y in zip(outs["eager"], outs["graph"]):
        assert torch.equal(x, y)
    assert eager.sync() == 0 and graphed.sync() == 0
    eager.close()
    graphed.close()


def test_profile_api_reports_each_kernel():
    """Tracing: every kernel of a step is bracketed by events and reported."""
    from workloads.device_loop import DeviceLoop
    w = W.WORKLOADS[2].scaled(V=40000, B=4)
    eng = engine_for(w)
    loop = DeviceLoop(w, eng)
    eng.profile_enable(True)
    loop.draft()
    loop.assemble()
    loop.make_logits()
    loop.verify_update()
    rec = eng.profile_read()
    names = [n for n, _ in rec]
    assert names == ["k_assemble", "k_umax", "k_select"], names
    assert all(ms > 0 for _, ms in rec)
    assert eng.profile_read() == []
    eng.profile_enable(False)
    loop.assemble()
    assert eng.profile_read() == []
    eng.close()
