"""Full-size, full-length parity: the CUDA library (through its C ABI) in
lock-step with the CPU oracle on the five workloads at their stated sizes
and decode lengths (100, 1000, 500, 200 and 300 steps), in the launch
configuration the benchmark times.  After every step the trees, positions,
masks, info records, acceptance lengths, emitted tokens and the WHOLE
continuation matrix are compared bit for bit; the matrix carries every
step's update into the next (popular-science article on arXiv 2605.20104,
section 二 third gear: every verified row rewrites its token's successors, so
a wrong row would surface in later trees).

The oracle holds its own matrix from the first step on; nothing of the GPU's
state is fed back into it.  Its logits come from the host generator of the
seeded inputs, driven by the oracle's own trees (rows filled by all host
threads; every row is a pure function of its key).  The oracle's
per-request top-8 scans run in a thread pool (independent requests, the GIL
released inside the C calls); its matrix updates run in (request, slot)
order on one thread, as the method states.
"""
import concurrent.futures as cf

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(scope="module")
def pool():
    oracle.lib()                                  # load once, before any thread calls it
    W.host()
    ex = cf.ThreadPoolExecutor(W.host_threads())
    yield ex
    ex.shutdown()


def engine_for(w):
    import hybrid_draft_tree_gb300 as g
    cfg = g.graft_default_config(w.V, w.B, w.mode, w.dtype, budget=w.budget, max_draft_nodes=w.draft_nodes)
    return g.Graft(cfg)


def oracle_logits(loop, trees):
    """Logits [B, S, V] of the oracle's own trees, from the host generator."""
    tt = np.stack([t.tok for t in trees])
    pp = np.stack([t.par for t in trees]).astype(np.int8)
    return loop.h.tree_logits(tt, pp, loop.ctx_h, loop.prev_h, threads=W.host_threads())


def assert_trees_equal(loop, trees, step):
    gt = loop.tok.cpu().numpy()
    gp = loop.par.cpu().numpy().astype(np.int32)
    gpos = loop.pos.cpu().numpy()
    gm = loop.mask.cpu().numpy().view(np.uint64)
    gi = loop.info.cpu().numpy()
    for b, tr in enumerate(trees):
        assert np.array_equal(gt[b], tr.tok), (step, b, "tok")
        assert np.array_equal(gp[b], tr.par), (step, b, "parent")
        assert np.array_equal(gpos[b], tr.pos), (step, b, "pos")
        assert np.array_equal(gm[b], tr.mask), (step, b, "mask")
        assert np.array_equal(gi[b], tr.info), (step, b, "info", gi[b], tr.info)


def decode_lockstep(w, g, loop, C, steps, pool):
    """`steps` decode steps of the GPU loop and the oracle side by side, the
    oracle on its own matrix C (updated in place).  Returns per-step
    statistics (events, accepted lengths)."""
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode)
    events, accepted = [], []
    for step in range(steps):
        tok, par, aux = loop.draft()
        loop.assemble()
        trees = [oracle.assemble(P, loop.root_h[b], tok[b], aux[b], C, None if par is None else par[b])
                 for b in range(w.B)]
        assert_trees_equal(loop, trees, step)
        loop.make_logits()
        lg = oracle_logits(loop, trees)
        loop.verify_update()
        res = list(pool.map(lambda b: oracle.verify(trees[b], lg[b], w.dtype), range(w.B)))
        acc_g = loop.accept_len.cpu().numpy()
        out_g = loop.out_tokens.cpu().numpy()
        for b, (acc, out, topk) in enumerate(res):
            oracle.update(C, trees[b], topk)
            assert acc_g[b] == acc, (step, b, "accept_len", acc_g[b], acc)
            assert np.array_equal(out_g[b], out), (step, b, "out_tokens", out_g[b], out)
            events.append(int(trees[b].info[0]))
            accepted.append(acc)
        assert np.array_equal(g.get_matrix(), C), (step, "matrix")
        loop.advance()
    assert g.sync() == 0
    return events, accepted


@pytest.mark.parametrize("wid", [0, 1, 2, 4])
def test_lockstep_full_size_full_length(wid, pool):
    """Workloads 0 (fp32 V = 32000, 100 steps), 1 (V = 128256 with its
    1280-row warm-up, 1000 steps), 2 (the headline: 16 requests x 61 slots,
    V = 151936, static trees, 500 steps) and 4 (64 blocks x 17 slots, tail
    grafts, 300 steps), each at its stated length."""
    from workloads.device_loop import DeviceLoop
    w = W.WORKLOADS[wid]
    g = engine_for(w)
    loop = DeviceLoop(w, g)
    C = oracle.new_matrix(w.V)
    if w.warm == "rollouts":
        toks_d, logits_d, (toks, rk, pl, bi) = loop.warm_inputs_device()
        g.warmup(toks_d, logits_d)
        rows = W.fill_rows(rk, pl, bi, w.V, w.dtype, threads=W.host_threads())
        oracle.warmup(C, toks, rows, w.dtype)
        assert np.array_equal(g.get_matrix(), C), "matrix after warm-up"
        del logits_d, rows
        torch.cuda.empty_cache()
    events, accepted = decode_lockstep(w, g, loop, C, w.steps, pool)
    assert sum(accepted) > 0
    if w.mode == W.MODE_STATIC:
        assert any(e > 0 for e in events)          # some slots were replaced in place
    g.close()


def test_warm_start_32k_full_size(pool):
    """Workload 3: the 32768-row warm start at V = 151936 (9.96 GB of bf16
    logits on the device), then its 200 decode steps.  The oracle loads
    every row in order into its own matrix (chunk by chunk: rows overwrite in
    order, so consecutive calls equal one call); the GPU's matrix must equal
    it everywhere, which covers every written row and every untouched one.
    Decoding then continues from each side's own matrix."""
    from workloads.device_loop import DeviceLoop
    w = W.WORKLOADS[3]
    g = engine_for(w)
    loop = DeviceLoop(w, g)
    toks_d, logits_d, (toks, rk, pl, bi) = loop.warm_inputs_device()
    g.warmup(toks_d, logits_d)
    del logits_d
    torch.cuda.empty_cache()
    C = oracle.new_matrix(w.V)
    n = len(toks)
    chunk = 2048
    buf = np.empty((chunk, w.V), np.uint16)
    for r0 in range(0, n, chunk):
        r1 = min(n, r0 + chunk)
        rows = W.fill_rows(rk[r0:r1], pl[r0:r1], bi[r0:r1], w.V, w.dtype, out=buf[:r1 - r0],
                           threads=W.host_threads())
        oracle.warmup(C, toks[r0:r1], rows, w.dtype)
    Cg = g.get_matrix()
    distinct = len(set(toks.tolist()))
    assert int((C[:, 0] >= 0).sum()) == distinct
    assert np.array_equal(Cg, C), "matrix after the 32K warm start"
    events, accepted = decode_lockstep(w, g, loop, C, w.steps, pool)
    assert sum(accepted) > 0
    g.close()
