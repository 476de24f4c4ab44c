"""The seeded input generators follow their stated recipe (CPU): the
counter-based hash is SplitMix64, logits noise is an exact Irwin-Hall(12)
normal rounded to bf16 by round-to-nearest-even, draft trees have the stated
shape and a softmax per sibling group, a target row is a pure function of its
token prefix, and the warm-start history draws from its active set.  The
generators hold none of the method's arithmetic; these tests pin the inputs
both sides consume, not the method."""
import numpy as np
import pytest

import workloads as W


def test_hash_is_splitmix64():
    """syn_sm64(x) is one SplitMix64 step from state x (Steele, Lea and Flood,
    2014): from state 0 the generator's first three outputs are the published
    0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F."""
    gamma = 0x9E3779B97F4A7C15
    got = [W.host().syn_sm64((i * gamma) % 2**64) for i in range(3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def _noise_rows(n, V, dtype, seed=5):
    rk = np.array([W.host().syn_sm64(seed * 1000 + i) for i in range(n)], np.uint64)
    planted = np.full(n, -1, np.int32)                  # no planted successor: pure noise
    bias = np.zeros(n, np.float32)
    return W.fill_rows(rk, planted, bias, V, dtype)


def test_logits_noise_is_an_exact_irwin_hall_normal():
    """z = (2 * sum of 12 16-bit uniforms - 12 * 65535) / 2^17: a multiple of
    2^-17 in [-6, 6] with mean 0 and variance 1 (each uniform has variance
    (2^32 - 1) / 12)."""
    z = _noise_rows(8, 32000, W.F32).astype(np.float64).ravel()
    k = z * 2.0**17
    assert np.array_equal(k, np.round(k))
    assert np.all(np.abs(z) <= 12 * 65535 / 2.0**17)
    assert abs(z.mean()) < 0.005
    assert abs(z.std() - 1.0) < 0.005


def test_bf16_rows_are_the_f32_rows_rounded_to_nearest_even():
    f = _noise_rows(4, 5000, W.F32)
    b = _noise_rows(4, 5000, W.BF16)
    u = f.view(np.uint32).astype(np.uint64)
    rne = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(b, rne)


def test_planted_successor_carries_the_bias():
    rk = np.array([W.host().syn_sm64(77)], np.uint64)
    noise = W.fill_rows(rk, np.array([-1], np.int32), np.zeros(1, np.float32), 1000, W.F32)
    planted = W.fill_rows(rk, np.array([123], np.int32), np.array([6.0], np.float32), 1000, W.F32)
    diff = planted - noise
    assert diff[0, 123] == np.float32(noise[0, 123] + np.float32(6.0)) - noise[0, 123]
    assert np.count_nonzero(diff) == 1


@pytest.mark.parametrize("wid", [0, 2, 3])
def test_draft_tree_shape_and_sibling_softmax(wid):
    """Full branching 4/3/2/2/1/1 (184 nodes) in BFS order; each sibling
    group's probabilities are a softmax (sum 1), sorted descending; sibling
    tokens are distinct and in range."""
    w = W.WORKLOADS[wid]
    h = W.Harness(w)
    root, prev, ctx = h.init_state()
    tok, par, prob = h.draft(3, root, prev)
    for b in range(w.B):
        p = par[b].astype(np.int64)
        assert p[0] == -1 and all(-1 <= p[i] < i for i in range(len(p)))
        depth = np.zeros(len(p), np.int64)
        for i in range(len(p)):
            depth[i] = 0 if p[i] < 0 else depth[p[i]] + 1
        assert [int((depth == d).sum()) for d in range(6)] == [4, 12, 24, 48, 48, 48]
        assert np.all((tok[b] >= 0) & (tok[b] < w.V))
        for parent in np.unique(p):
            kids = np.flatnonzero(p == parent)
            pk = prob[b][kids].astype(np.float64)
            assert abs(pk.sum() - 1.0) < 1e-5
            assert np.all(np.diff(pk) <= 0)
            assert len(set(tok[b][kids].tolist())) == len(kids)


def test_target_row_is_a_pure_function_of_the_prefix():
    """The same token path at different slots of different trees gets the
    same row parameters, and so the same logits row."""
    w = W.WORKLOADS[2].scaled(V=5000, B=1)
    h = W.Harness(w)
    root, prev, ctx = h.init_state()
    S = w.S
    a_tok, a_par = np.full((1, S), -1, np.int32), np.full((1, S), -1, np.int8)
    b_tok, b_par = np.full((1, S), -1, np.int32), np.full((1, S), -1, np.int8)
    a_tok[0, :3], a_par[0, :3] = [root[0], 11, 22], [-1, 0, 1]              # root -> 11 -> 22 at slots 0, 1, 2
    b_tok[0, :5], b_par[0, :5] = [root[0], 33, 11, 44, 22], [-1, 0, 0, 1, 2]  # the same path at slots 0, 2, 4
    ra = h.tree_rowparams(a_tok, a_par, ctx, prev)
    rb = h.tree_rowparams(b_tok, b_par, ctx, prev)
    for x, y in zip(ra, rb):
        assert x[0, 0] == y[0, 0] and x[0, 1] == y[0, 2] and x[0, 2] == y[0, 4]
    la = h.tree_logits(a_tok, a_par, ctx, prev)
    lb = h.tree_logits(b_tok, b_par, ctx, prev)
    assert np.array_equal(la[0, 2], lb[0, 4]) and not np.array_equal(la[0, 1], lb[0, 1])


def test_tail_blocks():
    w = W.WORKLOADS[4]
    h = W.Harness(w)
    root, prev, ctx = h.init_state()
    tok, par, conf = h.draft(0, root, prev)
    assert par is None and tok.shape == conf.shape == (w.B, 16)
    assert np.all((conf > 0) & (conf < 1)) and np.all((tok >= 0) & (tok < w.V))


def test_warm_start_history_uses_its_active_set():
    w = W.WORKLOADS[3]
    h = W.Harness(w)
    assert len(h.hist) == 32768 and len(np.unique(h.active)) == 2000
    assert set(np.unique(h.hist).tolist()) <= set(h.active.tolist())
    toks, rk, pl, bi = h.warm_rowparams()
    assert np.array_equal(toks, h.hist) and len(rk) == 32768
