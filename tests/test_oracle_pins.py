"""Pins of the CPU oracle against things other than itself: library sorts,
brute force on tiny inputs, closed forms, the pages' budget table, and the
pages' invariants (losslessness, the superset / monotonicity argument).

Sources: popular-science article on arXiv 2605.20104, sections 二 (three
gears), 三 (monotonicity and superset argument), 四 (static trees), 五
(ablations), 六 (warm-up), 七 (Graft-TAIL); Hugging Face paper page
2605.20104, abstract.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_to_f32(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def lexsort_topk(vals, k=8):
    """Stable library sort: value descending, id ascending."""
    ids = np.arange(len(vals))
    order = np.lexsort((ids, -vals.astype(np.float64)))
    out = np.full(k, -1, np.int32)
    out[:min(k, len(vals))] = order[:k]
    return out


# ----------------------------------------------------------------------------- top-k
@pytest.mark.parametrize("V", [1, 5, 8, 9, 16, 33, 64, 257])
@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_stable_sort_f32_with_ties(V, seed):
    rng = np.random.default_rng(seed * 1000 + V)
    vals = rng.integers(-3, 4, V).astype(np.float32)       # heavy ties
    vals[rng.random(V) < 0.2] = -0.0                         # -0 must tie with +0
    vals[rng.random(V) < 0.05] = np.inf
    vals[rng.random(V) < 0.05] = -np.inf
    assert np.array_equal(oracle.topk8_row(vals, oracle.F32), lexsort_topk(vals))


@pytest.mark.parametrize("seed", range(8))
def test_topk_matches_stable_sort_bf16(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(8, 400))
    f = rng.normal(size=V).astype(np.float32)
    u = (f.view(np.uint32) >> 16).astype(np.uint16)            # truncation: many ties after rounding
    u[rng.random(V) < 0.1] = 0x8000                            # -0.0
    u[rng.random(V) < 0.1] = 0x0000
    assert np.array_equal(oracle.topk8_row(u, oracle.BF16), lexsort_topk(bf16_to_f32(u)))


def test_topk_nan_is_an_error():
    v = np.zeros(16, np.float32)
    v[3] = np.nan
    with pytest.raises(oracle.OracleError):
        oracle.topk8_row(v, oracle.F32)


def test_argmax_tie_goes_to_lower_id():
    v = np.array([0, 2, 1, 2, 2], np.float32)
    assert oracle.topk8_row(v, oracle.F32)[0] == 1
    v = np.array([0.0, -0.0, -1.0], np.float32)
    assert list(oracle.topk8_row(v, oracle.F32)[:3]) == [0, 1, 2]


# ----------------------------------------------------------------------------- template
def _paths(par, rank):
    out = []
    for j in range(len(par)):
        p, q = [], j
        while q >= 0:
            p.append(int(rank[q]))
            q = par[q]
        out.append(tuple(reversed(p)))
    return out


def test_template_closed_form_counts_and_order():
    """Paths with rank sum 0 number 8 (one per depth 1..8); sum 1 has d paths
    at depth d (the position of the single 1); sum 2 has d + C(d,2) at depth
    d (one 2, or two 1s).  The order is (sum, depth, rank path)."""
    par, rank, dep = oracle.template(200)
    paths = _paths(par, rank)
    keys = [(sum(p), len(p), p) for p in paths]
    assert keys == sorted(keys)
    assert len(set(paths)) == len(paths)
    for s, count_at in [(0, lambda d: 1), (1, lambda d: d), (2, lambda d: d + math.comb(d, 2))]:
        for d in range(1, 9):
            got = sum(1 for p in paths if sum(p) == s and len(p) == d)
            assert got == count_at(d), (s, d, got)
    # first sum-2 entries follow the 44 entries of sums 0 and 1
    assert paths[:8] == [(0,) * d for d in range(1, 9)]
    assert paths[8:11] == [(1,), (0, 1), (1, 0)]
    assert paths[44:52] == [(2,), (0, 2), (1, 1), (2, 0), (0, 0, 2), (0, 1, 1), (0, 2, 0), (1, 0, 1)]


def test_template_structure():
    par, rank, dep = oracle.template(52)
    assert len(par) == 52
    for j in range(52):
        assert dep[j] <= 8
        if par[j] < 0:
            assert dep[j] == 1 and rank[j] < 8               # root width 8
        else:
            assert par[j] < j and dep[j] == dep[par[j]] + 1  # parents first
            assert rank[j] < max(1, 8 >> rank[par[j]])       # fan-out max(1, 8 >> r)
    # truncation is a prefix of the longer template
    p2, r2, d2 = oracle.template(20)
    assert np.array_equal(p2, par[:20]) and np.array_equal(r2, rank[:20])


def test_template_width_and_depth_parameters():
    par, rank, dep = oracle.template(60, depth=2, width=4)
    paths = _paths(par, rank)
    assert max(len(p) for p in paths) <= 2
    for p in paths:
        assert p[0] < 4
        for a, b in zip(p, p[1:]):
            assert b < max(1, 4 >> a)
    # depth 2, width 4: 4 roots; children 4, 2, 1, 1 -> 4 + 8 = 12 paths in total
    assert len(paths) == 12


# ----------------------------------------------------------------------------- conf / budget
def test_path_conf_is_product_along_path():
    rng = np.random.default_rng(1)
    h = W.Harness(W.WORKLOADS[0])
    root, prev, ctx = h.init_state()
    tok, par, prob = h.draft(3, root, prev)
    conf, depth = oracle.path_conf(par[0], prob[0])
    for i in rng.choice(len(conf), 40, replace=False):
        prod, j, d = 1.0, i, -1
        while j >= 0:
            prod *= float(prob[0][j])
            j = par[0][j]
            d += 1
        assert depth[i] == d
        assert abs(conf[i] - prod) <= 1e-6 * prod


def _budget_table():
    rows = {}
    with open(os.path.join(GOLDEN, "budget_table.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                d, a, b = map(int, line.split())
                rows[d] = (a, b)
    return rows


def _layered_tree(layer_probs, branching=(4, 3, 2, 2, 1, 1), V=1000):
    """Full tree whose layer-d nodes all have probability layer_probs[d]
    except node 0 of each layer, given layer_probs[d] * boost."""
    tok, par, prob = [], [], []
    prev_layer = [-1]
    t = 10
    for d, g in enumerate(branching):
        cur = []
        for p in prev_layer:
            for _ in range(g):
                cur.append(len(tok))
                tok.append(t)
                t += 1
                par.append(p)
                prob.append(layer_probs[d])
        prev_layer = cur
    return np.array(tok, np.int32), np.array(par, np.int16), np.array(prob, np.float32)


def test_checkpoint_firing_and_budget_table():
    """Hand-built trees that make each checkpoint fire; the slot split must be
    the pages' table, and the kept draft count min(D, nodes in layers <= d)."""
    table = _budget_table()
    for (d, a), (dd, b) in itertools.product(table.items(), table.items()):
        if d >= 0:
            assert a[0] + a[1] == 60
    V = 1000
    P = oracle.make_params(V)
    C = oracle.new_matrix(V)
    C[:, :] = (np.arange(V)[:, None] * 7 + np.arange(8)[None, :]) % V   # every retrieval realised
    cases = {
        0: [0.25, 1, 1, 1, 1, 1],            # best layer-0 conf 0.25 < 0.30
        1: [0.5, 0.3, 1, 1, 1, 1],           # layer 0: 0.5 ; layer 1: 0.15 < 0.20
        5: [0.9, 0.5, 0.5, 0.5, 0.6, 0.6],   # layer 5: 0.9*.5^3*.36 = 0.0405 < 0.10
        -1: [0.9, 0.9, 0.9, 0.9, 0.9, 0.9],  # nothing fires
    }
    avail = {0: 4, 1: 16, 5: 184, -1: 184}
    for d, probs in cases.items():
        tok, par, prob = _layered_tree(probs)
        tr = oracle.assemble(P, 5, tok, prob, C, par)
        D, R = table[d]
        assert tr.info[0] == d
        assert tr.info[1] == min(D, avail[d])
        assert tr.info[2] == R                                      # all retrieval realised
        assert tr.info[3] == 1 + tr.info[1] + tr.info[2] <= 61


def _brute_force_template(depth, width):
    """Every rank path of the template by exhaustive product over ranks,
    kept when each step obeys the fan-out (anchor: min(8, width); after rank
    r: min(8, max(1, width >> r))), in the order (rank sum, depth, path)."""
    paths = []
    for d in range(1, depth + 1):
        for p in itertools.product(range(8), repeat=d):
            if p[0] >= min(8, width):
                continue
            if all(b < min(8, max(1, width >> a)) for a, b in zip(p, p[1:])):
                paths.append(p)
    return sorted(paths, key=lambda p: (sum(p), len(p), p))


@pytest.mark.parametrize("depth", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("width", [1, 2, 3, 4, 8, 16])
def test_template_equals_brute_force_enumeration(depth, width):
    want = _brute_force_template(depth, width)
    for R in sorted({1, 7, 20, 52, min(len(want), 256)}):
        par, rank, dep = oracle.template(R, depth=depth, width=width)
        assert _paths(par, rank) == want[:R], (depth, width, R)
        assert list(dep) == [len(p) for p in want[:R]]


def test_template_width_above_eight_and_deep_chains():
    # width 16: the anchor's ranks are capped at the matrix row's 8; rank-r
    # nodes have min(8, max(1, 16 >> r)) children: 8+8+4+2+1+1+1+1 = 26
    par, rank, dep = oracle.template(60, depth=2, width=16)
    assert len(par) == 8 + 26
    # depth 12: the 12 rank-0 chain entries (rank sum 0) come first
    par, rank, dep = oracle.template(20, depth=12, width=8)
    assert list(dep[:12]) == list(range(1, 13)) and not rank[:12].any()
    assert list(par[:12]) == [-1] + list(range(11))


# ----------------------------------------------------------------------------- ablations (section 五)
def test_no_retrieval_ablation_is_the_pruned_tree():
    """Pruning without retrieval: the same tree as Graft with nothing to
    retrieve (the pruned slots stay empty), whatever the matrix holds."""
    V = 1000
    full = oracle.new_matrix(V)
    full[:, :] = (np.arange(V)[:, None] * 7 + np.arange(8)[None, :]) % V
    for probs in ([0.25, 1, 1, 1, 1, 1], [0.5, 0.3, 1, 1, 1, 1], [0.9, 0.5, 0.5, 0.5, 0.6, 0.6], [0.9] * 6):
        tok, par, prob = _layered_tree(probs)
        a = oracle.assemble(oracle.make_params(V, ablation=1), 5, tok, prob, full, par)
        b = oracle.assemble(oracle.make_params(V), 5, tok, prob, oracle.new_matrix(V), par)
        for x, y in ((a.tok, b.tok), (a.par, b.par), (a.pos, b.pos), (a.mask, b.mask), (a.info, b.info)):
            assert np.array_equal(x, y)
        assert a.info[2] == 0


@pytest.mark.parametrize("D", [0, 8, 40, 60])
def test_fixed_split_keeps_the_top_d_of_the_whole_tree(D):
    """No adaptive pruning: the top-D nodes of the whole tree by path
    confidence (ties: lower index), then budget - D retrieval slots, every
    step; no checkpoint is reported."""
    V = 500
    h = W.Harness(W.WORKLOADS[0].scaled(V=V, draft_sigma=0.75))
    root, prev, ctx = h.init_state()
    C = oracle.new_matrix(V)
    C[:, :] = (np.arange(V)[:, None] * 3 + np.arange(8)[None, :] * 5 + 1) % V
    for step in range(6):
        tok, par, prob = h.draft(step, root, prev)
        tok, par, prob = tok[0], par[0], prob[0]
        conf = np.zeros(len(tok), np.float32)
        for i in range(len(tok)):                       # fp32 product, root first
            conf[i] = prob[i] if par[i] < 0 else np.float32(conf[par[i]] * prob[i])
        kept = np.sort(np.lexsort((np.arange(len(tok)), -conf.astype(np.float64)))[:D])
        tr = oracle.assemble(oracle.make_params(V, ablation=2, fixed_draft=D), int(root[0]), tok, prob, C, par)
        assert tr.info[0] == -1 and tr.info[1] == D
        assert list(tr.tok[1:1 + D]) == list(tok[kept])
        assert tr.info[2] == 60 - D                     # the full matrix realises every entry


@pytest.mark.parametrize("ablation", [1, 2])
def test_ablations_are_lossless(ablation):
    w = W.WORKLOADS[0].scaled(V=600, B=1, draft_sigma=0.75)
    emitted, accs, _ = _run_loop(w, 10, ablation=ablation)
    assert emitted[0] == _greedy(w, 0, len(emitted[0]))


# ----------------------------------------------------------------------------- incremental drafting
def _np_conf(par, prob):
    conf = np.zeros(len(par), np.float32)
    depth = np.zeros(len(par), np.int32)
    for i in range(len(par)):                       # fp32 product, root first
        conf[i] = prob[i] if par[i] < 0 else np.float32(conf[par[i]] * prob[i])
        depth[i] = 0 if par[i] < 0 else depth[par[i]] + 1
    return conf, depth


@pytest.mark.parametrize("sigma", [0.5, 0.75, 2.0])
def test_incremental_checkpoints_match_brute_force(sigma):
    """Checkpoints evaluated layer by layer as the drafter completes them:
    the first checkpoint (in order 0, 1, 5) whose layer's best path
    confidence is below its threshold fires, and its verdict never changes."""
    V = 400
    h = W.Harness(W.WORKLOADS[0].scaled(V=V, draft_sigma=sigma))
    root, prev, ctx = h.init_state()
    P = oracle.make_params(V)
    for step in range(12):
        tok, par, prob = h.draft(step, root, prev)
        par, prob = par[0], prob[0]
        conf, depth = _np_conf(par, prob)
        expect = -1
        for d, thr in zip((0, 1, 5), (0.30, 0.20, 0.10)):
            layer = conf[depth == d]
            if len(layer) and layer.max() < np.float32(thr):
                expect = d
                break
        ev = ev_full = -1
        for L in range(6):
            n = int((depth <= L).sum())
            ev = oracle.check_layer(P, par[:n], prob[:n], L, ev)
            # the whole tree given early: layers past L are present but their
            # checkpoints are not evaluated yet
            ev_full = oracle.check_layer(P, par, prob, L, ev_full)
            if expect >= 0 and L >= expect:
                assert ev == expect and ev_full == expect
            elif L < (expect if expect >= 0 else 99):
                assert ev == -1 and ev_full == -1
        assert ev == expect
        assert oracle.assemble(P, int(root[0]), tok[0], prob, oracle.new_matrix(V), par).info[0] == expect


def test_retrieve_is_the_template_gather_of_the_fired_split():
    V = 64
    C = ((np.arange(V)[:, None] * 3 + np.arange(8)[None, :] * 11) % V).astype(np.int32)
    C[C[9, 0], 1] = -1                                # entry "01" is empty: its subtree is not realised
    P = oracle.make_params(V)
    for event, R in ((-1, 0), (0, 52), (1, 36), (5, 20)):
        out = oracle.retrieve(P, 9, event, C)
        tp, trk, td = oracle.template(R)
        ent = []
        for j in range(R):
            ptok = 9 if tp[j] < 0 else ent[tp[j]]
            ent.append(-1 if ptok < 0 else int(C[ptok, trk[j]]))
        assert list(out[:R]) == ent and (out[R:] == -1).all()
    assert (oracle.retrieve(oracle.make_params(V, ablation=1), 9, 0, C) == -1).all()
    assert (oracle.retrieve(oracle.make_params(V, ablation=2, fixed_draft=50), 9, -1, C)[:10] != -1).any()


# ----------------------------------------------------------------------------- coverage gain (section 三)
def _coverage_case():
    """Root 0 with kept draft children 10, 11 (slots 1, 2) and a kept draft
    grandchild 12 under slot 1 (slot 3); retrieved children 11, 12, 13 of the
    root (slots 4-6: 11 duplicates a drafted sibling, 12 only a drafted token
    elsewhere in the tree) plus a retrieved grandchild 14 (slot 7, not at the
    boundary)."""
    t = oracle.Tree(9)
    t.tok[:8] = [0, 10, 11, 12, 11, 12, 13, 14]
    t.par[:8] = [-1, 0, 0, 1, 0, 0, 0, 4]
    t.info[:] = [0, 3, 4, 8]
    return t


def test_coverage_of_a_uniform_row_counts_new_candidates():
    t = _coverage_case()
    V = 40
    rows = np.zeros((9, V), np.float32)
    assert abs(oracle.coverage(t, t.info, rows, oracle.F32) - 2 / V) < 1e-15   # 12 and 13 are new; 11 is not


# bfloat16 bit patterns of small integers (sign, 8 exponent bits with bias
# 127, 7 fraction bits): 0 -> 0x0000, 1 -> 0x3F80, 2 -> 0x4000, 3 -> 0x4040,
# 4 -> 0x4080, 5 -> 0x40A0, -1 -> 0xBF80, -2 -> 0xC000.
BF16_OF_INT = {0: 0x0000, 1: 0x3F80, 2: 0x4000, 3: 0x4040, 4: 0x4080, 5: 0x40A0, -1: 0xBF80, -2: 0xC000}


def _int_rows_both(shape, seed):
    """Integer logits in [-2, 5] as float32 and as bf16 bit patterns."""
    ints = np.random.default_rng(seed).integers(-2, 6, shape)
    bits = np.vectorize(BF16_OF_INT.get)(ints).astype(np.uint16)
    return ints.astype(np.float32), bits


@pytest.mark.parametrize("seed", range(4))
def test_coverage_of_bf16_rows_equals_their_values(seed):
    t = _coverage_case()
    f32, bits = _int_rows_both((9, 24), seed)
    x = f32[0].astype(np.float64)
    p = np.exp(x) / np.exp(x).sum()
    assert abs(oracle.coverage(t, t.info, bits, oracle.BF16) - (p[12] + p[13])) < 1e-12
    assert oracle.coverage(t, t.info, bits, oracle.BF16) == oracle.coverage(t, t.info, f32, oracle.F32)


def test_coverage_is_the_mass_of_the_new_tokens():
    t = _coverage_case()
    V = 40
    rows = np.full((9, V), -np.inf, np.float32)
    rows[0, 12] = 3.0
    assert oracle.coverage(t, t.info, rows, oracle.F32) == 1.0          # all the mass on a new candidate
    rows[0, 12], rows[0, 11] = -np.inf, 3.0
    assert oracle.coverage(t, t.info, rows, oracle.F32) == 0.0          # all of it on a drafted token
    rows[0, :] = np.log(np.arange(1, V + 1, dtype=np.float32))           # p(v) = (v + 1) / sum
    expect = (13 + 14) / (V * (V + 1) / 2)
    assert abs(oracle.coverage(t, t.info, rows, oracle.F32) - expect) < 1e-6 * expect   # fp32 logs of 1..V


# ----------------------------------------------------------------------------- stochastic verification
def _sample_tree():
    """Root (token 0) with children 2, 4, 2 (slots 1-3, a repeated token) and
    a grandchild 5 under slot 1 (slot 4)."""
    t = oracle.Tree(6)
    t.tok[:5] = [0, 2, 4, 2, 5]
    t.par[:5] = [-1, 0, 0, 0, 1]
    return t


def test_stochastic_verification_is_lossless():
    """Each emitted token is distributed as the target's softmax: the first
    as p(root row), the second, after the first was slot 1's token, as
    p(slot 1's row) -- Monte Carlo over seeded uniforms, 5-sigma bounds."""
    rng = np.random.default_rng(7)
    V = 6
    rows = rng.normal(0, 1, (6, V)).astype(np.float32)
    rows[0, 2] += 1.0
    t = _sample_tree()
    p0 = np.exp(rows[0].astype(np.float64) - rows[0].max()); p0 /= p0.sum()
    p1 = np.exp(rows[1].astype(np.float64) - rows[1].max()); p1 /= p1.sum()
    N = 20000
    first = np.zeros(V)
    second = np.zeros(V)
    n_after_2 = 0
    for _ in range(N):
        u = rng.random(6)
        acc, out, _ = oracle.verify_sample(t, rows, oracle.F32, 1.0, u, rng.random())
        first[out[0]] += 1
        if out[0] == 2 and acc >= 1:
            second[out[1]] += 1
            n_after_2 += 1
    for v in range(V):
        assert abs(first[v] / N - p0[v]) < 5 * np.sqrt(p0[v] * (1 - p0[v]) / N) + 1e-3, (v, first[v] / N, p0[v])
    # slot 1 (token 2) is tested before slot 3 (also 2), so an accepted 2 always descends into slot 1
    for v in range(V):
        m = n_after_2
        assert abs(second[v] / m - p1[v]) < 5 * np.sqrt(p1[v] * (1 - p1[v]) / m) + 2e-3, (v, second[v] / m, p1[v])


def test_stochastic_verification_of_bf16_rows_equals_their_values():
    """bf16 rows holding small integers walk exactly as the same values in
    float32 (whose walk the Monte Carlo pin above ties to the target)."""
    f32, bits = _int_rows_both((6, 8), 3)
    t = _sample_tree()
    rng = np.random.default_rng(11)
    for _ in range(300):
        u, ur = rng.random(6), rng.random()
        a32, o32, _ = oracle.verify_sample(t, f32, oracle.F32, 0.7, u, ur)
        a16, o16, _ = oracle.verify_sample(t, bits, oracle.BF16, 0.7, u, ur)
        assert a32 == a16 and np.array_equal(o32, o16)


@pytest.mark.parametrize("seed", range(10))
def test_stochastic_verification_at_low_temperature_is_greedy(seed):
    """As the temperature goes to 0 the target puts all its mass on the
    argmax, and on trees without repeated sibling tokens the walk accepts
    exactly the greedy path and emits the greedy bonus token."""
    rng = np.random.default_rng(seed)
    S, V = 16, 12
    rows = rng.normal(0, 1, (S, V)).astype(np.float32)
    t = oracle.Tree(S)
    t.tok[0], t.par[0] = 0, -1
    used = {}
    for i in range(1, S):
        p = int(rng.integers(0, i))
        cand = [v for v in range(V) if v not in used.setdefault(p, set())]
        tk = int(np.argmax(rows[p])) if rng.random() < 0.5 and np.argmax(rows[p]) in cand else int(rng.choice(cand))
        used[p].add(tk)
        t.tok[i], t.par[i] = tk, p
    acc_g, out_g, _ = oracle.verify(t, rows, oracle.F32)
    acc_s, out_s, _ = oracle.verify_sample(t, rows, oracle.F32, 1e4, rng.random(S) * 0.999, 0.5)
    assert acc_s == acc_g and np.array_equal(out_s, out_g)


def test_empty_matrix_gives_pruned_only_tree():
    V = 1000
    P = oracle.make_params(V)
    tok, par, prob = _layered_tree([0.25, 1, 1, 1, 1, 1])
    tr = oracle.assemble(P, 5, tok, prob, oracle.new_matrix(V), par)
    assert list(tr.info) == [0, 4, 0, 5]
    assert list(tr.tok[:5]) == [5] + list(tok[:4])


def test_retrieval_is_a_gather_along_the_template():
    V = 64
    P = oracle.make_params(V)
    C = ((np.arange(V)[:, None] * 3 + np.arange(8)[None, :] * 11) % V).astype(np.int32)
    tok, par, prob = _layered_tree([0.25, 1, 1, 1, 1, 1], V=V)
    tok %= V
    root = 9
    tr = oracle.assemble(P, root, tok, prob, C, par)
    tp, trk, td = oracle.template(52)
    base = 1 + 4
    ent_tok = []
    for j in range(52):
        ptok = root if tp[j] < 0 else ent_tok[tp[j]]
        ent_tok.append(C[ptok, trk[j]])
        s = base + j
        assert tr.tok[s] == ent_tok[j]
        assert tr.par[s] == (0 if tp[j] < 0 else base + tp[j])
        assert tr.pos[s] == td[j]


def test_unrealised_entry_drops_its_subtree():
    V = 64
    P = oracle.make_params(V)
    C = ((np.arange(V)[:, None] * 5 + np.arange(8)[None, :] * 3 + 1) % V).astype(np.int32)
    root = 9
    C[C[root, 0], 0] = -1          # entry "00" is empty -> "000".. chain and "001" etc vanish
    tok, par, prob = _layered_tree([0.25, 1, 1, 1, 1, 1], V=V)
    tr = oracle.assemble(P, root, tok % V, prob, C, par)
    tp, trk, td = oracle.template(52)
    paths = _paths(tp, trk)
    expected = sum(1 for p in paths if not (len(p) >= 2 and p[:2] == (0, 0)))
    assert tr.info[2] == expected


# ----------------------------------------------------------------------------- tree well-formedness
def _check_tree(tr, S):
    valid = tr.tok >= 0
    assert valid[0] and tr.pos[0] == 0 and tr.mask[0] == 1
    for i in range(1, S):
        if not valid[i]:
            assert tr.par[i] == -1 and tr.pos[i] == -1 and tr.mask[i] == 0
            continue
        p = tr.par[i]
        assert 0 <= p < i and valid[p]
        assert tr.pos[i] == tr.pos[p] + 1
        assert int(tr.mask[i]) == int(tr.mask[p]) | (1 << i)
        assert bin(int(tr.mask[i])).count("1") == tr.pos[i] + 1


@pytest.mark.parametrize("wid", [0, 2, 4])
def test_generated_trees_are_well_formed(wid):
    w = W.WORKLOADS[wid].scaled(V=512, B=2)
    h = W.Harness(w)
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode)
    C = oracle.new_matrix(w.V)
    rng = np.random.default_rng(wid)
    C[:] = rng.integers(-1, w.V, C.shape)
    root, prev, ctx = h.init_state()
    for step in range(6):
        tok, par, aux = h.draft(step, root, prev)
        for b in range(w.B):
            tr = oracle.assemble(P, root[b], tok[b], aux[b], C, None if par is None else par[b])
            _check_tree(tr, w.S)
            assert tr.info[3] == int((tr.tok >= 0).sum())


def test_static_mode_in_place_replacement():
    V = 50
    P = oracle.make_params(V, mode=oracle.MODE_STATIC)
    C = (np.arange(V)[:, None] * 100 + np.arange(8)[None, :]) % V
    C = C.astype(np.int32)
    # layer0 probs .9,.05,.03,.02; layer1 under node0 .1 (conf .09 < .15 -> replaced)
    tok, par, prob = _layered_tree([0.9, 0.1, 1, 1, 1, 1], V=V)
    prob[1:4] = [0.05, 0.03, 0.02]
    tok = tok % V
    tr = oracle.assemble(P, 7, tok, prob, C, par)
    # layer-0 node0 (slot 1) is kept with conf .9; its siblings are replaced with C[7][0..2]
    assert tr.tok[1] == tok[0]
    assert list(tr.tok[2:5]) == [C[7, 0], C[7, 1], C[7, 2]]
    # children of slot 1 (conf .09) are replaced with C[tok0][0], [1], [2]
    kids = [i for i in range(5, 61) if tr.par[i] == 1]
    assert [tr.tok[i] for i in kids] == [C[tok[0], s] for s in range(len(kids))]
    assert tr.info[3] == 61
    # an empty entry leaves the draft token in place; the slot count stays 61
    C2 = C.copy()
    C2[7, 1] = -1
    tr2 = oracle.assemble(P, 7, tok, prob, C2, par)
    assert tr2.tok[3] == tok[2]
    assert tr2.info[3] == 61 and tr2.info[2] == tr.info[2] - 1 - sum(
        1 for i in range(61) if tr.par[i] == 3)
    # children of the unreplaced slot 3 now gather from its draft token's row
    kids3 = [i for i in range(61) if tr2.par[i] == 3]
    assert [tr2.tok[i] for i in kids3] == [C2[tok[2], s] for s in range(len(kids3))]


def test_tail_mode():
    V = 100
    P = oracle.make_params(V, budget=16, mode=oracle.MODE_TAIL)
    C = ((np.arange(V)[:, None] * 13 + np.arange(8)[None, :] * 7 + 3) % V).astype(np.int32)
    btok = np.arange(20, 36, dtype=np.int32)
    conf = np.array([0.9, 0.8, 0.7, 0.35] + [0.9] * 12, np.float32)
    tr = oracle.assemble(P, 5, btok, conf, C)
    assert tr.info[0] == 3 and tr.info[1] == 3
    assert list(tr.tok[:4]) == [5, 20, 21, 22]
    tp, trk, td = oracle.template(13)
    ent = []
    for j in range(13):
        ptok = 22 if tp[j] < 0 else ent[tp[j]]
        ent.append(C[ptok, trk[j]])
        assert tr.tok[4 + j] == ent[j]
        assert tr.par[4 + j] == (3 if tp[j] < 0 else 4 + tp[j])
        assert tr.pos[4 + j] == 3 + td[j]
    conf[:] = 0.9
    tr = oracle.assemble(P, 5, btok, conf, C)
    assert list(tr.info) == [16, 16, 0, 17]
    conf[0] = 0.1
    tr = oracle.assemble(P, 5, btok, conf, C)
    assert tr.info[0] == 0 and tr.par[1] == 0 and tr.tok[1] == C[5, 0]


# ----------------------------------------------------------------------------- verification
def _random_tree(rng, S, V):
    tok = np.full(S, -1, np.int32)
    par = np.full(S, -1, np.int32)
    n = int(rng.integers(1, S + 1))
    tok[0] = rng.integers(0, V)
    for i in range(1, n):
        par[i] = rng.integers(0, i)
        tok[i] = rng.integers(0, V)
    t = oracle.Tree(S)
    t.tok[:] = tok
    t.par[:] = par
    return t


def _brute_accept(tok, par, vals):
    """Enumerate every root->node path; walk it step by step, accepting a
    token while it equals the target's argmax (lower id on ties) at the
    previous position.  Longest accepted prefix, lowest end slot on ties."""
    S = len(tok)
    arg = [int(lexsort_topk(vals[i])[0]) if tok[i] >= 0 else -1 for i in range(S)]
    best, best_end = 0, 0
    for end in range(S):
        if tok[end] < 0:
            continue
        path = []
        j = end
        while j != 0:
            path.append(j)
            j = par[j]
        path.reverse()
        ok = 0
        cur = 0
        for node in path:
            if tok[node] != arg[cur]:
                break
            ok += 1
            cur = node
        if ok == len(path) and ok > best:
            best, best_end = ok, end
    emitted = []
    j = best_end
    while j != 0:
        emitted.append(int(tok[j]))
        j = par[j]
    emitted.reverse()
    emitted.append(arg[best_end])
    return best, emitted


@pytest.mark.parametrize("seed", range(40))
def test_acceptance_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    S, V = int(rng.integers(2, 12)), int(rng.integers(2, 5))
    t = _random_tree(rng, S, V)
    vals = rng.integers(0, 3, (S, V)).astype(np.float32)     # many argmax ties
    # make the tree follow the target often
    for i in range(1, S):
        if t.tok[i] >= 0 and rng.random() < 0.6:
            t.tok[i] = lexsort_topk(vals[t.par[i]])[0]
    acc, out, topk = oracle.verify(t, vals, oracle.F32)
    best, emitted = _brute_accept(t.tok, t.par, vals)
    assert acc == best
    assert list(out[:acc + 1]) == emitted
    assert all(x == -1 for x in out[acc + 1:])


def test_pad_rows_are_not_read():
    t = oracle.Tree(4)
    t.tok[:] = [1, 0, -1, -1]
    t.par[:] = [-1, 0, -1, -1]
    vals = np.zeros((4, 3), np.float32)
    vals[2:] = np.nan
    acc, out, _ = oracle.verify(t, vals, oracle.F32)
    assert acc == 1 and list(out[:2]) == [0, 0]


# ----------------------------------------------------------------------------- closed loop invariants
def _run_loop(w, steps, C=None, retrieval=True, **params):
    h = W.Harness(w)
    P = oracle.make_params(w.V, budget=w.budget, mode=w.mode, **params)
    C = oracle.new_matrix(w.V) if C is None else C
    root, prev, ctx = h.init_state()
    emitted = [[] for _ in range(w.B)]
    accs = []
    for step in range(steps):
        tok, par, aux = h.draft(step, root, prev)
        Cuse = C if retrieval else oracle.new_matrix(w.V)

        def make_logits(trees):
            tt = np.stack([t.tok for t in trees])
            pp = np.stack([t.par for t in trees]).astype(np.int8)
            return h.tree_logits(tt, pp, ctx, prev)
        trees, res = oracle.step(P, Cuse, root, tok, aux, par, make_logits, w.dtype)
        outs = np.stack([r[1] for r in res])
        acc = np.array([r[0] for r in res], np.int32)
        accs.append(acc)
        for b in range(w.B):
            emitted[b].extend(outs[b][:acc[b] + 1].tolist())
        h.advance(root, prev, ctx, outs, acc)
    return emitted, accs, C


def _greedy(w, b, n):
    """Step-by-step greedy decoding of the synthetic target."""
    h = W.Harness(w)
    root, prev, ctx = h.init_state()
    r, p, c = int(root[b]), int(prev[b]), int(ctx[b])
    out = []
    for _ in range(n):
        rk, pl, bi = h.prefix_rowparams(b, c, p, r)
        row = W.fill_rows(rk, pl, bi, w.V, w.dtype)[0]
        vals = row if w.dtype == W.F32 else bf16_to_f32(row)
        nxt = int(np.argmax(vals))                               # first maximum = lower id
        out.append(nxt)
        p, r = r, nxt
        c = int(W.host().syn_ctx_push(c, nxt))
    return out


@pytest.mark.parametrize("wid,V,sigma", [(0, 700, 2.0), (0, 500, 0.75), (1, 900, 0.75), (2, 600, 2.0),
                                         (4, 800, 2.0)])
def test_lossless_equals_step_by_step_greedy(wid, V, sigma):
    """Tree decoding emits exactly the target's greedy sequence (lossless,
    article section 二 third gear)."""
    w = W.WORKLOADS[wid].scaled(V=V, B=min(W.WORKLOADS[wid].B, 2), draft_sigma=sigma)
    emitted, accs, _ = _run_loop(w, 12)
    for b in range(w.B):
        ref = _greedy(w, b, len(emitted[b]))
        assert emitted[b] == ref
    assert sum(int(a.sum()) for a in accs) > 0


def test_hybrid_tree_accepts_at_least_the_pruned_tree():
    """Superset argument (article section 三): the Graft tree contains every
    kept draft node, so with the same target its accepted length is never
    shorter than the pruned-only tree's."""
    w = W.WORKLOADS[0].scaled(V=300, B=1, draft_sigma=0.75)   # checkpoints fire often
    h = W.Harness(w)
    P = oracle.make_params(w.V)
    C = oracle.new_matrix(w.V)
    root, prev, ctx = h.init_state()
    wins = 0
    for step in range(40):
        tok, par, aux = h.draft(step, root, prev)
        hyb = oracle.assemble(P, root[0], tok[0], aux[0], C, par[0])
        pru = oracle.assemble(P, root[0], tok[0], aux[0], oracle.new_matrix(w.V), par[0])
        res = []
        for tr in (hyb, pru):
            lg = h.tree_logits(tr.tok[None], tr.par[None].astype(np.int8), ctx, prev)[0]
            res.append(oracle.verify(tr, lg, w.dtype))
        (a_h, out_h, topk_h), (a_p, _, _) = res
        assert a_h >= a_p
        wins += a_h > a_p
        oracle.update(C, hyb, topk_h)
        h.advance(root, prev, ctx, out_h[None], np.array([a_h], np.int32))
    assert wins > 0                     # retrieval does hit on this target


@pytest.mark.parametrize("seed", range(10))
def test_adding_nodes_never_shortens_acceptance(seed):
    """Monotonicity of tree verification (article section 三)."""
    rng = np.random.default_rng(seed)
    S, V = 16, 4
    vals = rng.integers(0, 3, (S, V)).astype(np.float32)
    t = _random_tree(rng, 10, V)
    n = int((t.tok >= 0).sum())
    big = oracle.Tree(S)
    big.tok[:10] = t.tok
    big.par[:10] = t.par
    for i in range(n, S):
        big.par[i] = rng.integers(0, i if i < n else n)
        big.tok[i] = rng.integers(0, V)
    big.tok[n:10] = big.tok[n:10]
    small = oracle.Tree(S)
    small.tok[:n] = t.tok[:n]
    small.par[:n] = t.par[:n]
    a_small = oracle.verify(small, vals, oracle.F32)[0]
    a_big = oracle.verify(big, vals, oracle.F32)[0]
    assert a_big >= a_small


def test_update_is_last_writer_topk():
    """After a step every written row holds the top-8 of the last (request,
    slot) writer of that token; untouched rows keep their value."""
    w = W.WORKLOADS[2].scaled(V=200, B=4)
    h = W.Harness(w)
    P = oracle.make_params(w.V, mode=w.mode)
    rng = np.random.default_rng(5)
    C0 = rng.integers(-1, w.V, (w.V, 8)).astype(np.int32)
    C = C0.copy()
    root, prev, ctx = h.init_state()
    tok, par, aux = h.draft(0, root, prev)
    saved = {}

    def make_logits(trees):
        tt = np.stack([t.tok for t in trees])
        pp = np.stack([t.par for t in trees]).astype(np.int8)
        lg = h.tree_logits(tt, pp, ctx, prev)
        saved["lg"], saved["tok"] = lg, tt
        return lg
    oracle.step(P, C, root, tok, aux, par, make_logits, w.dtype)
    last = {}
    for b in range(w.B):
        for i in range(w.S):
            t = int(saved["tok"][b, i])
            if t >= 0:
                last[t] = (b, i)
    for t in range(w.V):
        if t in last:
            b, i = last[t]
            assert np.array_equal(C[t], lexsort_topk(bf16_to_f32(saved["lg"][b, i])))
        else:
            assert np.array_equal(C[t], C0[t])


def test_warmup_equals_last_occurrence():
    """Sequential warm-up overwrite equals loading each token's last row."""
    rng = np.random.default_rng(3)
    V, N = 40, 300
    toks = rng.integers(0, 12, N).astype(np.int32)
    rows = rng.integers(-4, 5, (N, V)).astype(np.float32)
    C = oracle.new_matrix(V)
    oracle.warmup(C, toks, rows, oracle.F32)
    for t in range(V):
        occ = np.where(toks == t)[0]
        if len(occ):
            assert np.array_equal(C[t], lexsort_topk(rows[occ[-1]]))
        else:
            assert (C[t] == -1).all()


def test_invalid_inputs_are_errors():
    V = 100
    P = oracle.make_params(V)
    tok, par, prob = _layered_tree([0.5] * 6, V=V)
    tok %= V
    with pytest.raises(oracle.OracleError):
        oracle.assemble(P, V + 3, tok, prob, oracle.new_matrix(V), par)     # root out of range
    bad = prob.copy()
    bad[7] = np.nan
    with pytest.raises(oracle.OracleError):
        oracle.assemble(P, 1, tok, bad, oracle.new_matrix(V), par)
    C = oracle.new_matrix(V)
    C[1, 0] = V + 5                                                           # corrupt matrix entry
    tok2, par2, prob2 = _layered_tree([0.25] + [1] * 5, V=V)
    with pytest.raises(oracle.OracleError):
        oracle.assemble(P, 1, tok2 % V, prob2, C, par2)
