"""Graft CPU oracle (test infrastructure only).

A ctypes front-end for ``graft_oracle.c``, the plain single-threaded CPU
restatement of one Graft decode step (arXiv 2605.20104; the Hugging Face
paper page's abstract and the popular-science article's sections 二 to 七),
plus two fp64 numpy restatements written here: the coverage gain (section
三) and lossless stochastic verification (section 二, third gear).  Only the
test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline may
import this package; the CUDA library never does.

Parity unpinned beyond their stated rules (the pages give no procedure): the
coverage gain's boundary and novelty rule, and the stochastic walk's order of
candidates; the tests pin each by closed forms, Monte Carlo and limits.

All arrays are numpy.  Nothing here touches a GPU.  ``GRAFT_ORACLE_LIB``, when
set, names a prebuilt copy of the oracle library to load instead of building
this one (the mutation tests point it at copies with a planted mistake).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "graft_oracle.c")
_LIB = os.path.join(_HERE, "libgraft_oracle.so")

K = 8
MODE_CHECKPOINT, MODE_STATIC, MODE_TAIL = 0, 1, 2
F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no contraction of float expressions)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Params(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int32), ("K", ctypes.c_int32), ("budget", ctypes.c_int32),
                ("S", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("ckpt_depth", ctypes.c_int32 * 3), ("ckpt_thr", ctypes.c_float * 3),
                ("ckpt_draft", ctypes.c_int32 * 3), ("tpl_depth", ctypes.c_int32),
                ("tpl_width", ctypes.c_int32), ("static_thr", ctypes.c_float),
                ("tail_thr", ctypes.c_float), ("ablation", ctypes.c_int32), ("fixed_draft", ctypes.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(os.environ.get("GRAFT_ORACLE_LIB") or build())
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc < 0:
        raise OracleError(f"{what} failed with status {rc}")
    return rc


def make_params(V, budget=60, mode=MODE_CHECKPOINT, ckpt_depth=(0, 1, 5), ckpt_thr=(0.30, 0.20, 0.10),
                ckpt_draft=(8, 24, 40), tpl_depth=8, tpl_width=8, static_thr=0.15, tail_thr=0.4, ablation=0,
                fixed_draft=40):
    p = Params()
    p.V, p.K, p.budget, p.S, p.mode = V, K, budget, budget + 1, mode
    for i in range(3):
        p.ckpt_depth[i] = ckpt_depth[i]
        p.ckpt_thr[i] = ckpt_thr[i]
        p.ckpt_draft[i] = ckpt_draft[i]
    p.tpl_depth, p.tpl_width = tpl_depth, tpl_width
    p.static_thr, p.tail_thr = static_thr, tail_thr
    p.ablation, p.fixed_draft = ablation, fixed_draft
    return p


def check_layer(P, par, prob, layer, event):
    """Incremental checkpoint evaluation after layers 0..layer; returns the
    (possibly updated) event of one request."""
    par = np.ascontiguousarray(par, np.int16)
    prob = np.ascontiguousarray(prob, np.float32)
    ev = ctypes.c_int32(int(event))
    _check(lib().or_check_layer(ctypes.byref(P), len(par), _p(par), _p(prob), layer, ctypes.byref(ev)),
           "or_check_layer")
    return ev.value


def retrieve(P, root, event, C):
    """Retrieval entries of one request in template order ([budget], -1 = none)."""
    out = np.empty(P.budget, np.int32)
    _check(lib().or_retrieve(ctypes.byref(P), int(root), int(event), _p(np.ascontiguousarray(C, np.int32)), _p(out)),
           "or_retrieve")
    return out


def coverage(tree, info, rows, dtype):
    """Coverage gain of the retrieval graft (article section 三), fp64: the
    target probability mass that the new candidates at the prune boundary add.
    Retrieved slots follow the kept draft slots (checkpoint and tail modes);
    a retrieved slot whose parent is a kept slot is a boundary candidate, new
    unless a kept draft child of that parent has the same token; the gain is
    the sum of softmax(parent's row)[token] over the new candidates.
    rows: [S, V] logits of the tree (float32, or bf16 bit patterns)."""
    n_draft, n_retr = int(info[1]), int(info[2])
    r0, r1 = 1 + n_draft, 1 + n_draft + n_retr
    vals = np.asarray(rows)
    if dtype == BF16:
        vals = (vals.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
    vals = vals.astype(np.float64)
    gain = 0.0
    for p in range(r0):
        kids = [j for j in range(r0, r1) if tree.par[j] == p]
        if not kids:
            continue
        x = vals[p]
        m = x.max()
        z = np.exp(x - m).sum()
        drafted = {int(tree.tok[q]) for q in range(1, r0) if tree.par[q] == p}
        for j in kids:
            t = int(tree.tok[j])
            if t not in drafted:
                gain += np.exp(x[t] - m) / z
    return gain


def template(R, depth=8, width=8):
    """First R retrieval-template entries: (parent entry, rank, depth) arrays."""
    par = np.zeros(max(R, 1), np.int32)
    rank = np.zeros(max(R, 1), np.int32)
    dep = np.zeros(max(R, 1), np.int32)
    m = _check(lib().or_template(depth, width, R, _p(par), _p(rank), _p(dep)), "or_template")
    return par[:m].copy(), rank[:m].copy(), dep[:m].copy()


def topk8_row(row: np.ndarray, dtype: int) -> np.ndarray:
    """Top-8 ids of one row (float32, or bf16 given as uint16 bit patterns)."""
    row = np.ascontiguousarray(row)
    ids = np.zeros(K, np.int32)
    _check(lib().or_topk8_row(_p(row), dtype, row.shape[-1], _p(ids)), "or_topk8_row")
    return ids


def path_conf(parent: np.ndarray, prob: np.ndarray):
    parent = np.ascontiguousarray(parent, np.int16)
    prob = np.ascontiguousarray(prob, np.float32)
    conf = np.zeros(len(prob), np.float32)
    depth = np.zeros(len(prob), np.int32)
    _check(lib().or_path_conf(len(prob), _p(parent), _p(prob), _p(conf), _p(depth)), "or_path_conf")
    return conf, depth


class Tree:
    """Flattened hybrid tree of one request."""

    def __init__(self, S):
        self.tok = np.full(S, -1, np.int32)
        self.par = np.full(S, -1, np.int32)
        self.pos = np.full(S, -1, np.int32)
        self.mask = np.zeros(S, np.uint64)
        self.info = np.zeros(4, np.int32)


def assemble(params: Params, root_tok: int, draft_tok, draft_aux, C: np.ndarray, draft_parent=None) -> Tree:
    """One request's hybrid tree.  draft_aux is the per-node draft probability
    (checkpoint / static mode) or the per-position block confidence (tail)."""
    t = Tree(params.S)
    dtok = np.ascontiguousarray(draft_tok, np.int32)
    aux = np.ascontiguousarray(draft_aux, np.float32)
    L = lib()
    args = (_p(t.tok), _p(t.par), _p(t.pos), _p(t.mask), _p(t.info))
    if params.mode == MODE_TAIL:
        rc = L.or_assemble_tail(ctypes.byref(params), int(root_tok), len(dtok), _p(dtok), _p(aux), _p(C), *args)
    else:
        dpar = np.ascontiguousarray(draft_parent, np.int16)
        fn = L.or_assemble_checkpoint if params.mode == MODE_CHECKPOINT else L.or_assemble_static
        rc = fn(ctypes.byref(params), int(root_tok), len(dtok), _p(dtok), _p(dpar), _p(aux), _p(C), *args)
    _check(rc, "assemble")
    return t


def verify(tree: Tree, logits: np.ndarray, dtype: int):
    """Greedy verification of one request.  logits: [S, V] (float32 or uint16
    bf16 bits).  Returns (accept_len, emitted tokens [S] padded with -1,
    topk [S, 8])."""
    S = len(tree.tok)
    logits = np.ascontiguousarray(logits)
    topk = np.zeros((S, K), np.int32)
    out = np.zeros(S, np.int32)
    acc = np.zeros(1, np.int32)
    _check(lib().or_verify(S, _p(tree.tok), _p(tree.par), _p(logits), dtype, logits.shape[-1],
                           ctypes.c_int64(logits.shape[-1]), _p(topk), _p(acc), _p(out)), "or_verify")
    return int(acc[0]), out, topk


def verify_sample(tree: Tree, logits: np.ndarray, dtype: int, inv_temp: float, u: np.ndarray, u_res: float):
    """Lossless stochastic verification of one request (article section 二
    third gear: the output distribution equals sampling from the target), in
    fp64.  The candidates are deterministic (draft top-k and retrieved
    tokens), so they are tested one by one: at node n with target
    distribution p = softmax(row_n * inv_temp), child c (slot order) is
    accepted when u[c] * rem < p(tok_c), rem being the mass not yet rejected
    at n; a rejected token's mass leaves rem (a repeated token has none
    left).  On acceptance the walk descends into c.  When every child is
    rejected (or n is a leaf) the last token is drawn from p restricted to
    the unrejected tokens: the first v whose cumulative mass exceeds
    u_res * (their total).  Each token so emitted is distributed exactly as p.
    Returns (accept_len, emitted [S] padded with -1, smallest decision margin
    relative to the mass compared against)."""
    S = len(tree.tok)
    vals = np.asarray(logits)
    if dtype == BF16:
        vals = (vals.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
    vals = vals.astype(np.float64)
    out = np.full(S, -1, np.int32)
    if tree.tok[0] < 0:
        return 0, out, np.inf
    node, length, margin = 0, 0, np.inf
    while True:
        x = vals[node]
        w = np.exp((x - x.max()) * inv_temp)
        p = w / w.sum()
        rem, rejected, acc = 1.0, set(), -1
        for j in range(node + 1, S):
            tk = int(tree.tok[j])
            if tree.par[j] != node or tk < 0 or tk in rejected:
                continue
            margin = min(margin, abs(u[j] * rem - p[tk]) / max(p[tk], 1e-300))
            if u[j] * rem < p[tk]:
                acc = j
                break
            rem -= p[tk]
            rejected.add(tk)
        if acc >= 0:
            out[length] = tree.tok[acc]
            length += 1
            node = acc
            continue
        w2 = w.copy()
        w2[list(rejected)] = 0.0
        cum = np.cumsum(w2)
        if cum[-1] <= 0.0:                       # every token with mass was rejected: undefined
            out[length] = len(cum) - 1
            return length, out, 0.0
        target = u_res * cum[-1]
        v = int(np.searchsorted(cum, target, side="right"))
        v = min(v, len(cum) - 1)
        lo = cum[v - 1] if v > 0 else 0.0
        margin = min(margin, min(target - lo, cum[v] - target) / cum[-1])
        out[length] = v
        return length, out, margin


def update(C: np.ndarray, tree: Tree, topk: np.ndarray):
    _check(lib().or_update(_p(C), C.shape[0], len(tree.tok), _p(tree.tok),
                           _p(np.ascontiguousarray(topk, np.int32))), "or_update")


def warmup(C: np.ndarray, tokens: np.ndarray, logits: np.ndarray, dtype: int):
    tokens = np.ascontiguousarray(tokens, np.int32)
    logits = np.ascontiguousarray(logits)
    _check(lib().or_warmup(_p(C), C.shape[0], ctypes.c_int64(len(tokens)), _p(tokens), _p(logits), dtype,
                           ctypes.c_int64(logits.shape[-1])), "or_warmup")


def new_matrix(V: int) -> np.ndarray:
    return np.full((V, K), -1, np.int32)


def step(params: Params, C: np.ndarray, roots, draft_tok, draft_aux, draft_parent, make_logits, dtype):
    """One batched decode step in the order the method runs it: every request
    is assembled from the matrix as it stood at the start of the step, the
    target scores all trees (``make_logits(trees) -> [B, S, V]``), then each
    request in turn is verified and its rows update the matrix."""
    B = len(roots)
    trees = [assemble(params, roots[b], draft_tok[b], draft_aux[b], C,
                      None if draft_parent is None else draft_parent[b]) for b in range(B)]
    logits = make_logits(trees)
    results = []
    for b in range(B):
        acc, out, topk = verify(trees[b], logits[b], dtype)
        update(C, trees[b], topk)
        results.append((acc, out))
    return trees, results
