"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle (a dropped term, a
flipped comparison, a wrong index, a reversed order): in the C step (the copy
is compiled with gcc) or in the fp64 numpy restatements of the coverage gain
and of stochastic verification (the copy is loaded in place of the package).
The pin suite then runs against the copy; the case passes when at least one
pin fails.  A mistake that no pin notices would mean the oracle is checked only
against itself at that point.  Nothing here touches a GPU or the CUDA library.

Sources of the rules the mistakes break: popular-science article on arXiv
2605.20104, sections 二 (three gears), 四 (static trees), 五 (ablations), 六
(warm-up) and 七 (Graft-TAIL); section 三 (coverage) and section 二's third
gear (verification lossless at a temperature) for the numpy ones.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "graft_oracle.c")
PY_SRC = os.path.join(ROOT, "oracle", "__init__.py")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in the oracle, planted replacement); the text must occur once.
MUTANTS = [
    # top-8 of a row (gear 3)
    ("topk tie goes to the higher id", "return va > vb || (va == vb && ia < ib);",
     "return va > vb || (va == vb && ia > ib);"),
    ("topk keeps the smallest values", "return va > vb || (va == vb && ia < ib);",
     "return va < vb || (va == vb && ia < ib);"),
    ("bf16 decoded with a wrong shift", "uint32_t u = (uint32_t)((const uint16_t*)row)[v] << 16;",
     "uint32_t u = (uint32_t)((const uint16_t*)row)[v] << 15;"),
    ("topk drops its last entry", "for (int32_t k = 0; k < OR_K; ++k) ids[k] = k < cnt ? bi[k] : -1;",
     "for (int32_t k = 0; k < OR_K; ++k) ids[k] = k < cnt - 1 ? bi[k] : -1;"),
    # retrieval template (gear 2)
    ("template fan-out halves one rank late", "int f = width >> r[depth - 1];",
     "int f = width >> (r[depth - 1] + 1);"),
    ("template anchor fan-out off by one", "if (depth == 0) return width;                 /* the anchor */",
     "if (depth == 0) return width - 1;"),
    ("template ordered by depth first", "if (a->sum != b->sum) return a->sum < b->sum ? -1 : 1;\n  if (a->len != b->len) return a->len < b->len ? -1 : 1;",
     "if (a->len != b->len) return a->len < b->len ? -1 : 1;\n  if (a->sum != b->sum) return a->sum < b->sum ? -1 : 1;"),
    ("template rank path compared in reverse", "for (int i = 0; i < a->len; ++i) if (a->r[i] != b->r[i]) return a->r[i] < b->r[i] ? -1 : 1;",
     "for (int i = 0; i < a->len; ++i) if (a->r[i] != b->r[i]) return a->r[i] > b->r[i] ? -1 : 1;"),
    ("template depth limit off by one", "if (cur->len >= dmax) return;", "if (cur->len > dmax) return;"),
    # path confidence and checkpoints (gear 1)
    ("path confidence drops the parent's factor", "volatile float prod = pc * prob[i];",
     "volatile float prod = prob[i];"),
    ("depth does not grow along a path", "depth[i] = (p < 0) ? 0 : depth[p] + 1;",
     "depth[i] = (p < 0) ? 0 : depth[p];"),
    ("checkpoint fires above its threshold",
     "if (any && best < P->ckpt_thr[k]) { fired = d; D = P->ckpt_draft[k]; R = P->budget - D; cut = d; break; }",
     "if (any && best > P->ckpt_thr[k]) { fired = d; D = P->ckpt_draft[k]; R = P->budget - D; cut = d; break; }"),
    ("checkpoint looks at the worst path",
     "for (int32_t i = 0; i < n; ++i) if (depth[i] == d) { if (!any || conf[i] > best) best = conf[i]; any = 1; }\n"
     "      if (any && best < P->ckpt_thr[k]) { fired",
     "for (int32_t i = 0; i < n; ++i) if (depth[i] == d) { if (!any || conf[i] < best) best = conf[i]; any = 1; }\n"
     "      if (any && best < P->ckpt_thr[k]) { fired"),
    ("retrieval gets one slot too few", "fired = d; D = P->ckpt_draft[k]; R = P->budget - D; cut = d;",
     "fired = d; D = P->ckpt_draft[k]; R = P->budget - D - 1; cut = d;"),
    ("pruning keeps layers past the firing depth", "if (depth[i] <= cut) { items[m].conf",
     "if (depth[i] <= cut + 1) { items[m].conf"),
    ("kept nodes are the least confident", "if (a->conf != b->conf) return a->conf > b->conf ? -1 : 1;",
     "if (a->conf != b->conf) return a->conf < b->conf ? -1 : 1;"),
    ("confidence ties go to the later node", "return a->idx < b->idx ? -1 : (a->idx > b->idx);",
     "return a->idx > b->idx ? -1 : (a->idx < b->idx);"),
    # retrieval gather (gear 2)
    ("retrieval always takes rank 0", "int32_t t = C[(int64_t)ptok * OR_K + tr[j]];\n    if (t < -1 || t >= P->V) return OR_EDATA;\n    if (t < 0) continue;",
     "int32_t t = C[(int64_t)ptok * OR_K + 0];\n    if (t < -1 || t >= P->V) return OR_EDATA;\n    if (t < 0) continue;"),
    ("retrieval children hang off the root", "rslot[j] = s; tok[s] = t; par[s] = tp[j] < 0 ? 0 : rslot[tp[j]]; ++s; ++nr;",
     "rslot[j] = s; tok[s] = t; par[s] = 0; ++s; ++nr;"),
    ("an empty entry keeps its subtree", "int32_t ptok = tp[j] < 0 ? root_tok : rtok[tp[j]];\n    if (ptok < 0) continue;",
     "int32_t ptok = tp[j] < 0 ? root_tok : (rtok[tp[j]] < 0 ? root_tok : rtok[tp[j]]);\n    if (ptok < 0) continue;"),
    # ablations (section 五)
    ("the no-retrieval ablation still retrieves", "if (P->ablation == 1) R = 0;", "if (P->ablation == 3) R = 0;"),
    ("the fixed split swaps draft and retrieval", "D = P->fixed_draft; R = P->budget - D;",
     "R = P->fixed_draft; D = P->budget - R;"),
    # incremental checkpoints and retrieve
    ("a checkpoint is evaluated before its layer exists", "if (d > layer) continue;", "if (d > layer + 1) continue;"),
    ("retrieve ignores the fired split", "if (P->ckpt_depth[k] == event) { R = P->budget - P->ckpt_draft[k]; break; }",
     "if (P->ckpt_depth[k] == event) { R = P->budget - P->ckpt_draft[0]; break; }"),
    # flatten (gear 3)
    ("tree position is not the depth", "pos[i] = pos[par[i]] + 1;", "pos[i] = pos[par[i]] + (i & 1);"),
    ("mask row misses its ancestors", "mask[i] = mask[par[i]] | (1ull << i);", "mask[i] = mask[0] | (1ull << i);"),
    # static trees (section 四)
    ("static mode replaces confident nodes", "replaced[s] = conf[i] < P->static_thr;",
     "replaced[s] = conf[i] >= P->static_thr;"),
    ("static replacement rank counts every sibling", "for (int32_t q = 1; q < i; ++q) if (par[q] == p && replaced[q]) ++srank;",
     "for (int32_t q = 1; q < i; ++q) if (par[q] == p) ++srank;"),
    ("static replacement reads the draft token's row", "int32_t t = srank < OR_K ? C[(int64_t)tok[p] * OR_K + srank] : -1;",
     "int32_t t = srank < OR_K ? C[(int64_t)tok[i] * OR_K + srank] : -1;"),
    ("an empty static entry empties the slot", "if (t >= 0) { tok[i] = t; ++nr; }\n    else ++nd;",
     "if (t >= 0) { tok[i] = t; ++nr; }\n    else { tok[i] = -1; ++nd; }"),
    # Graft-TAIL (section 七)
    ("tail cut at the first confident position", "for (int32_t i = 0; i < n; ++i) if (bconf[i] < P->tail_thr) { t = i; break; }",
     "for (int32_t i = 0; i < n; ++i) if (bconf[i] >= P->tail_thr) { t = i; break; }"),
    ("tail retrieval anchored at the root", "int32_t anchor = t;", "int32_t anchor = 0;"),
    ("tail budget ignores the kept prefix", "int32_t R = P->budget - t;", "int32_t R = P->budget - n;"),
    # greedy verification (gear 3)
    ("a node is checked against its own row", "for (int32_t j = i; j != 0; j = par[j]) { if (tok[j] != y[par[j]]) ok = 0; ++d; }",
     "for (int32_t j = i; j != 0; j = par[j]) { if (tok[j] != y[j]) ok = 0; ++d; }"),
    ("only the leaf's own edge is checked", "for (int32_t j = i; j != 0; j = par[j]) { if (tok[j] != y[par[j]]) ok = 0; ++d; }",
     "for (int32_t j = i; j != 0; j = par[j]) { if (j == i && tok[j] != y[par[j]]) ok = 0; ++d; }"),
    ("depth ties go to the later slot", "if (ok && d > win_depth) { win = i; win_depth = d; }",
     "if (ok && d >= win_depth) { win = i; win_depth = d; }"),
    ("the bonus token is the root's choice", "out_tokens[win_depth] = y[win];", "out_tokens[win_depth] = y[0];"),
    # online update and warm-up (gear 3, section 六)
    ("the update skips the root", "for (int32_t i = 0; i < S; ++i) {\n    if (tok[i] < 0) continue;\n    if (tok[i] >= V) return OR_EINVAL;",
     "for (int32_t i = 1; i < S; ++i) {\n    if (tok[i] < 0) continue;\n    if (tok[i] >= V) return OR_EINVAL;"),
    ("the update's first writer wins", "for (int32_t i = 0; i < S; ++i) {\n    if (tok[i] < 0) continue;\n    if (tok[i] >= V) return OR_EINVAL;",
     "for (int32_t i = S - 1; i >= 0; --i) {\n    if (tok[i] < 0) continue;\n    if (tok[i] >= V) return OR_EINVAL;"),
    ("warm-up's first occurrence wins", "for (int64_t n = 0; n < N; ++n) {", "for (int64_t n = N - 1; n >= 0; --n) {"),
    ("warm-up writes a shifted row", "for (int k = 0; k < OR_K; ++k) C[(int64_t)toks[n] * OR_K + k] = ids[k];",
     "for (int k = 0; k < OR_K; ++k) C[(int64_t)toks[n] * OR_K + k] = ids[(k + 1) % OR_K];"),
]


# The same for the numpy restatements in the oracle package.
PY_MUTANTS = [
    # coverage gain (section 三)
    ("coverage counts tokens the draft already has", "            if t not in drafted:\n",
     "            if True:\n"),
    ("coverage counts candidates below the boundary", "    for p in range(r0):\n        kids =",
     "    for p in range(r1):\n        kids ="),
    ("coverage is not normalised", "                gain += np.exp(x[t] - m) / z", "                gain += np.exp(x[t] - m)"),
    ("coverage compares against every sibling", "drafted = {int(tree.tok[q]) for q in range(1, r0) if tree.par[q] == p}",
     "drafted = {int(tree.tok[q]) for q in range(1, r0)}"),
    ("coverage decodes bf16 with a wrong shift",
     "        vals = (vals.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)\n    vals = vals.astype(np.float64)\n    gain",
     "        vals = (vals.astype(np.uint16).astype(np.uint32) << 15).view(np.float32)\n    vals = vals.astype(np.float64)\n    gain"),
    # stochastic verification (section 二, third gear)
    ("acceptance ignores the rejected mass", "            if u[j] * rem < p[tk]:", "            if u[j] < p[tk]:"),
    ("the rejected mass is not removed", "            rem -= p[tk]\n", "            rem -= 0.0\n"),
    ("the residual draw keeps rejected tokens", "        w2[list(rejected)] = 0.0\n", "        pass\n"),
    ("the temperature is ignored", "        w = np.exp((x - x.max()) * inv_temp)", "        w = np.exp(x - x.max())"),
    ("a repeated token is tested again", "if tree.par[j] != node or tk < 0 or tk in rejected:",
     "if tree.par[j] != node or tk < 0:"),
    ("acceptance stays at the root", "            node = acc\n            continue", "            continue"),
    ("the residual draw ignores its uniform", "        target = u_res * cum[-1]", "        target = 0.5 * cum[-1]"),
    ("sampling decodes bf16 with a wrong shift",
     "        vals = (vals.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)\n    vals = vals.astype(np.float64)\n    out",
     "        vals = (vals.astype(np.uint16).astype(np.uint32) << 15).view(np.float32)\n    vals = vals.astype(np.float64)\n    out"),
]

def _source():
    with open(SRC) as f:
        return f.read()


# Loaded with -p before any test module: the mutated package takes the name
# "oracle", so the pins import it instead of the real one.
_PLUGIN = """
import importlib.util, os, sys
_spec = importlib.util.spec_from_file_location("oracle", os.environ["GRAFT_MUTANT_ORACLE"])
_mod = importlib.util.module_from_spec(_spec)
sys.modules["oracle"] = _mod
_spec.loader.exec_module(_mod)
"""


def _tag(name):
    return "".join(c if c.isalnum() else "_" for c in name)


def _pins(env):
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"] +
                       (["-p", "graft_mutant_plugin"] if "GRAFT_MUTANT_ORACLE" in env else []),
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    return r.returncode, r.stdout[-600:]


def _run(name, old, new, workdir):
    src = _source()
    assert src.count(old) == 1, f"{name}: the planted text must occur once in the oracle"
    cfile = os.path.join(workdir, _tag(name) + ".c")
    lib = os.path.join(workdir, _tag(name) + ".so")
    with open(cfile, "w") as f:
        f.write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-w",
                           "-o", lib, cfile, "-lm"])
    rc, out = _pins(dict(os.environ, GRAFT_ORACLE_LIB=lib))
    return name, rc, out


def _run_py(name, old, new, workdir, lib):
    with open(PY_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"{name}: the planted text must occur once in the oracle package"
    d = os.path.join(workdir, _tag(name))
    os.makedirs(d)
    with open(os.path.join(d, "oracle.py"), "w") as f:
        f.write(src.replace(old, new))
    with open(os.path.join(d, "graft_mutant_plugin.py"), "w") as f:
        f.write(_PLUGIN)
    env = dict(os.environ, GRAFT_ORACLE_LIB=lib, GRAFT_MUTANT_ORACLE=os.path.join(d, "oracle.py"),
               PYTHONPATH=d + os.pathsep + os.environ.get("PYTHONPATH", ""))
    rc, out = _pins(env)
    return name, rc, out


def _check(results):
    survived = [name for name, rc, _ in results if rc == 0]
    crashed = [(name, rc, out) for name, rc, out in results if rc not in (0, 1)]
    assert not crashed, f"mutants that broke the pin run instead of failing a pin: {crashed}"
    assert not survived, "mistakes that no pin catches: " + ", ".join(survived)


def _workers():
    return min(8, os.cpu_count() or 1)


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with ThreadPoolExecutor(max_workers=_workers()) as ex:
        _check(list(ex.map(lambda m: _run(*m, str(tmp_path)), MUTANTS)))


def test_every_planted_numpy_mistake_fails_a_pin(tmp_path):
    import oracle
    lib = oracle.build()
    with ThreadPoolExecutor(max_workers=_workers()) as ex:
        _check(list(ex.map(lambda m: _run_py(*m, str(tmp_path), lib), PY_MUTANTS)))


def test_the_unmutated_oracle_passes_the_pins(tmp_path):
    """The harness itself: copies with no planted mistake pass."""
    name, rc, out = _run("unmutated", "#define OR_K 8", "#define OR_K 8", str(tmp_path))
    assert rc == 0, out
    import oracle
    name, rc, out = _run_py("unmutated py", "K = 8\n", "K = 8\n", str(tmp_path), oracle.build())
    assert rc == 0, out


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_text_is_present(name, old, new):
    assert _source().count(old) == 1
    assert old != new


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_planted_numpy_text_is_present(name, old, new):
    with open(PY_SRC) as f:
        assert f.read().count(old) == 1
    assert old != new
