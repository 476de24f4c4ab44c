"""Seeded synthetic workloads for the Graft hot path.

This package only generates inputs: draft trees / draft blocks, token
histories, and the logits rows of a synthetic target whose row at a prefix is
a pure function of that prefix.  It holds none of the method's arithmetic.
Both the CPU oracle and the CUDA library consume what it produces; the host
generator (``synth_host.c``) and its device twin (``synth_dev.cu``) agree bit
for bit (checked by the GPU tests).

The five workloads mirror the paper's settings with synthetic data:
  0  V=32000  batch 1, checkpoint mode, fp32 logits, bigram target (+6, always)
  1  V=128256 batch 1, checkpoint mode, bf16, trigram target (+5, 70 %),
     warm-up from 5 roll-outs x 256 positions
  2  V=151936 batch 16, static-tree mode, bf16, per-request bigram (+5, 60 %)
  3  V=151936 batch 1, checkpoint mode, bf16, warm start from a 32768-token
     history (Zipf(1.1) over 2000 ids, 30 % copied spans), then decode with a
     history-successor target (+6, always)
  4  V=151936 batch 64, tail mode (16-token blocks), bf16, bigram (+5, 50 %)
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SRC = os.path.join(_HERE, "synth_host.c")
_HOST_LIB = os.path.join(_HERE, "libsynth_host.so")
_DEV_SRC = os.path.join(_HERE, "synth_dev.cu")
_DEV_LIB = os.path.join(_HERE, "libsynth_dev.so")

F32, BF16 = 0, 1
MODE_CHECKPOINT, MODE_STATIC, MODE_TAIL = 0, 1, 2
TREE_BRANCHING = (4, 3, 2, 2, 1, 1)
TREE_NODES = 184


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    V: int
    B: int
    mode: int
    dtype: int
    steps: int
    seed: int
    kind: int                 # target: 0 bigram, 1 trigram, 2 per-request bigram, 3 table
    bias: float
    hit_rate: float           # 1.0 = every context hits
    budget: int = 60
    warm: str = "none"        # "none" | "rollouts" | "history"
    warm_rollouts: int = 5
    warm_positions: int = 256
    hist_len: int = 32768
    hist_active: int = 2000
    draft_sigma: float = 2.0
    block_len: int = 16
    block_mu: float = 1.0
    block_sd: float = 1.5
    block_decay: float = 0.25

    @property
    def S(self) -> int:
        return self.budget + 1

    @property
    def draft_nodes(self) -> int:
        return self.block_len if self.mode == MODE_TAIL else TREE_NODES

    @property
    def hit_all(self) -> int:
        return 1 if self.hit_rate >= 1.0 else 0

    @property
    def hit_num(self) -> int:
        return min(int(self.hit_rate * 2**32), 2**32 - 1)

    @property
    def esize(self) -> int:
        return 4 if self.dtype == F32 else 2

    def logits_bytes_per_step(self) -> int:
        return self.B * self.S * self.V * self.esize

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    0: Workload("v32000-b1-checkpoint-f32", 32000, 1, MODE_CHECKPOINT, F32, 100, 0, 0, 6.0, 1.0),
    1: Workload("v128256-b1-checkpoint-bf16-warm1280", 128256, 1, MODE_CHECKPOINT, BF16, 1000, 1, 1, 5.0, 0.7,
                warm="rollouts"),
    2: Workload("v151936-b16-static-bf16", 151936, 16, MODE_STATIC, BF16, 500, 2, 2, 5.0, 0.6),
    3: Workload("v151936-b1-warm32768-checkpoint-bf16", 151936, 1, MODE_CHECKPOINT, BF16, 200, 3, 3, 6.0, 1.0,
                warm="history"),
    4: Workload("v151936-b64-tail16-bf16", 151936, 64, MODE_TAIL, BF16, 300, 4, 0, 5.0, 0.5, budget=16),
}


# --------------------------------------------------------------------------- host library
def _build(src, out, cmd):
    if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(cmd + ["-o", tmp, src])
        os.replace(tmp, out)
    return out


def build_host() -> str:
    return _build(_HOST_SRC, _HOST_LIB, ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                                         "-Wall", "-lm"])


def build_dev() -> str:
    return _build(_DEV_SRC, _DEV_LIB, ["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a",
                                       "-Xcompiler", "-fPIC", "-shared", "-fmad=false", "-lineinfo"])


_host = None
_dev = None


def host():
    global _host
    if _host is None:
        _host = ctypes.CDLL(build_host())
        _host.syn_sm64.restype = ctypes.c_uint64
        _host.syn_sm64.argtypes = [ctypes.c_uint64]
        _host.syn_ctx_push.restype = ctypes.c_uint64
        _host.syn_ctx_push.argtypes = [ctypes.c_uint64, ctypes.c_int32]
        _host.syn_succ.restype = ctypes.c_int32
        _host.syn_succ.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p,
                                   ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
    return _host


def dev():
    """Device twin of the generator (needs a CUDA build; harness only)."""
    global _dev
    if _dev is None:
        _dev = ctypes.CDLL(build_dev())
    return _dev


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _ok(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with status {rc}")


u64 = ctypes.c_uint64
i64 = ctypes.c_int64


def host_threads() -> int:
    """Threads for the host row filler: the cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def fill_rows(rowkey, planted, bias, V, dtype, out=None, threads=1):
    """Host row filler: returns [n, V] float32 or uint16 (bf16 bits).  With
    threads > 1 the rows are split into contiguous blocks filled in parallel
    (the C filler releases the GIL; every row is a pure function of its own
    key, so the result is identical)."""
    rowkey = np.ascontiguousarray(rowkey, np.uint64)
    planted = np.ascontiguousarray(planted, np.int32)
    bias = np.ascontiguousarray(bias, np.float32)
    n = len(rowkey)
    if out is None:
        out = np.empty((n, V), np.float32 if dtype == F32 else np.uint16)
    stride = out.shape[-1]
    lib = host()

    def fill(r0, r1):
        if r1 > r0:
            lib.syn_fill_rows(_p(rowkey[r0:]), _p(planted[r0:]), _p(bias[r0:]), i64(r1 - r0), V, dtype,
                              _p(out.reshape(n, stride)[r0:]), i64(stride))

    threads = max(1, min(int(threads), n))
    if threads == 1:
        fill(0, n)
        return out
    import concurrent.futures as cf
    cuts = [n * k // threads for k in range(threads + 1)]
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda k: fill(cuts[k], cuts[k + 1]), range(threads)))
    return out


class Harness:
    """Host-side state of one workload: request state, draft inputs, target
    row parameters.  Purely input generation."""

    def __init__(self, w: Workload):
        self.w = w
        self.table = None
        self.hist = None
        self.active = None
        if w.kind == 3:
            self.hist, self.active = self.history()
            self.table = np.empty(w.V, np.int32)
            host().syn_history_successors(w.V, len(self.hist), _p(self.hist), _p(self.table))

    # --- target description passed to the C functions
    def _tgt(self):
        w = self.w
        return (w.V, w.kind, w.hit_all, ctypes.c_uint32(w.hit_num), ctypes.c_float(w.bias), u64(w.seed),
                _p(self.table))

    def init_state(self):
        B = self.w.B
        root = np.empty(B, np.int32)
        prev = np.empty(B, np.int32)
        ctx = np.empty(B, np.uint64)
        host().syn_init_state(u64(self.w.seed), self.w.V, B, _p(root), _p(prev), _p(ctx))
        return root, prev, ctx

    def advance(self, root, prev, ctx, emitted, accept_len):
        """emitted: [B, S] (path then bonus); accept_len: [B]."""
        emitted = np.ascontiguousarray(emitted, np.int32)
        count = np.ascontiguousarray(accept_len, np.int32) + 1
        host().syn_advance(self.w.B, emitted.shape[-1], _p(emitted), _p(count), _p(root), _p(prev), _p(ctx))

    def draft(self, step, root, prev):
        """Draft inputs for every request: (tok, parent or None, aux)."""
        w = self.w
        B = w.B
        if w.mode == MODE_TAIL:
            tok = np.empty((B, w.block_len), np.int32)
            conf = np.empty((B, w.block_len), np.float32)
            for b in range(B):
                host().syn_draft_block(w.V, w.kind, u64(w.seed), _p(self.table), i64(step), b, int(root[b]),
                                       int(prev[b]), w.block_len, ctypes.c_float(w.block_mu),
                                       ctypes.c_float(w.block_sd), ctypes.c_float(w.block_decay),
                                       _p(tok[b]), _p(conf[b]))
            return tok, None, conf
        tok = np.empty((B, TREE_NODES), np.int32)
        par = np.empty((B, TREE_NODES), np.int16)
        prob = np.empty((B, TREE_NODES), np.float32)
        br = np.array(TREE_BRANCHING, np.int32)
        for b in range(B):
            n = host().syn_draft_tree(w.V, w.kind, u64(w.seed), _p(self.table), ctypes.c_float(w.draft_sigma),
                                      i64(step), b, int(root[b]), int(prev[b]), _p(br), len(br), TREE_NODES,
                                      _p(tok[b]), _p(par[b]), _p(prob[b]))
            if n != TREE_NODES:
                raise RuntimeError(f"syn_draft_tree returned {n} nodes, expected {TREE_NODES}")
        return tok, par, prob

    def tree_rowparams(self, tok, par, root_ctx, root_prev):
        """Row parameters of flattened trees tok/par: [B, S]."""
        tok = np.ascontiguousarray(tok, np.int32)
        par = np.ascontiguousarray(par, np.int8)
        B, S = tok.shape
        rowkey = np.empty((B, S), np.uint64)
        planted = np.empty((B, S), np.int32)
        bias = np.empty((B, S), np.float32)
        host().syn_tree_rowparams(*self._tgt(), B, S, _p(tok), _p(par), _p(np.ascontiguousarray(root_ctx, np.uint64)),
                                  _p(np.ascontiguousarray(root_prev, np.int32)), _p(rowkey), _p(planted), _p(bias))
        return rowkey, planted, bias

    def tree_logits(self, tok, par, root_ctx, root_prev, threads=1):
        rk, pl, bi = self.tree_rowparams(tok, par, root_ctx, root_prev)
        B, S = rk.shape
        return fill_rows(rk.reshape(-1), pl.reshape(-1), bi.reshape(-1), self.w.V, self.w.dtype,
                         threads=threads).reshape(B, S, -1)

    def prefix_rowparams(self, b, ctx, prev, t):
        rk = np.zeros(1, np.uint64)
        pl = np.zeros(1, np.int32)
        bi = np.zeros(1, np.float32)
        host().syn_prefix_rowparams(*self._tgt(), b, u64(int(ctx)), int(prev), int(t), _p(rk), _p(pl), _p(bi))
        return rk, pl, bi

    # --- warm-up inputs
    def history(self):
        w = self.w
        hist = np.empty(w.hist_len, np.int32)
        active = np.empty(w.hist_active, np.int32)
        rc = host().syn_history(u64(w.seed), w.V, w.hist_len, w.hist_active, ctypes.c_double(1.1),
                                ctypes.c_double(0.3), 16, 64, _p(hist), _p(active))
        _ok(rc, "syn_history")
        return hist, active

    def warm_rowparams(self):
        """(tokens, rowkey, planted, bias) of the warm-up rows, or None."""
        w = self.w
        if w.warm == "history":
            n = len(self.hist)
            rk = np.empty(n, np.uint64)
            pl = np.empty(n, np.int32)
            bi = np.empty(n, np.float32)
            host().syn_history_rowparams(u64(w.seed), n, _p(self.hist), ctypes.c_float(5.0), _p(rk), _p(pl), _p(bi))
            return self.hist.copy(), rk, pl, bi
        if w.warm == "rollouts":
            n = w.warm_rollouts * w.warm_positions
            toks = np.empty(n, np.int32)
            rk = np.empty(n, np.uint64)
            pl = np.empty(n, np.int32)
            bi = np.empty(n, np.float32)
            host().syn_rollouts(*self._tgt(), w.warm_rollouts, w.warm_positions, _p(toks), _p(rk), _p(pl), _p(bi))
            return toks, rk, pl, bi
        return None


# --------------------------------------------------------------------------- device twin
def _dp(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


class DeviceSynth:
    """Device twin of the row filler and of the tree row parameters (torch
    tensors in, torch tensors out; runs on the given CUDA stream)."""

    def __init__(self, harness: Harness, device):
        import torch
        self.h = harness
        self.w = harness.w
        self.torch = torch
        self.device = device
        self.lib = dev()
        self.table = None if harness.table is None else torch.from_numpy(harness.table).to(device)

    def tree_rowparams(self, tok, par, root_ctx, root_prev, stream):
        torch = self.torch
        B, S = tok.shape
        rk = torch.empty((B, S), dtype=torch.int64, device=self.device)
        pl = torch.empty((B, S), dtype=torch.int32, device=self.device)
        bi = torch.empty((B, S), dtype=torch.float32, device=self.device)
        w = self.w
        rc = self.lib.synd_tree_rowparams(w.V, w.kind, w.hit_all, ctypes.c_uint32(w.hit_num), ctypes.c_float(w.bias),
                                          u64(w.seed), _dp(self.table), B, S, _dp(tok), _dp(par), _dp(root_ctx),
                                          _dp(root_prev), _dp(rk), _dp(pl), _dp(bi), ctypes.c_void_p(stream))
        _ok(rc, "synd_tree_rowparams")
        return rk, pl, bi

    def fill_rows(self, rk, pl, bi, out, stream):
        n = rk.numel()
        rc = self.lib.synd_fill_rows(_dp(rk), _dp(pl), _dp(bi), i64(n), self.w.V, self.w.dtype, _dp(out),
                                     i64(out.stride(-2)), ctypes.c_void_p(stream))
        _ok(rc, "synd_fill_rows")

    def advance(self, out_tokens, accept_len, root, prev, ctx, stream):
        B, S = out_tokens.shape
        rc = self.lib.synd_advance(B, S, _dp(out_tokens), _dp(accept_len), _dp(root), _dp(prev), _dp(ctx),
                                   ctypes.c_void_p(stream))
        _ok(rc, "synd_advance")
