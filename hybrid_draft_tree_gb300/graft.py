"""Python binding of libgraft (the C ABI declared in include/graft.h).

Argument marshalling only: every step of the Graft hot path runs in the CUDA
kernels of libgraft.so.  Device buffers are torch CUDA tensors (their
data_ptr is passed through); the stream is torch's current stream unless one
is given.  Before a pointer is passed, its tensor is checked against what the
C ABI expects of that buffer (CUDA memory, element type, contiguous layout,
enough elements for the batch), because the library cannot see a tensor's
size or memory kind: a violation raises GraftError(GRAFT_EINVAL) and nothing
is queued.  There is no CPU fallback: if the library is missing or no CUDA
device is present, these calls raise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

GRAFT_OK, GRAFT_EINVAL, GRAFT_ENOMEM, GRAFT_ECUDA, GRAFT_EDEVICE = 0, -1, -2, -3, -4
GRAFT_ERR_TOKEN, GRAFT_ERR_NAN, GRAFT_ERR_TREE, GRAFT_ERR_TIMEOUT = 1, 2, 4, 8
GRAFT_MODE_CHECKPOINT, GRAFT_MODE_STATIC, GRAFT_MODE_TAIL = 0, 1, 2
GRAFT_F32, GRAFT_BF16 = 0, 1
K = 8

# Entry points declared in include/graft.h (checked by the CPU tests).
EXPORTS = ("graft_default_config", "graft_init", "graft_destroy", "graft_warmup", "graft_assemble", "graft_assemble_src",
           "graft_verify_update", "graft_get_matrix", "graft_set_matrix", "graft_matrix_device_ptr",
           "graft_sync", "graft_last_error", "graft_last_launch_count", "graft_verify_update_noalloc",
           "graft_profile_enable", "graft_profile_read", "graft_check", "graft_retrieve", "graft_assemble_staged",
           "graft_confidence", "graft_calibrate_thresholds", "graft_set_thresholds", "graft_coverage",
           "graft_verify_update_sample", "graft_template", "graft_set_wait_limit")


def calibrate_thresholds(best: np.ndarray, quantile: float) -> np.ndarray:
    """Nearest-rank `quantile` of each checkpoint's best path confidences
    (best: [n, 3], -1 = empty layer), computed by the library (host code)."""
    best = np.ascontiguousarray(best, np.float32)
    out = np.zeros(3, np.float32)
    rc = load().graft_calibrate_thresholds(best.ctypes.data_as(vp), best.shape[0], ctypes.c_double(quantile),
                                           out.ctypes.data_as(vp))
    if rc != 0:
        raise GraftError(rc, "graft_calibrate_thresholds")
    return out


def template(depth: int = 8, width: int = 8, length: int = 60):
    """The first `length` retrieval-template entries the library uses for
    (depth, width), computed by the library (host code): arrays of the parent
    entry (-1 = the anchor), the rank (matrix column) and the depth."""
    par, rank, dep = (np.zeros(max(length, 1), np.int32) for _ in range(3))
    n = load().graft_template(depth, width, length, par.ctypes.data_as(vp), rank.ctypes.data_as(vp),
                              dep.ctypes.data_as(vp))
    if n < 0:
        raise GraftError(n, "graft_template")
    return par[:n].copy(), rank[:n].copy(), dep[:n].copy()


class GraftError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"graft error {code}: {msg}")
        self.code = code


class graft_config(ctypes.Structure):
    _fields_ = [("vocab", ctypes.c_int32), ("topk", ctypes.c_int32), ("budget", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("mode", ctypes.c_int32), ("logits_dtype", ctypes.c_int32),
                ("ckpt_depth", ctypes.c_int32 * 3), ("ckpt_thr", ctypes.c_float * 3),
                ("ckpt_draft", ctypes.c_int32 * 3), ("tpl_depth", ctypes.c_int32), ("tpl_width", ctypes.c_int32),
                ("static_thr", ctypes.c_float), ("tail_thr", ctypes.c_float), ("max_draft_nodes", ctypes.c_int32),
                ("scan_kernel", ctypes.c_int32), ("ablation", ctypes.c_int32), ("fixed_draft", ctypes.c_int32)]


_lib = None
vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libgraft.so (building it with nvcc when absent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise ImportError("libgraft.so is not built; run __graft_entry__.build()")
        _build.build()
    L = ctypes.CDLL(_build.LIB)
    L.graft_default_config.argtypes = [ctypes.POINTER(graft_config), i32, i32, i32, i32]
    L.graft_default_config.restype = None
    L.graft_init.argtypes = [ctypes.POINTER(graft_config), ctypes.POINTER(vp)]
    L.graft_destroy.argtypes = [vp]
    L.graft_warmup.argtypes = [vp, vp, vp, i64, i64, vp]
    L.graft_assemble.argtypes = [vp, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]
    L.graft_verify_update.argtypes = [vp, i32, vp, vp, vp, vp, vp, i64, vp, vp, vp]
    L.graft_check.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp]
    L.graft_retrieve.argtypes = [vp, i32, vp, vp, vp, vp]
    L.graft_assemble_staged.argtypes = [vp, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    L.graft_confidence.argtypes = [vp, i32, vp, vp, i32, vp, vp]
    L.graft_calibrate_thresholds.argtypes = [vp, i32, ctypes.c_double, vp]
    L.graft_set_thresholds.argtypes = [vp, vp]
    L.graft_template.argtypes = [i32, i32, i32, vp, vp, vp]
    L.graft_coverage.argtypes = [vp, i32, vp, vp, vp, vp, i64, vp, vp]
    L.graft_verify_update_sample.argtypes = [vp, i32, vp, vp, vp, vp, vp, i64, ctypes.c_float, vp, vp, vp, vp, vp]
    L.graft_get_matrix.argtypes = [vp, vp, vp]
    L.graft_set_matrix.argtypes = [vp, vp, vp]
    L.graft_matrix_device_ptr.argtypes = [vp]
    L.graft_matrix_device_ptr.restype = vp
    L.graft_sync.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    L.graft_last_error.argtypes = [vp]
    L.graft_last_error.restype = ctypes.c_char_p
    L.graft_last_launch_count.argtypes = [vp]
    L.graft_last_launch_count.restype = i32
    L.graft_set_wait_limit.argtypes = [vp, ctypes.c_uint32]
    L.graft_set_wait_limit.restype = ctypes.c_int
    L.graft_profile_enable.argtypes = [vp, i32]
    L.graft_profile_enable.restype = ctypes.c_int
    L.graft_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), i32]
    L.graft_profile_read.restype = ctypes.c_int
    L.graft_verify_update_noalloc.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp]
    L.graft_verify_update_noalloc.restype = ctypes.c_int
    for name in ("graft_init", "graft_destroy", "graft_warmup", "graft_assemble", "graft_assemble_src",
                 "graft_verify_update", "graft_get_matrix", "graft_set_matrix", "graft_sync"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    return vp(t.data_ptr())


def _dtypes(*names):
    import torch
    return tuple(getattr(torch, n) for n in names if hasattr(torch, n))


def _on_device(t) -> bool:
    return bool(t.is_cuda)


def _buf(t, name, dtypes, numel):
    """Pointer to a caller's device buffer of at least `numel` elements of
    one of `dtypes`, laid out contiguously.  None passes through as a null
    pointer (the library decides where one is allowed)."""
    if t is None:
        return None
    if not hasattr(t, "data_ptr") or not hasattr(t, "is_cuda"):
        raise GraftError(GRAFT_EINVAL, f"{name}: expected a torch tensor, got {type(t).__name__}")
    if t.dtype not in dtypes:
        raise GraftError(GRAFT_EINVAL, f"{name}: dtype {t.dtype}, expected {' or '.join(map(str, dtypes))}")
    if not t.is_contiguous():
        raise GraftError(GRAFT_EINVAL, f"{name}: must be contiguous")
    if t.numel() < numel:
        raise GraftError(GRAFT_EINVAL, f"{name}: {t.numel()} elements, the call needs {numel}")
    if not _on_device(t):
        raise GraftError(GRAFT_EINVAL, f"{name}: expected a CUDA tensor (device buffer), got {t.device}")
    return vp(t.data_ptr())


def _rows(t, name, dtype, rows, vocab):
    """(pointer, row stride) of logits rows: rows of >= `vocab` unit-stride
    elements at one common stride (any leading shape that merges into one row
    dimension), at least `rows` of them."""
    if t is None:
        return None, vocab
    if not hasattr(t, "data_ptr") or not hasattr(t, "is_cuda"):
        raise GraftError(GRAFT_EINVAL, f"{name}: expected a torch tensor, got {type(t).__name__}")
    if t.dtype != dtype:
        raise GraftError(GRAFT_EINVAL, f"{name}: dtype {t.dtype}, the handle's logits are {dtype}")
    if t.dim() < 2 or t.stride(-1) != 1 or t.shape[-1] < vocab:
        raise GraftError(GRAFT_EINVAL, f"{name}: expected rows [..., >= {vocab}] with unit stride in the last dim")
    try:
        t2 = t.view(-1, t.shape[-1])
    except RuntimeError:
        raise GraftError(GRAFT_EINVAL, f"{name}: the leading dims do not merge into rows at one stride") from None
    if t2.shape[0] < rows:
        raise GraftError(GRAFT_EINVAL, f"{name}: {t2.shape[0]} rows, the call needs {rows}")
    if not _on_device(t):
        raise GraftError(GRAFT_EINVAL, f"{name}: expected a CUDA tensor (device buffer), got {t.device}")
    return vp(t.data_ptr()), (t2.stride(0) if t2.shape[0] > 1 else max(t2.stride(0), t.shape[-1]))


def _stream(stream):
    if stream is None:
        import torch
        return vp(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return vp(stream)
    return vp(stream.cuda_stream)


def graft_default_config(vocab, max_batch, mode=GRAFT_MODE_CHECKPOINT, logits_dtype=GRAFT_BF16, **overrides):
    cfg = graft_config()
    load().graft_default_config(ctypes.byref(cfg), vocab, max_batch, mode, logits_dtype)
    for k, v in overrides.items():
        if k in ("ckpt_depth", "ckpt_thr", "ckpt_draft"):
            arr = getattr(cfg, k)
            for i in range(3):
                arr[i] = v[i]
        else:
            setattr(cfg, k, v)
    return cfg


class Graft:
    """One libgraft handle (owns the continuation matrix on the current device)."""

    def __init__(self, cfg: graft_config):
        self.L = load()
        self.cfg = cfg
        self.S = cfg.budget + 1
        h = vp()
        rc = self.L.graft_init(ctypes.byref(cfg), ctypes.byref(h))
        if rc != GRAFT_OK:
            raise GraftError(rc, "graft_init failed (bad config, no CUDA device, or out of memory)")
        self.h = h

    def _check(self, rc):
        if rc != GRAFT_OK:
            raise GraftError(rc, self.L.graft_last_error(self.h).decode())

    def close(self):
        if self.h:
            self.L.graft_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- entry points (same names as the C ABI, without the prefix) ---------------
    def _logits_dtype(self):
        import torch
        return torch.bfloat16 if self.cfg.logits_dtype == GRAFT_BF16 else torch.float32

    def _tree(self, batch, tree_tok, tree_parent, tree_pos, tree_mask):
        n = max(batch, 0) * self.S
        return (_buf(tree_tok, "tree_tok", _dtypes("int32"), n), _buf(tree_parent, "tree_parent", _dtypes("int8"), n),
                _buf(tree_pos, "tree_pos", _dtypes("int32"), n),
                _buf(tree_mask, "tree_mask", _dtypes("int64", "uint64"), n))

    def _draft(self, batch, draft_tok, draft_parent, draft_aux, n):
        m = max(batch, 0) * n
        return (_buf(draft_tok, "draft_tok", _dtypes("int32"), m), _buf(draft_parent, "draft_parent", _dtypes("int16"), m),
                _buf(draft_aux, "draft_prob", _dtypes("float32"), m))

    def warmup(self, tokens, logits, stream=None):
        """tokens: int32 [N] CUDA; logits: [N, >=V] CUDA (bf16 or float32)."""
        n = tokens.numel()
        pt = _buf(tokens, "tokens", _dtypes("int32"), n)
        pl, stride = _rows(logits, "logits", self._logits_dtype(), n, self.cfg.vocab)
        self._check(self.L.graft_warmup(self.h, pt, pl, n, stride if n else self.cfg.vocab, _stream(stream)))

    def assemble(self, batch, root_tok, draft_tok, draft_parent, draft_aux, tree_tok, tree_parent, tree_pos, tree_mask,
                 info, stream=None, slot_src=None):
        """With slot_src (int8 [batch, S]), also where each slot's token came
        from: 0 root, 1 draft, 2 matrix (retrieval), -1 pad."""
        n = draft_tok.shape[-1]
        args = (_buf(root_tok, "root_tok", _dtypes("int32"), max(batch, 0)),
                *self._draft(batch, draft_tok, draft_parent, draft_aux, n),
                *self._tree(batch, tree_tok, tree_parent, tree_pos, tree_mask),
                _buf(info, "info", _dtypes("int32"), max(batch, 0) * 4))
        if slot_src is None:
            self._check(self.L.graft_assemble(self.h, batch, *args[:4], n, *args[4:], _stream(stream)))
        else:
            src = _buf(slot_src, "slot_src", _dtypes("int8"), max(batch, 0) * self.S)
            self._check(self.L.graft_assemble_src(self.h, batch, *args[:4], n, *args[4:], src, _stream(stream)))

    # incremental drafting (checkpoint mode): see graft_check in include/graft.h
    def check(self, batch, draft_parent, draft_prob, layer, event, stream=None):
        n = draft_parent.shape[-1]
        m = max(batch, 0) * n
        self._check(self.L.graft_check(self.h, batch, _buf(draft_parent, "draft_parent", _dtypes("int16"), m),
                                       _buf(draft_prob, "draft_prob", _dtypes("float32"), m), n, layer,
                                       _buf(event, "event", _dtypes("int32"), max(batch, 0)), _stream(stream)))

    def retrieve(self, batch, root_tok, event, retrieved, stream=None):
        b = max(batch, 0)
        self._check(self.L.graft_retrieve(self.h, batch, _buf(root_tok, "root_tok", _dtypes("int32"), b),
                                          _buf(event, "event", _dtypes("int32"), b),
                                          _buf(retrieved, "retrieved", _dtypes("int32"), b * self.cfg.budget),
                                          _stream(stream)))

    def assemble_staged(self, batch, root_tok, draft_tok, draft_parent, draft_prob, event, retrieved, tree_tok,
                        tree_parent, tree_pos, tree_mask, info, stream=None):
        n = draft_tok.shape[-1]
        b = max(batch, 0)
        args = (_buf(root_tok, "root_tok", _dtypes("int32"), b),
                *self._draft(batch, draft_tok, draft_parent, draft_prob, n),
                _buf(event, "event", _dtypes("int32"), b),
                _buf(retrieved, "retrieved", _dtypes("int32"), b * self.cfg.budget),
                *self._tree(batch, tree_tok, tree_parent, tree_pos, tree_mask),
                _buf(info, "info", _dtypes("int32"), b * 4))
        self._check(self.L.graft_assemble_staged(self.h, batch, *args[:4], n, *args[4:], _stream(stream)))

    # threshold calibration and the coverage diagnostic
    def confidence(self, batch, draft_parent, draft_prob, best, stream=None):
        n = draft_parent.shape[-1]
        m = max(batch, 0) * n
        self._check(self.L.graft_confidence(self.h, batch, _buf(draft_parent, "draft_parent", _dtypes("int16"), m),
                                            _buf(draft_prob, "draft_prob", _dtypes("float32"), m), n,
                                            _buf(best, "best", _dtypes("float32"), max(batch, 0) * 3),
                                            _stream(stream)))

    def set_thresholds(self, thr):
        t = (ctypes.c_float * 3)(*[float(x) for x in thr])
        self._check(self.L.graft_set_thresholds(self.h, t))

    def coverage(self, batch, tree_tok, tree_parent, info, logits, gain, stream=None):
        b = max(batch, 0)
        pl, stride = _rows(logits, "logits", self._logits_dtype(), b * self.S, self.cfg.vocab)
        self._check(self.L.graft_coverage(self.h, batch, _buf(tree_tok, "tree_tok", _dtypes("int32"), b * self.S),
                                          _buf(tree_parent, "tree_parent", _dtypes("int8"), b * self.S),
                                          _buf(info, "info", _dtypes("int32"), b * 4), pl, stride,
                                          _buf(gain, "gain", _dtypes("float32"), b), _stream(stream)))

    def verify_update(self, batch, tree_tok, tree_parent, tree_pos, tree_mask, logits, accept_len, out_tokens,
                      stream=None):
        """logits: [batch*S, >=V] rows (any leading shape that merges into rows; the last dim's stride is 1)."""
        b = max(batch, 0)
        tree = self._tree(batch, tree_tok, tree_parent, tree_pos, tree_mask)
        pl, stride = _rows(logits, "logits", self._logits_dtype(), b * self.S, self.cfg.vocab)
        self._check(self.L.graft_verify_update(self.h, batch, *tree, pl, stride,
                                               _buf(accept_len, "accept_len", _dtypes("int32"), b),
                                               _buf(out_tokens, "out_tokens", _dtypes("int32"), b * self.S),
                                               _stream(stream)))

    def verify_update_sample(self, batch, tree_tok, tree_parent, tree_pos, tree_mask, logits, temperature, u_accept,
                             u_resid, accept_len, out_tokens, stream=None):
        b = max(batch, 0)
        tree = self._tree(batch, tree_tok, tree_parent, tree_pos, tree_mask)
        pl, stride = _rows(logits, "logits", self._logits_dtype(), b * self.S, self.cfg.vocab)
        self._check(self.L.graft_verify_update_sample(self.h, batch, *tree, pl, stride, ctypes.c_float(temperature),
                                                      _buf(u_accept, "u_accept", _dtypes("float32"), b * self.S),
                                                      _buf(u_resid, "u_resid", _dtypes("float32"), b),
                                                      _buf(accept_len, "accept_len", _dtypes("int32"), b),
                                                      _buf(out_tokens, "out_tokens", _dtypes("int32"), b * self.S),
                                                      _stream(stream)))

    def get_matrix(self, stream=None) -> np.ndarray:
        out = np.empty((self.cfg.vocab, K), np.int32)
        self._check(self.L.graft_get_matrix(self.h, out.ctypes.data_as(vp), _stream(stream)))
        return out

    def set_matrix(self, m: np.ndarray, stream=None):
        m = np.ascontiguousarray(m, np.int32)
        if m.shape != (self.cfg.vocab, K):
            raise GraftError(GRAFT_EINVAL, f"set_matrix: shape {m.shape}, expected ({self.cfg.vocab}, {K})")
        self._check(self.L.graft_set_matrix(self.h, m.ctypes.data_as(vp), _stream(stream)))

    def matrix_device_ptr(self) -> int:
        return int(self.L.graft_matrix_device_ptr(self.h))

    def sync(self, stream=None, raise_on_error=True) -> int:
        flags = ctypes.c_uint32(0)
        rc = self.L.graft_sync(self.h, _stream(stream), ctypes.byref(flags))
        if raise_on_error:
            self._check(rc)
        return int(flags.value)

    def last_error(self) -> str:
        return self.L.graft_last_error(self.h).decode()

    def profile_enable(self, on=True):
        self._check(self.L.graft_profile_enable(self.h, 1 if on else 0))

    def profile_read(self, max_kernels=64):
        """[(kernel name, milliseconds)] of the kernels launched since the last read."""
        names = (ctypes.c_char_p * max_kernels)()
        ms = (ctypes.c_float * max_kernels)()
        n = self.L.graft_profile_read(self.h, names, ms, max_kernels)
        if n < 0:
            self._check(n)
        return [(names[i].decode(), float(ms[i])) for i in range(n)]

    def last_launch_count(self) -> int:
        return int(self.L.graft_last_launch_count(self.h))

    def set_wait_limit(self, polls: int):
        """Poll limit of the bulk-copy kernels' mbarrier waits (0 = the default)."""
        self._check(self.L.graft_set_wait_limit(self.h, int(polls)))


class TreeBuffers:
    """Device buffers of flattened trees for `batch` requests of S slots."""

    def __init__(self, batch, S, device):
        import torch
        self.tok = torch.empty((batch, S), dtype=torch.int32, device=device)
        self.parent = torch.empty((batch, S), dtype=torch.int8, device=device)
        self.pos = torch.empty((batch, S), dtype=torch.int32, device=device)
        self.mask = torch.empty((batch, S), dtype=torch.int64, device=device)
        self.info = torch.empty((batch, 4), dtype=torch.int32, device=device)
        self.accept_len = torch.empty((batch,), dtype=torch.int32, device=device)
        self.out_tokens = torch.empty((batch, S), dtype=torch.int32, device=device)
