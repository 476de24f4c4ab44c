"""The binding's argument checks, on the CPU: a buffer the C ABI would read
or write through a raw device pointer is refused (GraftError, GRAFT_EINVAL)
when it is not CUDA memory, has the wrong element type or layout, or is too
small for the batch -- before anything reaches the library.  Host tensors
stand in for every buffer, so each call must stop in the binding."""
import ctypes

import pytest

torch = pytest.importorskip("torch")

import hybrid_draft_tree_gb300 as g  # noqa: E402
from hybrid_draft_tree_gb300 import graft as gb  # noqa: E402


class _FakeLib:
    """Stands in for the loaded library: records each entry point's
    arguments and returns GRAFT_OK."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


def _handle(mode=g.GRAFT_MODE_CHECKPOINT, dtype=g.GRAFT_BF16, V=100, B=2):
    eng = object.__new__(g.Graft)
    eng.L = _FakeLib()
    eng.cfg = g.graft_default_config(V, B, mode, dtype)
    eng.S = eng.cfg.budget + 1
    eng.h = None
    return eng


def _bufs(B=2, S=61, n=184, V=100, ldt=torch.bfloat16):
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32)
    return dict(root=i32(B), dtok=i32(B, n), dpar=torch.zeros((B, n), dtype=torch.int16),
                daux=torch.zeros((B, n)), ttok=i32(B, S), tpar=torch.zeros((B, S), dtype=torch.int8),
                tpos=i32(B, S), tmask=torch.zeros((B, S), dtype=torch.int64), info=i32(B, 4),
                logits=torch.zeros((B * S, V), dtype=ldt), acc=i32(B), out=i32(B, S), event=i32(B),
                retrieved=i32(B, 60), best=torch.zeros((B, 3)), gain=torch.zeros(B),
                u=torch.zeros((B, S)), ur=torch.zeros(B))


def _calls(eng, b):
    s = dict(stream=0)
    return {
        "assemble": lambda: eng.assemble(2, b["root"], b["dtok"], b["dpar"], b["daux"], b["ttok"], b["tpar"],
                                         b["tpos"], b["tmask"], b["info"], **s),
        "assemble_staged": lambda: eng.assemble_staged(2, b["root"], b["dtok"], b["dpar"], b["daux"], b["event"],
                                                       b["retrieved"], b["ttok"], b["tpar"], b["tpos"], b["tmask"],
                                                       b["info"], **s),
        "check": lambda: eng.check(2, b["dpar"], b["daux"], 0, b["event"], **s),
        "retrieve": lambda: eng.retrieve(2, b["root"], b["event"], b["retrieved"], **s),
        "confidence": lambda: eng.confidence(2, b["dpar"], b["daux"], b["best"], **s),
        "coverage": lambda: eng.coverage(2, b["ttok"], b["tpar"], b["info"], b["logits"], b["gain"], **s),
        "verify_update": lambda: eng.verify_update(2, b["ttok"], b["tpar"], b["tpos"], b["tmask"], b["logits"],
                                                   b["acc"], b["out"], **s),
        "verify_update_sample": lambda: eng.verify_update_sample(2, b["ttok"], b["tpar"], b["tpos"], b["tmask"],
                                                                 b["logits"], 1.0, b["u"], b["ur"], b["acc"],
                                                                 b["out"], **s),
        "warmup": lambda: eng.warmup(b["root"], b["logits"][:2], **s),
    }


CALLS = ["assemble", "assemble_staged", "check", "retrieve", "confidence", "coverage", "verify_update",
         "verify_update_sample", "warmup"]


@pytest.fixture
def as_device(monkeypatch):
    """Host tensors pass the device test, so the other checks and the
    marshalling can be exercised without a GPU."""
    monkeypatch.setattr(gb, "_on_device", lambda t: True)


@pytest.mark.parametrize("call", CALLS)
def test_host_buffers_are_refused(call):
    eng = _handle()
    with pytest.raises(g.GraftError, match="CUDA tensor") as e:
        _calls(eng, _bufs())[call]()
    assert e.value.code == gb.GRAFT_EINVAL
    assert eng.L.calls == []


def _p(t):
    return None if t is None else t.data_ptr()


def _vals(args):
    return [a.value if isinstance(a, (ctypes.c_void_p, ctypes.c_float)) else a for a in args]


def test_valid_buffers_reach_the_library_in_abi_order(as_device):
    """Every entry point receives the handle, the batch, the buffers' data
    pointers in the order include/graft.h declares, the draft width, the row
    stride and the stream."""
    eng = _handle()
    b = _bufs()
    for name in CALLS:
        _calls(eng, b)[name]()
    got = {name: _vals(args) for name, args in eng.L.calls}
    assert len(got) == len(CALLS)
    h, S, V = None, 61, 100
    assert got["graft_assemble"] == [h, 2, _p(b["root"]), _p(b["dtok"]), _p(b["dpar"]), _p(b["daux"]), 184,
                                     _p(b["ttok"]), _p(b["tpar"]), _p(b["tpos"]), _p(b["tmask"]), _p(b["info"]), None]
    assert got["graft_assemble_staged"] == [h, 2, _p(b["root"]), _p(b["dtok"]), _p(b["dpar"]), _p(b["daux"]), 184,
                                            _p(b["event"]), _p(b["retrieved"]), _p(b["ttok"]), _p(b["tpar"]),
                                            _p(b["tpos"]), _p(b["tmask"]), _p(b["info"]), None]
    assert got["graft_check"] == [h, 2, _p(b["dpar"]), _p(b["daux"]), 184, 0, _p(b["event"]), None]
    assert got["graft_retrieve"] == [h, 2, _p(b["root"]), _p(b["event"]), _p(b["retrieved"]), None]
    assert got["graft_confidence"] == [h, 2, _p(b["dpar"]), _p(b["daux"]), 184, _p(b["best"]), None]
    assert got["graft_coverage"] == [h, 2, _p(b["ttok"]), _p(b["tpar"]), _p(b["info"]), _p(b["logits"]), V,
                                     _p(b["gain"]), None]
    assert got["graft_verify_update"] == [h, 2, _p(b["ttok"]), _p(b["tpar"]), _p(b["tpos"]), _p(b["tmask"]),
                                          _p(b["logits"]), V, _p(b["acc"]), _p(b["out"]), None]
    assert got["graft_verify_update_sample"] == [h, 2, _p(b["ttok"]), _p(b["tpar"]), _p(b["tpos"]), _p(b["tmask"]),
                                                 _p(b["logits"]), V, 1.0, _p(b["u"]), _p(b["ur"]), _p(b["acc"]),
                                                 _p(b["out"]), None]
    assert got["graft_warmup"] == [h, _p(b["root"]), _p(b["logits"]), 2, V, None]
    assert S == eng.S


def test_tail_mode_draft_parent_may_be_null(as_device):
    eng = _handle(mode=g.GRAFT_MODE_TAIL, B=2)
    b = _bufs(S=17, n=16)
    eng.assemble(2, b["root"], b["dtok"], None, b["daux"], b["ttok"], b["tpar"], b["tpos"], b["tmask"], b["info"],
                 stream=0)
    (name, args), = eng.L.calls
    assert name == "graft_assemble" and _vals(args)[4] is None and _vals(args)[6] == 16


def test_batch_zero_takes_null_buffers(as_device):
    eng = _handle()
    eng.verify_update(0, None, None, None, None, torch.zeros((1, 100), dtype=torch.bfloat16), None, None, stream=0)
    (name, args), = eng.L.calls
    assert _vals(args)[2:6] == [None] * 4 and _vals(args)[7] == 100


def test_strided_rows_pass_their_stride(as_device):
    """Rows at a wider stride (padding after the vocabulary) and [B, S, V]
    logits are passed with their row stride."""
    eng = _handle()
    b = _bufs()
    wide = torch.zeros((2 * 61, 136), dtype=torch.bfloat16)[:, :100]
    b["logits"] = wide
    _calls(eng, b)["verify_update"]()
    b["logits"] = torch.zeros((2, 61, 100), dtype=torch.bfloat16)
    _calls(eng, b)["verify_update"]()
    assert [_vals(a)[7] for _, a in eng.L.calls] == [136, 100]


@pytest.mark.parametrize("key,bad", [
    ("ttok", torch.zeros((2, 61), dtype=torch.int64)),        # wrong element type
    ("tpar", torch.zeros((2, 61), dtype=torch.int32)),
    ("tmask", torch.zeros((2, 61), dtype=torch.int32)),
    ("acc", torch.zeros(1, dtype=torch.int32)),               # too small for the batch
    ("out", torch.zeros((2, 60), dtype=torch.int32)),
    ("tpos", torch.zeros((61, 2), dtype=torch.int32).t()),    # not contiguous
    ("logits", torch.zeros((2 * 61, 100), dtype=torch.float32)),   # not the handle's logits type
    ("logits", torch.zeros((2 * 61, 99), dtype=torch.bfloat16)),   # rows shorter than the vocabulary
    ("logits", torch.zeros((2 * 61 - 1, 100), dtype=torch.bfloat16)),   # too few rows
    ("logits", torch.zeros((100, 2 * 61), dtype=torch.bfloat16).t()),   # elements not at unit stride
])
def test_verify_update_checks_each_buffer(as_device, key, bad):
    eng = _handle()
    b = _bufs()
    b[key] = bad
    with pytest.raises(g.GraftError) as e:
        _calls(eng, b)["verify_update"]()
    assert e.value.code == gb.GRAFT_EINVAL and eng.L.calls == []


@pytest.mark.parametrize("key,bad", [
    ("root", torch.zeros(1, dtype=torch.int32)),
    ("dtok", torch.zeros((2, 184), dtype=torch.int16)),
    ("dpar", torch.zeros((2, 184), dtype=torch.int32)),
    ("daux", torch.zeros((2, 184), dtype=torch.float64)),
    ("info", torch.zeros((2, 3), dtype=torch.int32)),
])
def test_assemble_checks_each_buffer(as_device, key, bad):
    eng = _handle()
    b = _bufs()
    b[key] = bad
    with pytest.raises(g.GraftError) as e:
        _calls(eng, b)["assemble"]()
    assert e.value.code == gb.GRAFT_EINVAL and eng.L.calls == []


def test_retrieved_must_hold_the_budget(as_device):
    eng = _handle()
    b = _bufs()
    b["retrieved"] = torch.zeros((2, 59), dtype=torch.int32)
    with pytest.raises(g.GraftError, match="elements"):
        _calls(eng, b)["retrieve"]()


def test_logits_rows_must_merge_into_one_stride(as_device):
    """Leading dims that do not merge into rows at one stride are refused
    (the library takes one row stride)."""
    x = torch.zeros((2, 61, 128), dtype=torch.bfloat16)
    assert gb._rows(x[:, :, :100], "logits", torch.bfloat16, 122, 100)[1] == 128
    with pytest.raises(g.GraftError, match="merge"):
        gb._rows(x[:, :60, :], "logits", torch.bfloat16, 120, 100)


def test_none_is_a_null_pointer():
    assert gb._buf(None, "x", gb._dtypes("int32"), 10) is None
    assert gb._rows(None, "logits", torch.bfloat16, 0, 100) == (None, 100)
    assert isinstance(ctypes.c_void_p(None), ctypes.c_void_p)


def test_empty_draft_is_passed_with_width_zero(as_device):
    eng = _handle(B=1)
    b = _bufs(B=1)
    empty = lambda dt: torch.zeros((1, 0), dtype=dt)
    eng.assemble(1, b["root"], empty(torch.int32), empty(torch.int16), empty(torch.float32), b["ttok"], b["tpar"],
                 b["tpos"], b["tmask"], b["info"], stream=0)
    (name, args), = eng.L.calls
    assert _vals(args)[6] == 0


def test_set_matrix_checks_its_shape():
    import numpy as np
    eng = _handle(V=100)
    with pytest.raises(g.GraftError, match="shape"):
        eng.set_matrix(np.zeros((99, 8), np.int32), stream=0)
    eng.set_matrix(np.zeros((100, 8), np.int64), stream=0)        # converted to int32 on the host
    (name, args), = eng.L.calls
    assert name == "graft_set_matrix"


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libgraft.so (and without building it) the binding raises; it
    has no other path to run the step on."""
    from hybrid_draft_tree_gb300 import _build
    monkeypatch.setattr(gb, "_lib", None)
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "libgraft.so"))
    with pytest.raises(ImportError):
        gb.load(build_if_missing=False)

    def no_nvcc(*a, **k):
        raise RuntimeError("nvcc failed")
    monkeypatch.setattr(_build, "build", no_nvcc)
    with pytest.raises(RuntimeError):
        gb.load()
    with pytest.raises(RuntimeError):
        g.Graft(g.graft.graft_config())
