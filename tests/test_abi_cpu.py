"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, and
exports every entry point include/graft.h declares; the binding's struct
matches the header's layout.  No kernel runs here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "graft.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(graft_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("graft_init", "graft_destroy", "graft_warmup", "graft_assemble", "graft_verify_update",
              "graft_get_matrix", "graft_set_matrix", "graft_sync", "graft_last_error"):
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    import hybrid_draft_tree_gb300 as g
    from hybrid_draft_tree_gb300 import _build
    _build.build()
    lib = ctypes.CDLL(g.library_path())
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert sorted(g.EXPORTS) == declared_functions()


def test_config_struct_layout_and_defaults():
    import hybrid_draft_tree_gb300 as g
    cfg = g.graft_default_config(151936, 16, g.GRAFT_MODE_STATIC, g.GRAFT_BF16)
    assert ctypes.sizeof(cfg) == 4 * 23
    assert (cfg.vocab, cfg.topk, cfg.budget, cfg.max_batch) == (151936, 8, 60, 16)
    assert list(cfg.ckpt_depth) == [0, 1, 5]
    assert [round(x, 6) for x in cfg.ckpt_thr] == [0.3, 0.2, 0.1]
    assert list(cfg.ckpt_draft) == [8, 24, 40]
    assert (cfg.tpl_depth, cfg.tpl_width) == (8, 8)
    assert abs(cfg.static_thr - 0.15) < 1e-7 and abs(cfg.tail_thr - 0.4) < 1e-7
    assert (cfg.scan_kernel, cfg.ablation, cfg.fixed_draft) == (0, 0, 40)
    tail = g.graft_default_config(151936, 64, g.GRAFT_MODE_TAIL, g.GRAFT_BF16)
    assert tail.budget == 16 and tail.max_draft_nodes == 16


def test_config_struct_matches_the_c_header(tmp_path):
    """The binding's graft_config has the header's size and field offsets."""
    import shutil
    import subprocess
    import hybrid_draft_tree_gb300 as g
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    names = [f[0] for f in g.graft.graft_config._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stddef.h>\n#include <stdio.h>\n#include \"graft.h\"\nint main(void) {\n"
                   "  printf(\"%zu\\n\", sizeof(graft_config));\n" +
                   "".join(f"  printf(\"%zu\\n\", offsetof(graft_config, {n}));\n" for n in names) + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(root, "include"), str(src), "-o", str(exe)])
    out = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert out[0] == ctypes.sizeof(g.graft.graft_config)
    assert out[1:] == [getattr(g.graft.graft_config, n).offset for n in names]


def test_init_without_gpu_fails_cleanly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    import hybrid_draft_tree_gb300 as g
    with pytest.raises(g.GraftError):
        g.Graft(g.graft_default_config(100, 1, 0, g.GRAFT_BF16))


def test_config_validation_before_any_device_call():
    """graft_init checks the configuration before it touches a device: on a
    machine without a GPU a bad config is GRAFT_EINVAL and a good one reaches
    the device query (GRAFT_ECUDA)."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    import hybrid_draft_tree_gb300 as g
    from hybrid_draft_tree_gb300 import graft as gb
    L = g.load()

    def init(**kw):
        mode = kw.pop("mode", g.GRAFT_MODE_CHECKPOINT)
        cfg = g.graft_default_config(kw.pop("vocab", 1000), kw.pop("max_batch", 4), mode, kw.pop("dtype", g.GRAFT_BF16),
                                     **kw)
        h = ctypes.c_void_p()
        return L.graft_init(ctypes.byref(cfg), ctypes.byref(h))

    for mode in (g.GRAFT_MODE_CHECKPOINT, g.GRAFT_MODE_STATIC, g.GRAFT_MODE_TAIL):
        for dtype in (g.GRAFT_F32, g.GRAFT_BF16):
            assert init(mode=mode, dtype=dtype) == gb.GRAFT_ECUDA
    assert init(ablation=2, fixed_draft=0, tpl_depth=16, tpl_width=64, scan_kernel=4) == gb.GRAFT_ECUDA
    assert init(scan_kernel=5) == gb.GRAFT_ECUDA
    assert init(budget=63, max_batch=1000) == gb.GRAFT_ECUDA          # the largest budget and batch * slots
    bad = [dict(vocab=0), dict(topk=4), dict(budget=0), dict(budget=64), dict(max_batch=0), dict(max_batch=1100),
           dict(mode=3), dict(dtype=2), dict(ckpt_draft=(8, 24, 61)), dict(ckpt_depth=(0, -1, 5)),
           dict(tpl_depth=0), dict(tpl_depth=17), dict(tpl_width=0), dict(tpl_width=65), dict(ablation=3),
           dict(ablation=1, mode=g.GRAFT_MODE_STATIC), dict(ablation=2, fixed_draft=61), dict(max_draft_nodes=-1),
           dict(max_draft_nodes=17, mode=g.GRAFT_MODE_TAIL), dict(scan_kernel=6), dict(ckpt_thr=(0.3, 1.5, 0.1)),
           dict(ckpt_thr=(float("nan"), 0.2, 0.1)), dict(static_thr=-0.1, mode=g.GRAFT_MODE_STATIC),
           dict(tail_thr=float("inf"), mode=g.GRAFT_MODE_TAIL)]
    for kw in bad:
        assert init(**dict(kw)) == gb.GRAFT_EINVAL, kw


def test_noalloc_argument_checks_before_any_device_call():
    """graft_verify_update_noalloc refuses bad sizes and null buffers before
    it touches a device; a batch of 0 is a no-op.  No pointer is
    dereferenced on these paths (the last call stops at the device setup)."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    import hybrid_draft_tree_gb300 as g
    from hybrid_draft_tree_gb300 import graft as gb
    L = g.load()
    some = ctypes.c_void_p(4096)            # never dereferenced: every call below returns before any access

    def call(V=1000, dt=g.GRAFT_BF16, B=2, S=61, stride=1000, ptr=some, logits=None, mask=None):
        lg = ptr if logits is None else logits
        mk = ptr if mask is None else mask
        return L.graft_verify_update_noalloc(V, dt, B, S, ptr, ptr, ptr, mk, lg, ctypes.c_int64(stride), ptr, ptr,
                                             ptr, ptr, ctypes.c_void_p(0))

    assert call(B=0) == gb.GRAFT_OK
    for kw in (dict(V=0), dict(dt=2), dict(S=0), dict(S=65), dict(B=-1), dict(B=2048 // 61 + 1), dict(stride=999),
               dict(ptr=ctypes.c_void_p(None)), dict(ptr=ctypes.c_void_p(4098)),       # int32 buffers off 4 bytes
               dict(logits=ctypes.c_void_p(4097)),                                      # bf16 logits off 2 bytes
               dict(dt=g.GRAFT_F32, logits=ctypes.c_void_p(4098)),                      # fp32 logits off 4 bytes
               dict(mask=ctypes.c_void_p(4100))):                                       # uint64 masks off 8 bytes
        assert call(**kw) == gb.GRAFT_EINVAL, kw
    assert call() not in (gb.GRAFT_OK, gb.GRAFT_EINVAL)     # valid arguments: stops at the missing device
    assert call(logits=ctypes.c_void_p(4098)) not in (gb.GRAFT_OK, gb.GRAFT_EINVAL)   # bf16 on a 2-byte boundary


def test_product_code_never_loads_the_oracle():
    """The library, its binding and the input generators neither import the
    oracle nor name its library; the benchmark imports it only inside the
    CPU-baseline function (its reference leg), and libgraft.so links nothing
    of it."""
    import ast
    import subprocess
    for sub in ("hybrid_draft_tree_gb300", "workloads", "include"):
        for dirpath, _, files in os.walk(os.path.join(ROOT, sub)):
            for f in files:
                path = os.path.join(dirpath, f)
                if f.endswith(".py"):
                    tree = ast.parse(open(path).read())
                    for node in ast.walk(tree):
                        if isinstance(node, ast.Import):
                            assert all(a.name.split(".")[0] != "oracle" for a in node.names), path
                        if isinstance(node, ast.ImportFrom):
                            assert (node.module or "").split(".")[0] != "oracle", path
                if f.endswith((".py", ".cu", ".cuh", ".c", ".h")):
                    assert "graft_oracle" not in open(path).read(), path
    bench = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    importers = [fn.name for fn in ast.walk(bench) if isinstance(fn, ast.FunctionDef)
                 for node in ast.walk(fn) if isinstance(node, ast.Import) and any(a.name == "oracle" for a in node.names)]
    assert importers == ["oracle_sample"]
    assert not any(isinstance(node, ast.Import) and any(a.name == "oracle" for a in node.names) for node in bench.body)
    import hybrid_draft_tree_gb300 as g
    from hybrid_draft_tree_gb300 import _build
    _build.build()
    deps = subprocess.run(["ldd", g.library_path()], capture_output=True, text=True).stdout
    assert "oracle" not in deps


def test_oracle_shares_no_code_with_the_library():
    """The oracle neither imports the package nor includes the library's
    headers or sources (the two share only the seeded input generators)."""
    odir = os.path.join(ROOT, "oracle")
    for f in os.listdir(odir):
        if f.endswith((".py", ".c", ".h")):
            src = open(os.path.join(odir, f)).read()
            for needle in ("hybrid_draft_tree_gb300", "graft.h", "graft_internal", "csrc", "libgraft.so"):
                assert needle not in src, (f, needle)
