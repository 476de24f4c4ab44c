"""The allocation-free verify + update entry point.

graft_verify_update_noalloc serves callers that cannot call cudaMalloc (a
decode step being captured into a CUDA graph, or an engine whose device
memory is fully pre-planned by its own arena): it takes the continuation
matrix as a caller buffer and keeps its scratch in a fixed device array
compiled into the library.  These tests call it through the C ABI and check
it, for two calls in a row (the second sees the matrix the first updated),
against graft_verify_update on a handle holding the same matrix and against
the CPU oracle's verification and update on its own copy of the matrix.
They cover fp32 and bf16 logits, a vocabulary with a tail (V % 8 != 0),
rows that start off 16-byte boundaries (the scalar-load path) and a call of
exactly GRAFT_NOALLOC_MAX_ROWS rows.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _random_trees(rng, B, S, V, logits_host):
    """Valid flattened trees; about half the nodes carry their parent's argmax
    so that acceptance paths are non-trivial; tokens repeat across rows so the
    last-writer rule matters."""
    tok = np.full((B, S), -1, np.int32)
    par = np.full((B, S), -1, np.int8)
    pos = np.full((B, S), -1, np.int32)
    mask = np.zeros((B, S), np.uint64)
    for b in range(B):
        n = int(rng.integers(S // 2, S + 1))
        tok[b, :n] = rng.integers(0, min(V, 400), n)
        pos[b, 0], mask[b, 0] = 0, 1
        for i in range(1, n):
            p = int(rng.integers(0, i))
            par[b, i] = p
            if rng.random() < 0.5:
                tok[b, i] = int(np.argmax(logits_host[b * S + p]))
            pos[b, i] = pos[b, p] + 1
            mask[b, i] = np.uint64(int(mask[b, p]) | (1 << i))
    return tok, par, pos, mask


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hybrid_draft_tree_gb300 as g
    return g, g.load()


@pytest.mark.parametrize("dtype_name,V,B,S,pad", [
    ("bf16", 40000, 8, 61, 0),       # 16-byte aligned rows, vector loads
    ("f32", 40003, 8, 61, 5),        # a tail of V % 4 elements; padded rows stay 16-byte aligned
    ("bf16", 40003, 8, 61, 0),       # odd row stride: rows start off 16-byte boundaries (scalar loads)
    ("f32", 12001, 6, 33, 2),        # odd row stride in fp32 (scalar loads)
    ("bf16", 5000, 32, 64, 0),       # batch x slots == GRAFT_NOALLOC_MAX_ROWS, 64 slots per request
])
def test_noalloc_matches_handle_and_oracle_on_two_calls(lib, dtype_name, V, B, S, pad):
    g, L = lib
    dt = g.GRAFT_BF16 if dtype_name == "bf16" else g.GRAFT_F32
    rng = np.random.default_rng(V + B + pad)
    eng = g.Graft(g.graft_default_config(V, B, g.GRAFT_MODE_CHECKPOINT, dt, budget=S - 1,
                                         ckpt_draft=(min(8, S - 1), min(24, S - 1), min(40, S - 1))))
    m0 = rng.integers(-1, V, (V, 8)).astype(np.int32)
    eng.set_matrix(m0)
    C = m0.copy()                                  # the oracle's own matrix
    d_matrix = torch.from_numpy(m0).cuda()
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    stride = V + pad
    tdt = torch.bfloat16 if dt == g.GRAFT_BF16 else torch.float32
    for call in range(2):
        full = torch.randn((B * S, stride), device="cuda").to(tdt)
        logits = full[:, :V]                       # rows at stride V + pad
        if dt == g.GRAFT_BF16:
            host_bits = full.view(torch.int16).cpu().numpy().view(np.uint16)[:, :V]
        else:
            host_bits = full.cpu().numpy()[:, :V]
        host = logits.float().cpu().numpy()
        tok, par, pos, mask = _random_trees(rng, B, S, V, host)
        t_tok = torch.from_numpy(tok).cuda()
        t_par = torch.from_numpy(par).cuda()
        t_pos = torch.from_numpy(pos).cuda()
        t_mask = torch.from_numpy(mask.view(np.int64)).cuda()
        acc_h = torch.empty(B, dtype=torch.int32, device="cuda")
        out_h = torch.empty((B, S), dtype=torch.int32, device="cuda")
        eng.verify_update(B, t_tok, t_par, t_pos, t_mask, logits, acc_h, out_h)
        acc_n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        out_n = torch.full((B, S), -7, dtype=torch.int32, device="cuda")
        rc = L.graft_verify_update_noalloc(V, dt, B, S, _p(t_tok), _p(t_par), _p(t_pos), _p(t_mask),
                                           _p(logits), ctypes.c_int64(stride), _p(d_matrix), _p(acc_n),
                                           _p(out_n), _p(d_err), ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(acc_n, acc_h), call
        assert torch.equal(out_n, out_h), call
        assert np.array_equal(d_matrix.cpu().numpy(), eng.get_matrix()), call
        # the oracle: greedy verification per request, then the update in (request, slot) order
        acc_g, out_g = acc_n.cpu().numpy(), out_n.cpu().numpy()
        for b in range(B):
            tr = oracle.Tree(S)
            tr.tok[:], tr.par[:] = tok[b], par[b].astype(np.int32)
            acc, out, topk = oracle.verify(tr, host_bits[b * S:(b + 1) * S], dt)
            oracle.update(C, tr, topk)
            assert acc_g[b] == acc and np.array_equal(out_g[b], out), (call, b)
        assert np.array_equal(d_matrix.cpu().numpy(), C), call
        assert int(d_err.item()) == 0
        assert eng.sync() == 0
    assert int(acc_h.sum().item()) > 0          # some paths were accepted
    eng.close()


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    g, L = lib
    V, S = 1000, 61
    B = 2048 // S + 1                              # rows > GRAFT_NOALLOC_MAX_ROWS
    dummy = torch.zeros(16, dtype=torch.int64, device="cuda")
    logits = torch.zeros((1, V), dtype=torch.bfloat16, device="cuda")
    rc = L.graft_verify_update_noalloc(V, g.GRAFT_BF16, B, S, _p(dummy), _p(dummy), _p(dummy), _p(dummy),
                                       _p(logits), ctypes.c_int64(V), _p(dummy), _p(dummy), _p(dummy), _p(dummy),
                                       ctypes.c_void_p(0))
    assert rc == g.graft.GRAFT_EINVAL
    rc = L.graft_verify_update_noalloc(V, g.GRAFT_BF16, 1, 65, _p(dummy), _p(dummy), _p(dummy), _p(dummy),
                                       _p(logits), ctypes.c_int64(V), _p(dummy), _p(dummy), _p(dummy), _p(dummy),
                                       ctypes.c_void_p(0))
    assert rc == g.graft.GRAFT_EINVAL           # more than 64 slots per request
