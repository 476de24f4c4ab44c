"""The allocation-free verify + update entry point.

graft_verify_update_noalloc serves callers that cannot call cudaMalloc (a
decode step being captured into a CUDA graph, or an engine whose device
memory is fully pre-planned by its own arena): it takes the continuation
matrix as a caller buffer and keeps its scratch in a fixed device array
compiled into the library.  These tests call it through the C ABI and check
it against graft_verify_update on a handle holding the same matrix, for two
calls in a row (the second sees the matrix the first updated).  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest

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
        tok[b, :n] = rng.integers(0, 400, n)
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


def test_noalloc_matches_handle_entry_point_on_two_calls(lib):
    g, L = lib
    rng = np.random.default_rng(11)
    V, B, S = 40000, 8, 61
    eng = g.Graft(g.graft_default_config(V, B, g.GRAFT_MODE_CHECKPOINT, g.GRAFT_BF16))
    m0 = rng.integers(-1, V, (V, 8)).astype(np.int32)
    eng.set_matrix(m0)
    d_matrix = torch.from_numpy(m0).cuda()
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    for call in range(2):
        logits = torch.randn((B * S, V), device="cuda").to(torch.bfloat16)
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
        rc = L.graft_verify_update_noalloc(V, g.GRAFT_BF16, B, S, _p(t_tok), _p(t_par), _p(t_pos), _p(t_mask),
                                           _p(logits), ctypes.c_int64(logits.stride(0)), _p(d_matrix), _p(acc_n),
                                           _p(out_n), _p(d_err), ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(acc_n, acc_h), call
        assert torch.equal(out_n, out_h), call
        assert np.array_equal(d_matrix.cpu().numpy(), eng.get_matrix()), call
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
