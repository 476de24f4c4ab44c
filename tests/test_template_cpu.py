"""The library's retrieval template (host code in libgraft.so, built by
best-first expansion) against the oracle's (enumerated by rank-sum bound and
sorted) on the CPU, for every depth and width the configuration accepts.

The two are written independently; the GPU parity tests compare them only
through the trees of a few configurations.  Source: popular-science article
on arXiv 2605.20104, section 二 (second gear: the asymmetric template) and
section 五 (template depth and width ablations).
"""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def lib_template():
    import hybrid_draft_tree_gb300 as g
    from hybrid_draft_tree_gb300 import _build
    _build.build()
    return g.template


@pytest.mark.parametrize("depth", [1, 2, 3, 5, 8, 10, 12, 16])
@pytest.mark.parametrize("width", [1, 2, 3, 4, 7, 8, 16, 64])
def test_library_template_equals_the_oracle(lib_template, depth, width):
    for length in (0, 1, 8, 20, 36, 52, 60, 256):
        lp, lr, ld = lib_template(depth, width, length)
        op, orank, od = oracle.template(length, depth=depth, width=width)
        assert np.array_equal(lp, op) and np.array_equal(lr, orank) and np.array_equal(ld, od), (depth, width, length)


def test_library_template_rejects_bad_arguments(lib_template):
    import hybrid_draft_tree_gb300 as g
    for depth, width, length in ((0, 8, 10), (17, 8, 10), (8, 0, 10), (8, 65, 10), (8, 8, -1), (8, 8, 65537)):
        with pytest.raises(g.GraftError):
            lib_template(depth, width, length)


def test_default_template_head(lib_template):
    """The default (depth 8, width 8): the rank-0 chain to depth 8 first,
    then the single-deviation branches of rank sum 1."""
    par, rank, dep = lib_template(8, 8, 11)
    assert list(dep[:8]) == list(range(1, 9)) and not rank[:8].any()
    assert list(par[:8]) == [-1] + list(range(7))
    assert list(zip(par[8:], rank[8:], dep[8:])) == [(-1, 1, 1), (0, 1, 2), (8, 0, 2)]
