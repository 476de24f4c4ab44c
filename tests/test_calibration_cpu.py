"""Threshold calibration on the host (article section 二: checkpoint
thresholds set from the path confidences seen during warm-up): the library's
nearest-rank quantile equals numpy's inverted-CDF quantile.  No GPU needed."""
import numpy as np
import pytest


@pytest.mark.parametrize("n", [1, 2, 7, 50, 333])
@pytest.mark.parametrize("q", [0.05, 0.1, 0.3, 0.5, 0.9, 1.0])
def test_calibration_is_the_nearest_rank_quantile(n, q):
    import hybrid_draft_tree_gb300 as g
    rng = np.random.default_rng(n)
    best = rng.random((n, 3)).astype(np.float32)
    best[rng.random((n, 3)) < 0.1] = -1.0          # empty checkpoint layers are skipped
    best[0] = 0.5
    got = g.calibrate_thresholds(best, q)
    expect = [np.quantile(best[best[:, k] >= 0, k], q, method="inverted_cdf") for k in range(3)]
    assert np.array_equal(got, np.array(expect, np.float32))


def test_calibration_rejects_bad_input():
    import hybrid_draft_tree_gb300 as g
    with pytest.raises(g.GraftError):
        g.calibrate_thresholds(np.full((4, 3), -1.0, np.float32), 0.5)    # no sample at all
    with pytest.raises(g.GraftError):
        g.calibrate_thresholds(np.full((4, 3), 0.5, np.float32), 0.0)     # quantile outside (0, 1]
