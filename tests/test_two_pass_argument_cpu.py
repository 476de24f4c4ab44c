"""The exactness argument of the two-pass verify scan, checked on a model of
its selection rule (CPU, numpy; the GPU parity tests check the kernels).

Pass 1 keeps the maximum of every unit (32 lanes x one 16-byte vector: 256
bf16 or 128 fp32 elements; the row's last V mod (elements per vector) elements
belong to no unit).  Pass 2 gives lane l of a warp the units 4i .. 4i + 3 for
i = l, l + 32, ..., takes T0 = the 8th largest of the 32 lane maxima (with
multiplicity: each knock-out round removes one lane), and keeps every element
>= T0 of the units whose maximum is >= T0 plus the tail elements >= T0.  Eight
distinct elements reach T0 (one in each of the 8 lanes holding the largest
maxima), so every element of the row's top-8 is >= T0; everything left out is
below T0.  The top-8 of the kept elements (value descending, id ascending) is
therefore the row's.  The kernel falls back to an exact rescan when T0 is
-inf (fewer than 8 finite lane maxima), when more than 128 units or more than
192 elements are kept; the model reports those cases instead.

With unit records, pass 1 also keeps each unit's second largest element
(with multiplicity: equal to the maximum when it repeats) and the lowest
position of its maximum.  A kept unit whose second largest element is below
T0 holds exactly one element >= T0, its maximum, at the recorded position;
pass 2 reads only the other kept units again.  The model checks that this
gives the same kept elements, hence the same top-8.
"""
import numpy as np
import pytest

UCAP, ECAP = 128, 192


def reference_top8(x):
    order = np.lexsort((np.arange(len(x)), -x.astype(np.float64)))
    return order[:8]


def two_pass_top8(x, epl, records=False):
    """(top-8 ids, None) from the selection rule, or (None, reason) where the
    kernel takes its exact rescan.  records: pass 2 takes single-element
    units from the unit records instead of reading them again."""
    V = len(x)
    nslot = V // epl
    upr = -(-nslot // 32)
    body = np.full(upr * 32 * epl, -np.inf)
    body[:nslot * epl] = x[:nslot * epl]
    umax = body.reshape(upr, 32 * epl).max(axis=1) if upr else np.zeros(0)
    n4 = -(-upr // 4)
    padded = np.full(n4 * 4, -np.inf)
    padded[:upr] = umax
    group_max = padded.reshape(n4, 4).max(axis=1) if n4 else np.zeros(0)   # units 4i .. 4i + 3
    lane_max = np.full(32, -np.inf)
    for i, m in enumerate(group_max):
        lane_max[i % 32] = max(lane_max[i % 32], m)
    T0 = np.sort(lane_max)[::-1][7]
    if not T0 > -np.inf:
        return None, "T0 = -inf"
    units = np.flatnonzero(umax >= T0)
    if len(units) > UCAP:
        return None, "units"
    ue = 32 * epl
    usort = -np.sort(-body.reshape(upr, ue), axis=1) if upr else np.zeros((0, 2))
    usec = usort[:, 1] if upr else np.zeros(0)                     # second largest, with multiplicity
    upos = body.reshape(upr, ue).argmax(axis=1) if upr else np.zeros(0, np.int64)   # lowest on ties
    ids = []
    for u in units:
        lo, hi = u * ue, min((u + 1) * ue, nslot * epl)
        if records and not usec[u] >= T0:
            ids.append(lo + int(upos[u]))                        # the only element >= T0
        else:
            ids.extend(lo + np.flatnonzero(x[lo:hi] >= T0))
    ids.extend(nslot * epl + np.flatnonzero(x[nslot * epl:] >= T0))
    if len(ids) > ECAP:
        return None, "elements"
    ids = np.array(ids, np.int64)
    order = np.lexsort((ids, -x[ids].astype(np.float64)))
    out = np.full(8, -1, np.int64)
    out[:min(8, len(ids))] = ids[order[:8]]
    return out, None


def _check(x, epl):
    got, why = two_pass_top8(x, epl)
    rec, why_r = two_pass_top8(x, epl, records=True)
    assert why_r == why
    if got is None:
        return why
    want = np.full(8, -1, np.int64)
    ref = reference_top8(x)
    want[:len(ref)] = ref
    assert np.array_equal(got, want)
    assert np.array_equal(rec, want)
    return None


@pytest.mark.parametrize("V", [151936, 151937, 128256, 32000, 32005, 4099, 1000])
@pytest.mark.parametrize("epl", [8, 4])
def test_selection_rule_is_exact_on_random_rows(V, epl):
    """Rows with at least 8 four-unit groups (29+ units) are decided by the
    rule; shorter rows give fewer than 8 finite lane maxima and take the
    exact rescan."""
    rng = np.random.default_rng(V * 10 + epl)
    groups = -(-(-(-(V // epl) // 32)) // 4)
    for _ in range(4):
        x = rng.normal(0, 1, V).astype(np.float32)
        x[rng.integers(0, V)] += 5                  # a planted successor
        assert _check(x, epl) == (None if groups >= 8 else "T0 = -inf")


@pytest.mark.parametrize("epl", [8, 4])
def test_selection_rule_with_ties_and_clusters(epl):
    rng = np.random.default_rng(3)
    V = 20000
    reasons = []
    for trial in range(40):
        kind = trial % 5
        if kind == 0:      # few distinct values: ties at T0 everywhere
            x = rng.integers(0, 4, V).astype(np.float32)
        elif kind == 1:    # the 12 largest values in one unit
            x = rng.normal(0, 1, V).astype(np.float32)
            u = int(rng.integers(0, V // (32 * epl)))
            x[u * 32 * epl + rng.choice(32 * epl, 12, replace=False)] = 10 + rng.random(12).astype(np.float32)
        elif kind == 2:    # ties exactly at the 8th value across units
            x = rng.normal(0, 1, V).astype(np.float32)
            x[rng.choice(V, 20, replace=False)] = 7.0
        elif kind == 3:    # mostly -inf with a few finite values, some in the tail
            x = np.full(V + 3, -np.inf, np.float32)
            x[rng.choice(V + 3, 30, replace=False)] = rng.normal(0, 1, 30)
            x[-2] = 50.0
        else:              # bf16-like coarse values (3 mantissa bits)
            x = np.round(rng.normal(0, 1, V) * 8).astype(np.float32) / 8
        reasons.append(_check(x, epl))
    assert any(r is None for r in reasons)          # the rule decided some; the others took the rescan


def test_fallbacks_are_taken_where_the_caps_bind():
    assert two_pass_top8(np.zeros(50000, np.float32), 8)[1] in ("units", "elements")  # all equal
    assert two_pass_top8(np.arange(7, dtype=np.float32), 8)[1] == "T0 = -inf"          # fewer than 8 lanes
    small = np.random.default_rng(1).normal(0, 1, 300).astype(np.float32)             # 2 units only
    assert two_pass_top8(small, 8)[1] == "T0 = -inf"


@pytest.mark.parametrize("epl", [8, 4])
def test_unit_records_decide_most_rows_without_a_reload(epl):
    """On the synthetic rows (normal noise plus a planted successor) most
    kept units hold a single element >= T0, so the records replace the
    reload; a unit holding two of the top elements is read again."""
    rng = np.random.default_rng(11 + epl)
    V = 151936
    single = multi = 0
    for _ in range(6):
        x = rng.normal(0, 1, V).astype(np.float32)
        x[rng.integers(0, V)] += 5
        x[3 * 32 * epl + 1] = x[3 * 32 * epl + 2] = 9.0           # two top elements in one unit
        assert _check(x, epl) is None
        nslot = V // epl
        upr = -(-nslot // 32)
        body = np.full(upr * 32 * epl, -np.inf)
        body[:nslot * epl] = x[:nslot * epl]
        srt = -np.sort(-body.reshape(upr, 32 * epl), axis=1)
        T0 = np.sort(x)[::-1][7]                                   # the 8th largest element (>= the rule's T0)
        kept = srt[:, 0] >= T0
        single += int((kept & (srt[:, 1] < T0)).sum())
        multi += int((kept & (srt[:, 1] >= T0)).sum())
    assert multi >= 6 and single > 5 * multi
