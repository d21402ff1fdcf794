"""Depth of the long-row bridge searches (the paper's Section 5.2, Theorem 5.2).

A segment-list merge moves the bridge's ends alternately to each other's
tangent points for ISO_BRIDGE_MAX_PASSES passes at most, then finishes by
nested bisection; a flat merge narrows 32 candidates per round for
ISO_BRIDGE_MAX_ROUNDS rounds at most.  The library's debugging counters
(iso_bridge_stats_mode / iso_bridge_stats_read) show both bounds held on the
adversarial families (a cliff that pulls the top bridge across the whole row,
sawtooth teeth whose bridges span a tooth, dense increasing hulls), and mode 2
sends every segment-list search through the nested bisection, whose fits must
match the oracle as well."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture
def stats_mode(cuda_ok):
    import convex_hull_pava_gb300 as chp

    def set_mode(m):
        chp.bridge_stats_mode(m)

    yield set_mode
    chp.bridge_stats_mode(0)


def fit_and_stats(y, w, increasing=True, control=False):
    import torch
    import convex_hull_pava_gb300 as chp
    yt = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    wt = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).cuda()
    fn = chp.iso_fit_copy_control if control else chp.iso_fit
    out, blocks, st = fn(yt, wt, increasing)
    s = chp.bridge_stats_read()
    return out.cpu().numpy(), blocks.cpu().numpy(), st.cpu().numpy(), s


def check(y, w, out, blocks, st, increasing, label):
    z, zb, zst = oracle.pava(y, w, increasing)
    assert np.array_equal(np.atleast_1d(st).astype(np.uint32), np.atleast_1d(zst)), label
    check_rows(y, out, blocks, z, zb, label)


def check_bounds(s, label):
    import convex_hull_pava_gb300 as chp
    assert s["list_searches"] <= s["list_merges"], (label, s)
    assert s["nested"] <= s["list_searches"], (label, s)
    assert s["max_passes"] <= chp.BRIDGE_MAX_PASSES, (label, s)
    assert s["passes"] <= s["list_searches"] * chp.BRIDGE_MAX_PASSES, (label, s)
    assert s["max_rounds"] <= chp.BRIDGE_MAX_ROUNDS, (label, s)
    assert s["flat_unfinished"] == 0, (label, s)


FAMS = ["cliff", "sawtooth", "increasing", "random_walk", "noise"]


@pytest.mark.parametrize("fam", FAMS)
@pytest.mark.parametrize("weighting", ["none", "extreme"])
@pytest.mark.parametrize("n", [300_007, 2_000_000])
def test_bridge_depth_bounded(stats_mode, fam, weighting, n):
    y = wl.family(fam, 1, n, seed=n % 97)
    w = wl.weights(weighting, 1, n, seed=n % 89)
    stats_mode(1)
    out, blocks, st, s = fit_and_stats(y, w)
    label = f"{fam}/{weighting} n={n}"
    check(y, w, out, blocks, st, True, label)
    check_bounds(s, label)
    assert s["list_merges"] + s["flat_searches"] > 0, (label, s)


@pytest.mark.parametrize("fam", ["cliff", "sawtooth", "increasing", "random_walk"])
@pytest.mark.parametrize("weighting", ["none", "uniform"])
@pytest.mark.parametrize("increasing", [True, False])
def test_nested_bisection_everywhere(stats_mode, fam, weighting, increasing):
    """Every segment-list search takes the nested bisection from its first pass;
    the fit still matches the oracle, here and in the materialised-copy control."""
    n = 400_003
    y = wl.family(fam, 2, n, seed=7)
    w = wl.weights(weighting, 2, n, seed=7)
    label = f"forced {fam}/{weighting} inc={increasing}"
    for control in (False, True):
        stats_mode(2)
        out, blocks, st, s = fit_and_stats(y, w, increasing, control)
        check(y, w, out, blocks, st, increasing, f"{label} control={control}")
        check_bounds(s, label)
        assert s["max_passes"] == 0, (label, s)
        assert s["nested"] == s["list_searches"], (label, s)
        if fam in ("increasing", "cliff") and increasing:
            # dense hulls overflow the flat arrays: segment lists do the merging
            assert s["list_merges"] > 0, (label, control, s)
        if fam == "cliff" and increasing:
            # (strictly increasing hulls only append; the cliff's bridge searches)
            assert s["list_searches"] > 0, (label, control, s)


def test_counters_off_by_default(cuda_ok):
    """Mode 0 counts nothing: a fit after switching off leaves the counters as
    they were."""
    import convex_hull_pava_gb300 as chp
    y = wl.family("cliff", 1, 300_007, seed=1)
    chp.bridge_stats_mode(1)
    _, _, _, s1 = fit_and_stats(y, None)
    chp.bridge_stats_mode(0)
    _, _, _, s2 = fit_and_stats(y, None)
    assert s1 == s2
    assert s1["list_merges"] + s1["flat_searches"] > 0
