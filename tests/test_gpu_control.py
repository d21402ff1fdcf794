"""The materialised-copy control (iso_fit_copy_control, the paper's grid
copying of Section 7.3): the same chunk hulls, bridge search and schedule, with
every merged hull copied into flat arrays, so its fit and block starts must be
those of iso_fit bit for bit -- and both match the oracle."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import check_rows

pytestmark = pytest.mark.gpu


def both(y, w=None, increasing=True):
    import torch
    import convex_hull_pava_gb300 as chp
    yt = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    wt = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).cuda()
    a = chp.iso_fit(yt, wt, increasing)
    b = chp.iso_fit_copy_control(yt, wt, increasing)
    torch.cuda.synchronize()
    return a, b


def assert_same(a, b, label):
    import torch
    oa, ba, sa = a
    ob, bb, sb = b
    assert torch.equal(sa, sb), label
    assert torch.equal(ba, bb), f"{label}: block starts differ at {torch.nonzero(ba != bb)[:5].tolist()}"
    same = (oa == ob) | (torch.isnan(oa) & torch.isnan(ob))
    assert bool(same.all()), f"{label}: fit differs at {torch.nonzero(~same)[:5].tolist()}"


@pytest.mark.parametrize("n", [8193, 12_289, 100_003, 1_000_000])
def test_noise_rows(cuda_ok, n):
    y = wl.noisy_ramp(2, n, 3)
    a, b = both(y)
    assert_same(a, b, f"noise n={n}")
    z, zb, _ = oracle.pava(y)
    check_rows(y, b[0].cpu().numpy(), b[1].cpu().numpy(), z, zb, f"noise n={n}")


@pytest.mark.parametrize("fam", ["increasing", "cliff", "sawtooth", "random_walk", "cancellation",
                                 "collinear", "offset"])
@pytest.mark.parametrize("weighting", ["none", "extreme"])
def test_families(cuda_ok, fam, weighting):
    n = 70_001
    y = wl.family(fam, 3, n, seed=4)
    w = wl.weights(weighting, y.shape[0], y.shape[1], seed=5)
    for inc in (True, False):
        a, b = both(y, w, inc)
        assert_same(a, b, f"{fam}/{weighting}/{inc}")
    z, zb, _ = oracle.pava(y, w, False)
    check_rows(y, b[0].cpu().numpy(), b[1].cpu().numpy(), z, zb, f"{fam}/{weighting}")


def test_dense_weighted_batch(cuda_ok):
    y, w = wl.dense_increasing(8, 300_000, 6)
    a, b = both(y, w)
    assert_same(a, b, "dense weighted")


def test_bad_row_in_batch(cuda_ok):
    y = wl.noisy_ramp(3, 50_000, 7)
    y[1, 777] = np.nan
    a, b = both(y)
    assert_same(a, b, "bad row")
    assert int(b[2][1]) == oracle.BAD_Y and int(b[2][0]) == 0


def test_short_rows_take_the_row_kernels(cuda_ok):
    y = wl.noisy_ramp(64, 3000, 8)
    a, b = both(y)
    assert_same(a, b, "short rows")


@pytest.mark.parametrize("name", ["row1e7", "dense16x4m"])
def test_named_workloads_full_size(cuda_ok, name):
    W = wl.make(name)
    a, b = both(W.y, W.w, W.increasing)
    assert_same(a, b, name)
