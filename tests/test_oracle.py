"""Pins of the fp64 oracle against facts fixed by the pages and by the mathematics,
not against itself (CPU only).

Citations are to "Merge Hulls Without Copying Vertices: GPU Isotonic Regression"
(the paper), the "groupant" page on the Rust PAVA (mod.rs) and the blog post
"Isotonic Regression on GPU".
"""
from fractions import Fraction
import itertools

import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from golden_io import load as load_golden


# ---------------------------------------------------------------------------
# independent exact helpers (rational arithmetic, tiny n)
# ---------------------------------------------------------------------------
def _frac(a):
    return [Fraction(float(v)) for v in a]


def brute_force(y, w):
    """Minimum of eq. (1) over every contiguous partition whose block means are
    non-decreasing, in exact rational arithmetic ("groupant" page, kkt_prefix:
    enumerated contiguous partitions independently select the minimum squared
    loss).  Returns (objective, fit, starts)."""
    n = len(y)
    yf, wf = _frac(y), _frac(w)
    best = None
    for cuts in itertools.product((0, 1), repeat=n - 1):
        starts = [0] + [i + 1 for i, c in enumerate(cuts) if c]
        ends = starts[1:] + [n]
        means = []
        for a, b in zip(starts, ends):
            sw = sum(wf[a:b])
            means.append(sum(wf[i] * yf[i] for i in range(a, b)) / sw)
        if any(means[k + 1] < means[k] for k in range(len(means) - 1)):
            continue
        z = []
        for m, a, b in zip(means, starts, ends):
            z += [m] * (b - a)
        obj = sum(wf[i] * (z[i] - yf[i]) ** 2 for i in range(n))
        if best is None or obj < best[0]:
            best = (obj, z, starts)
    return best


def minmax_formula(y, w):
    """z_i = max_{s<=i} min_{t>=i} Av_w(s..t): the textbook min-max formula of
    isotonic regression (not printed on the pages), O(n^3) in floats."""
    y = np.asarray(y, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    n = y.size
    cw = np.concatenate([[0.0], np.cumsum(w)])
    cs = np.concatenate([[0.0], np.cumsum(w * y)])
    z = np.empty(n)
    for i in range(n):
        best = -np.inf
        for s in range(i + 1):
            t = np.arange(i, n)
            av = (cs[t + 1] - cs[s]) / (cw[t + 1] - cw[s])
            best = max(best, av.min())
        z[i] = best
    return z


def kkt_residuals(y, w, z):
    """Prefix residuals r_k = sum_{j<=k} w_j (y_j - z_j) in fp64 (paper Section 7.6;
    groupant page, Invariant)."""
    w = np.ones_like(y, dtype=np.float64) if w is None else np.asarray(w, np.float64)
    return np.cumsum(w * (np.asarray(y, np.float64) - z))


# ---------------------------------------------------------------------------
# worked examples printed on the pages (tests/golden/worked_examples.txt)
# ---------------------------------------------------------------------------
GOLDEN = load_golden()


@pytest.mark.parametrize("case", [c for c in GOLDEN if "z" in c], ids=lambda c: c["name"])
@pytest.mark.parametrize("route", ["pava", "hull"])
def test_golden_fit(case, route):
    y = np.array([float(v) for v in case["y"]], dtype=np.float32)
    w = None if "w" not in case else np.array([float(v) for v in case["w"]], np.float32)
    fn = oracle.pava if route == "pava" else oracle.hull_fit
    z, starts, st = fn(y, w, bool(case.get("inc", 1)))
    assert st == 0
    np.testing.assert_allclose(z, [float(v) for v in case["z"]], rtol=0, atol=1e-15)
    if "starts" in case:
        assert list(starts) == [int(v) for v in case["starts"]]


def test_golden_running_totals():
    case = [c for c in GOLDEN if c["name"] == "running_totals"][0]
    W, S = oracle.points(np.array([float(v) for v in case["y"]], np.float32))
    assert list(W) == [float(v) for v in case["W"]]
    assert list(S) == [float(v) for v in case["S"]]


def test_golden_gradient():
    case = [c for c in GOLDEN if c["name"] == "grad_four"][0]
    y = np.array([float(v) for v in case["y"]], np.float32)
    _, starts, _ = oracle.pava(y)
    dy = oracle.backward(np.array([float(v) for v in case["g"]], np.float32), starts)
    np.testing.assert_allclose(dy, [float(v) for v in case["dy"]], atol=1e-15)


# ---------------------------------------------------------------------------
# brute force over contiguous partitions, n <= 10
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(12))
def test_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 11))
    if seed % 3 == 0:
        y = rng.integers(-3, 4, size=n).astype(np.float32)      # many ties
    else:
        y = rng.standard_normal(n).astype(np.float32)
    w = None if seed % 2 == 0 else rng.uniform(0.1, 3.0, n).astype(np.float32)
    obj, zb, _ = brute_force(y, np.ones(n, np.float32) if w is None else w)
    for fn in (oracle.pava, oracle.hull_fit):
        z, starts, st = fn(y, w)
        assert st == 0
        np.testing.assert_allclose(z, [float(v) for v in zb], rtol=0, atol=1e-12)
    # the oracle's objective equals the brute-force minimum
    z, _, _ = oracle.pava(y, w)
    ww = np.ones(n) if w is None else w.astype(np.float64)
    assert abs(float(np.sum(ww * (z - y) ** 2)) - float(obj)) <= 1e-10 * (1 + float(obj))


def test_brute_force_catches_wrong_fits():
    """The brute-force pin itself rejects plausible mistakes: a fit that pools on
    a strict rise, or a plain (unweighted) mean used with weights."""
    y = np.array([1, 3, 2, 4], np.float32)
    w = np.array([1, 2, 1, 1], np.float32)
    obj, zb, _ = brute_force(y, w)
    assert [float(v) for v in zb] == [1.0, 8 / 3, 8 / 3, 4.0]   # weighted mean of (3,2) with w (2,1)
    assert float(obj) > 0


# ---------------------------------------------------------------------------
# min-max formula (textbook identity), n <= 40
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(6))
def test_minmax_formula(seed):
    rng = np.random.default_rng(100 + seed)
    n = 40
    y = wl.family(wl.FAMILIES[seed % len(wl.FAMILIES)], 1, n, seed)[0]
    w = rng.uniform(0.2, 2.0, n).astype(np.float32)
    z, _, _ = oracle.pava(y, w)
    scale = 1.0 + np.abs(y).max()
    np.testing.assert_allclose(z, minmax_formula(y, w), rtol=0, atol=1e-12 * scale)


# ---------------------------------------------------------------------------
# KKT conditions (paper Section 7.6; groupant page Invariant / kkt_prefix)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fam", wl.FAMILIES)
@pytest.mark.parametrize("weighting", wl.WEIGHTINGS)
def test_kkt(fam, weighting):
    n = 3000
    y = wl.family(fam, 1, n, 3)[0]
    w = wl.weights(weighting, 1, n, 3)
    w = None if w is None else w[0]
    z, starts, st = oracle.pava(y, w)
    assert st == 0
    ww = np.ones(n) if w is None else w.astype(np.float64)
    tau = 1e-12 * float(np.sum(ww * np.abs(y.astype(np.float64)))) + 1e-300
    r = kkt_residuals(y, w, z)
    assert r.min() >= -tau                      # every prefix residual >= 0
    assert abs(r[-1]) <= tau                    # total residual zero
    rises = np.nonzero(z[1:] > z[:-1])[0]       # strict rise between k and k+1
    assert np.all(np.abs(r[rises]) <= tau)      # prefix residual zero at every strict rise
    assert np.all(np.diff(z) >= 0)              # feasible
    # blocks partition the row and the fit is constant on each block (block conservation)
    assert starts[0] == 1
    b = np.cumsum(starts) - 1
    for k in range(b[-1] + 1):
        sel = b == k
        zz = z[sel]
        assert np.all(zz == zz[0])
        mean = np.sum(ww[sel] * y[sel]) / np.sum(ww[sel])
        mag = np.sum(ww[sel] * np.abs(y[sel])) / np.sum(ww[sel])   # cancellation scale
        assert abs(mean - zz[0]) <= 1e-12 * (1 + mag)


# ---------------------------------------------------------------------------
# idempotence, invariances, closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_idempotent_on_monotone(seed):
    """Already non-decreasing vectors, ties included, are fixed points (groupant
    page, ties_and_idempotence)."""
    rng = np.random.default_rng(seed)
    y = np.sort(rng.integers(0, 20, 500)).astype(np.float32)
    z, _, _ = oracle.pava(y)
    assert np.array_equal(z, y.astype(np.float64))
    z2, _, _ = oracle.pava(z.astype(np.float32))
    assert np.array_equal(z2, z)


def test_shift_and_weight_scale():
    rng = np.random.default_rng(5)
    y = rng.integers(-50, 50, 400).astype(np.float32) / 8        # exact in fp32 under +3
    w = rng.uniform(0.5, 2, 400).astype(np.float32)
    z, _, _ = oracle.pava(y, w)
    zs, _, _ = oracle.pava(y + np.float32(3.0), w)
    np.testing.assert_allclose(zs, z + 3.0, atol=1e-12)
    zw, _, _ = oracle.pava(y, w * np.float32(4.0))                # power of two: exact
    np.testing.assert_allclose(zw, z, atol=1e-13)


def test_decreasing_is_increasing_of_negated():
    """The decreasing problem is the increasing one for -y (paper Section 2.1)."""
    y = wl.family("gaussian", 1, 777, 9)[0]
    w = wl.weights("uniform", 1, 777, 9)[0]
    zd, bd, _ = oracle.pava(y, w, increasing=False)
    zi, bi, _ = oracle.pava(-y, w, increasing=True)
    np.testing.assert_array_equal(zd, -zi)
    np.testing.assert_array_equal(bd, bi)
    assert np.all(np.diff(zd) <= 0)


def test_closed_forms():
    # constant row: one block, identity
    y = np.full(100, 2.5, np.float32)
    z, s, _ = oracle.pava(y)
    assert np.all(z == 2.5) and s.sum() == 1
    # strictly decreasing row with weights: one block equal to the weighted mean
    y = np.arange(50, 0, -1).astype(np.float32)
    w = np.linspace(0.5, 2.0, 50).astype(np.float32)
    z, s, _ = oracle.pava(y, w)
    mean = np.sum(w.astype(np.float64) * y) / np.sum(w.astype(np.float64))
    np.testing.assert_allclose(z, mean, atol=1e-12)
    assert s.sum() == 1
    # soft rank at eps = 1 pools every row into one block (paper Section 7.9)
    ys = wl.soft_rank_rows(8, 512, 1.0, 0)
    z, s, _ = oracle.pava(ys, None, increasing=False)
    assert np.all(s.sum(axis=1) == 1)
    np.testing.assert_allclose(z, np.broadcast_to(ys.astype(np.float64).mean(1, keepdims=True),
                                                  ys.shape), atol=1e-9)
    # n = 1: identity
    z, s, _ = oracle.pava(np.array([-7.25], np.float32))
    assert z[0] == -7.25 and s[0] == 1


def test_every_point_a_vertex_on_increasing_data():
    """Strictly increasing data: the fit is the data and every element starts a
    block (paper Section 7.1, "in strictly increasing data all points are vertices")."""
    y = np.cumsum(np.full(300, 0.25, np.float32)).astype(np.float32)
    z, s, _ = oracle.pava(y)
    assert np.array_equal(z, y.astype(np.float64)) and s.all()


# ---------------------------------------------------------------------------
# cross-checks: two routes of the oracle, and scipy / scikit-learn where installed
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fam", wl.FAMILIES)
def test_pava_matches_hull(fam):
    y = wl.family(fam, 3, 2500, 11)
    w = wl.weights("uniform", 3, 2500, 11)
    for inc in (True, False):
        zp, _, _ = oracle.pava(y, w, inc)
        zh, _, _ = oracle.hull_fit(y, w, inc)
        scale = 1.0 + np.abs(y).max()
        np.testing.assert_allclose(zp, zh, rtol=0, atol=1e-9 * scale)


def test_against_scipy():
    so = pytest.importorskip("scipy.optimize")
    if not hasattr(so, "isotonic_regression"):
        pytest.skip("scipy without isotonic_regression")
    y = wl.noisy_ramp(1, 20000, 4)[0]
    w = wl.weights("uniform", 1, 20000, 4)[0]
    ref = so.isotonic_regression(y.astype(np.float64), weights=w.astype(np.float64)).x
    z, _, _ = oracle.pava(y, w)
    np.testing.assert_allclose(z, ref, rtol=0, atol=1e-10)


def test_against_sklearn():
    iso = pytest.importorskip("sklearn.isotonic")
    y = wl.noisy_ramp(1, 5000, 6)[0]
    ref = iso.isotonic_regression(y.astype(np.float64), increasing=False)
    z, _, _ = oracle.pava(y, None, increasing=False)
    np.testing.assert_allclose(z, ref, rtol=0, atol=1e-10)


# ---------------------------------------------------------------------------
# gradients: finite differences in fp64 on data without near-ties (paper App. C)
# ---------------------------------------------------------------------------
def test_backward_finite_differences():
    rng = np.random.default_rng(21)
    n = 60
    y = (rng.integers(-64, 64, n) / 16).astype(np.float32)
    y = y + (np.arange(n) % 7) * np.float32(1 / 256)             # break exact ties
    w = rng.uniform(0.5, 2.0, n).astype(np.float32)
    g = rng.standard_normal(n).astype(np.float32)
    z0, starts, _ = oracle.pava(y, w)
    dy = oracle.backward(g, starts, w)
    dw = oracle.backward_w(g, starts, w, y, z0)
    h = np.float32(2.0 ** -12)
    for j in range(n):
        yp = y.copy(); yp[j] += h
        zp, sp, _ = oracle.pava(yp, w)
        fd = float(np.dot(g.astype(np.float64), (zp - z0))) / float(h)
        if np.array_equal(sp, starts):
            assert abs(fd - dy[j]) <= 1e-6 * (1 + abs(dy[j])), j
        wp = w.copy(); wp[j] += h
        zq, sq, _ = oracle.pava(y, wp)
        fdw = float(np.dot(g.astype(np.float64), (zq - z0))) / float(np.float32(wp[j]) - w[j])
        if np.array_equal(sq, starts):
            assert abs(fdw - dw[j]) <= 1e-3 * (1 + abs(dw[j])), j


def test_backward_row_mean_closed_form():
    """One block per row: the gradient is the row mean of g, broadcast."""
    ys = wl.soft_rank_rows(4, 256, 1.0, 2)
    _, s, _ = oracle.pava(ys, None, increasing=False)
    g = wl.normal((4, 256), 3)
    out = oracle.backward(g, s)
    np.testing.assert_allclose(out, np.broadcast_to(g.astype(np.float64).mean(1, keepdims=True),
                                                    g.shape), atol=1e-12)


# ---------------------------------------------------------------------------
# error convention
# ---------------------------------------------------------------------------
def test_bad_rows_flagged():
    y = wl.noisy_ramp(3, 50, 1)
    y[1, 7] = np.nan
    w = np.ones_like(y)
    w[2, 3] = 0.0
    z, _, st = oracle.pava(y, w)
    assert list(st) == [0, oracle.BAD_Y, oracle.BAD_W]
    assert np.isnan(z[1]).all() and np.isnan(z[2]).all() and np.isfinite(z[0]).all()


# ---- the soft rank composition (Section 7.9) on the oracle ----
def test_soft_rank_composition_finite_differences():
    """d/dx of the host soft rank is (g_s - A g_s) back through the sort, / eps
    (A: block averaging over the fit's blocks), by fp64 finite differences on a
    small row whose fit has no near-ties."""
    from soft_rank_ref import ref_soft_rank
    rng = np.random.default_rng(9)
    x = rng.standard_normal((1, 12)) * 3
    eps = 0.7
    g = rng.standard_normal(12)

    def f(v):
        r, _, _ = ref_soft_rank(v, eps)
        return float((r[0] * g).sum())
    _, blocks, perms = ref_soft_rank(x, eps)
    gs = g[perms[0]]
    gs = gs - oracle.backward(gs[None, :].astype(np.float32), blocks)[0]
    an = np.empty(12)
    an[perms[0]] = gs / eps
    h = 1e-3
    for i in range(12):
        d = np.zeros((1, 12))
        d[0, i] = h
        fd = (f(x + d) - f(x - d)) / (2 * h)
        assert abs(fd - an[i]) <= 2e-2 * (1 + abs(an[i]))


def test_soft_rank_composition_small_eps_is_hard_rank():
    from soft_rank_ref import ref_soft_rank
    x = np.random.default_rng(4).standard_normal((3, 50))
    r, _, _ = ref_soft_rank(x, 1e-6)
    hard = np.argsort(np.argsort(x, axis=1), axis=1) + 1
    assert np.abs(r - hard).max() <= 1e-3



# ---- ragged batches (segments of unequal lengths end to end) ----
def _quarter_rates(lengths, seed):
    """Calibration-style targets on a grid of 1/4 (exact in float32 after a
    lift by an even integer), with their weights and offsets."""
    y, w, off = wl.ragged_calibration(lengths, seed)
    return (np.floor(4.0 * y) / 4.0).astype(np.float32), w, off


@pytest.mark.parametrize("increasing", [True, False])
@pytest.mark.parametrize("weighted", [False, True])
def test_ragged_oracle_equals_lifted_single_row(increasing, weighted):
    """The paper's Section 7.7 fits per-segment curves as ONE row whose targets
    in segment s are lifted by 2 s (they lie in [0, 1]), so that no block can
    cross a segment boundary, and subtracts the lift from the fit.  With the
    targets on a grid of 1/4 the lift is exact in float32, and the single-row
    PAVA (minus the lift) must equal the per-segment fits."""
    lengths = np.array([1, 7, 33, 2, 100, 64, 5, 250, 1, 17], dtype=np.int64)
    y, w, off = _quarter_rates(lengths, 3)
    w = w if weighted else None
    seg = np.repeat(np.arange(lengths.size), lengths)
    lift = (2.0 * seg) if increasing else (-2.0 * seg)
    lifted = (y.astype(np.float64) + lift).astype(np.float32)
    assert np.array_equal(lifted.astype(np.float64) - lift, y.astype(np.float64))
    zl, bl, _ = oracle.pava(lifted, w, increasing)
    z, b, st = oracle.pava_ragged(y, off, w, increasing)
    assert not st.any()
    np.testing.assert_allclose(zl - lift, z, rtol=0, atol=1e-12)
    assert bl[off[:-1]].all()             # every segment start starts a lifted block
    assert np.array_equal(bl, b)


def test_ragged_oracle_equal_lengths_is_the_batch():
    y = wl.noisy_ramp(6, 50, 4)
    off = np.arange(0, 301, 50, dtype=np.int64)
    z, b, st = oracle.pava_ragged(y.ravel(), off)
    z2, b2, st2 = oracle.pava(y)
    assert np.array_equal(z, z2.ravel()) and np.array_equal(b, b2.ravel())
    assert np.array_equal(st, st2)


def test_ragged_oracle_shapes_and_bad_values():
    y = wl.noisy_ramp(1, 40, 5).ravel()
    y[22] = np.nan
    # segments: [0,5) ok, [5,5) empty, [5,3) out of order, [3,20) overlaps but is
    # well formed, [20,30) holds the NaN, [30,41) ends past the array, [38,40) ok
    off = np.array([0, 5, 5, 3, 20, 30, 41, 40], dtype=np.int64)
    # the 7th segment runs from 41 down to 40: out of order as well
    z, b, st = oracle.pava_ragged(y, off)
    assert list(st) == [0, 0, oracle.BAD_SHAPE, 0, oracle.BAD_Y, oracle.BAD_SHAPE,
                        oracle.BAD_SHAPE]
    assert np.isnan(z[20:30]).all() and b[20] == 1 and not b[21:30].any()
    z5, _, _ = oracle.pava(y[0:5])
    z17, _, _ = oracle.pava(y[3:20])
    assert np.array_equal(z[0:3], z5[0:3]) and np.array_equal(z[3:20], z17)
    zl, _, st3 = oracle.pava_ragged(y, np.array([0, 10, 40], dtype=np.int64), max_len=12)
    assert list(st3) == [0, oracle.BAD_SHAPE] and np.isnan(zl[10:]).all()


# ---- float64 inputs (double-double sums) ----
def _f64_row(rng, n, kind):
    if kind == "ties":
        return rng.integers(-3, 4, size=n).astype(np.float64)
    if kind == "near_ties":        # gaps far below float32 resolution
        return 1.0 + 1e-13 * rng.integers(-3, 4, size=n)
    if kind == "cancel":           # magnitudes 1e-8 .. 1e8: plain double sums lose the small terms
        return rng.standard_normal(n) * 10.0 ** rng.integers(-8, 9, size=n)
    return rng.standard_normal(n) + 1e-9 * rng.standard_normal(n)


def _plain_double_pava(y, w):
    """PAVA with plain double sums (what a float64 oracle without the
    double-double arithmetic would compute)."""
    bs, bw, b0 = [], [], []
    for i, (yi, wi) in enumerate(zip(y, w)):
        bs.append(wi * yi); bw.append(wi); b0.append(i)
        while len(bs) >= 2 and bs[-2] * bw[-1] >= bs[-1] * bw[-2]:
            s, ww = bs.pop(), bw.pop(); b0.pop()
            bs[-1] += s; bw[-1] += ww
    z = np.empty(len(y))
    for k, a in enumerate(b0):
        b = b0[k + 1] if k + 1 < len(b0) else len(y)
        z[a:b] = bs[k] / bw[k]
    return z


@pytest.mark.parametrize("seed", range(16))
def test_f64_brute_force(seed):
    """float64 inputs against the exact rational optimum over every contiguous
    partition: the fit is the optimum rounded to double (within 2 ulp)."""
    rng = np.random.default_rng(500 + seed)
    n = int(rng.integers(1, 10))
    kind = ("ties", "near_ties", "cancel", "normal")[seed % 4]
    y = _f64_row(rng, n, kind)
    w = np.ones(n) if seed % 2 == 0 else rng.uniform(0.1, 3.0, n) * (1 + 1e-9 * rng.standard_normal(n))
    obj, zb, _ = brute_force(y, w)
    z, _, st = oracle.pava_f64(y, None if seed % 2 == 0 else w)
    assert st == 0
    exact = np.array([float(v) for v in zb])
    assert np.all(np.abs(z - exact) <= 4.5e-16 * np.maximum(np.abs(exact), 1e-300)), (z, exact)


def test_f64_cancellation_needs_double_double():
    """A row on which plain double block sums give a wrong fit while the
    double-double oracle matches the rational optimum: the pin above would
    catch an oracle that dropped the error terms."""
    y = np.array([1e16, 1.0, -1e16, 3.0, 2.0])
    w = np.ones(5)
    exact = np.array([float(v) for v in brute_force(y, w)[1]])
    z, _, _ = oracle.pava_f64(y)
    assert np.array_equal(z, exact)
    assert not np.allclose(_plain_double_pava(y, w), exact, rtol=1e-12, atol=0)


@pytest.mark.parametrize("fam", ["noise", "random_walk", "sawtooth", "cliff", "offset", "gaussian"])
@pytest.mark.parametrize("weighting", wl.WEIGHTINGS)
def test_f64_kkt_and_float32_agreement(fam, weighting):
    """KKT conditions of the float64 fit (prefix residuals >= 0, zero at the end
    and at every strict rise), and agreement with the float32 oracle on
    float32-representable inputs (the same definition computed with plain
    double sums, exact there)."""
    n = 2000
    y32 = wl.family(fam, 1, n, seed=9)[0]
    w32 = wl.weights(weighting, 1, n, seed=9)
    w32 = None if w32 is None else w32[0]
    z, b, st = oracle.pava_f64(y32.astype(np.float64), None if w32 is None else w32.astype(np.float64))
    z32, b32, _ = oracle.pava(y32, w32)
    assert st == 0
    scale = 1.0 + np.abs(y32).max()
    np.testing.assert_allclose(z, z32, rtol=0, atol=1e-13 * scale)
    yd = y32.astype(np.float64) + 1e-10 * np.random.default_rng(3).standard_normal(n)
    wd = None if w32 is None else w32.astype(np.float64)
    z, b, _ = oracle.pava_f64(yd, wd)
    r = kkt_residuals(yd, wd, z)
    tot = np.sum((np.ones(n) if wd is None else wd) * np.abs(yd))
    assert r.min() >= -1e-13 * tot and abs(r[-1]) <= 1e-13 * tot
    rises = np.nonzero(z[1:] > z[:-1] + 1e-12 * scale)[0]
    assert np.all(np.abs(r[rises]) <= 1e-13 * tot)


def test_f64_against_scipy():
    sp = pytest.importorskip("scipy.optimize")
    rng = np.random.default_rng(8)
    y = rng.standard_normal(5000) + np.linspace(0, 2, 5000) + 1e-11 * rng.standard_normal(5000)
    w = rng.uniform(0.5, 2.0, 5000)
    ref = sp.isotonic_regression(y, weights=w).x
    z, _, _ = oracle.pava_f64(y, w)
    np.testing.assert_allclose(z, ref, rtol=0, atol=1e-13)


def test_f64_backward():
    """Block averaging of float64 gradients: exact rational block means on a
    small case, and the float32 oracle on float32-representable inputs."""
    rng = np.random.default_rng(12)
    g = rng.standard_normal(9) * 10.0 ** rng.integers(-6, 7, 9)
    w = rng.uniform(0.1, 2.0, 9)
    blocks = np.array([1, 0, 0, 1, 0, 1, 1, 0, 0], np.uint8)
    out = oracle.backward_f64(g, blocks, w)
    starts = [0, 3, 5, 6, 9]
    for a, b in zip(starts[:-1], starts[1:]):
        G = sum(Fraction(float(v)) for v in g[a:b])
        W = sum(Fraction(float(v)) for v in w[a:b])
        for i in range(a, b):
            assert abs(out[i] - float(Fraction(float(w[i])) * G / W)) <= 4.5e-16 * abs(out[i]) + 1e-300
    g32 = g.astype(np.float32)
    np.testing.assert_allclose(oracle.backward_f64(g32.astype(np.float64), blocks),
                               oracle.backward(g32, blocks), rtol=1e-14, atol=0)
    y = rng.standard_normal(9)
    z = oracle.pava_f64(y, w)[0]
    dw = oracle.backward_w_f64(g, blocks, w, y, z)
    np.testing.assert_allclose(dw, (y - z) * out / w, rtol=1e-14, atol=1e-300)


def test_f64_backward_w_exact_rationals():
    """The float64 weight gradient against its definition in exact rationals:
    d/dw_i = (y_i - z_i) * G_B / W_B with G_B, W_B the block sums of g and w
    (the paper's Section 6 "Gradient"), on magnitudes from 1e-6 to 1e6 where
    plain double block sums lose digits."""
    rng = np.random.default_rng(41)
    for trial in range(20):
        n = int(rng.integers(2, 40))
        g = rng.standard_normal(n) * 10.0 ** rng.integers(-6, 7, n)
        w = rng.uniform(0.05, 3.0, n) * 10.0 ** rng.integers(-3, 4, n)
        y = rng.standard_normal(n) * 10.0 ** rng.integers(-2, 3, n)
        z, blocks, st = oracle.pava_f64(y, w)
        assert st == 0
        dw = oracle.backward_w_f64(g, blocks, w, y, z)
        starts = list(np.nonzero(blocks)[0]) + [n]
        for a, b in zip(starts[:-1], starts[1:]):
            G = sum(Fraction(float(v)) for v in g[a:b])
            W = sum(Fraction(float(v)) for v in w[a:b])
            for i in range(a, b):
                exact = (Fraction(float(y[i])) - Fraction(float(z[i]))) * G / W
                # one rounding of y - z, of G / W and of the product
                assert abs(dw[i] - float(exact)) <= 8e-16 * abs(float(exact)) + 1e-300, (trial, i)


def test_f64_backward_w_finite_differences():
    """The float64 weight gradient is the derivative of <g, fit(y, w)> in w:
    central differences in float64 on data without near-ties, wherever the
    perturbation keeps the block partition (Section 6 "Gradient", App. C)."""
    rng = np.random.default_rng(42)
    n = 50
    y = np.cumsum(rng.uniform(-1.0, 1.0, n)) + 0.3 * rng.standard_normal(n)
    w = rng.uniform(0.5, 2.0, n)
    g = rng.standard_normal(n)
    z0, b0, _ = oracle.pava_f64(y, w)
    dw = oracle.backward_w_f64(g, b0, w, y, z0)
    checked = 0
    for j in range(n):
        h = 1e-6 * w[j]
        wp = w.copy(); wp[j] += h
        wm = w.copy(); wm[j] -= h
        zp, bp, _ = oracle.pava_f64(y, wp)
        zm, bm, _ = oracle.pava_f64(y, wm)
        if not (np.array_equal(bp, b0) and np.array_equal(bm, b0)):
            continue
        fd = float(np.dot(g, zp - zm)) / (wp[j] - wm[j])
        assert abs(fd - dw[j]) <= 1e-7 * (1.0 + abs(dw[j])), (j, fd, dw[j])
        checked += 1
    assert checked >= n // 2
