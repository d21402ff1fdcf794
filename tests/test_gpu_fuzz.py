"""Randomised parity: seeded random shapes (1 .. 300,000 elements per row, one to
hundreds of rows), data families, weightings, directions and I/O types, through
iso_fit, the ragged entry point and the backward, each against the oracle."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import check_row, f64_params

pytestmark = pytest.mark.gpu

CASES = 60


def draw(rng):
    n = int(np.exp(rng.uniform(0, np.log(300_000))))
    rows = max(1, min(int(rng.integers(1, 300)), 400_000 // max(n, 1)))
    fam = wl.FAMILIES[int(rng.integers(len(wl.FAMILIES)))]
    weighting = wl.WEIGHTINGS[int(rng.integers(len(wl.WEIGHTINGS)))]
    return n, rows, fam, weighting, bool(rng.integers(2)), bool(rng.integers(4) == 0)


@pytest.mark.parametrize("case", range(CASES))
def test_fit_and_backward(cuda_ok, case):
    import torch
    import convex_hull_pava_gb300 as chp
    rng = np.random.default_rng(10_000 + case)
    n, rows, fam, weighting, inc, f64 = draw(rng)
    seed = int(rng.integers(1 << 30))
    y = wl.family(fam, rows, n, seed)
    w = wl.weights(weighting, rows, n, seed)
    if f64:
        y = y.astype(np.float64) * (1 + 1e-10 * rng.standard_normal(y.shape))
        w = None if w is None else w.astype(np.float64)
    label = f"case {case}: {rows}x{n} {fam}/{weighting} inc={inc} f64={f64}"
    yt = torch.from_numpy(y).cuda()
    wt = None if w is None else torch.from_numpy(w).cuda()
    out, blocks, st = chp.iso_fit(yt, wt, inc)
    g = rng.standard_normal(y.shape).astype(y.dtype)
    dy = chp.iso_backward(torch.from_numpy(g).cuda(), blocks, wt)
    out, blocks, st, dy = out.cpu().numpy(), blocks.cpu().numpy(), st.cpu().numpy(), dy.cpu().numpy()
    z, zb, zst = (oracle.pava_f64 if f64 else oracle.pava)(y, w, inc)
    assert np.array_equal(st.astype(np.uint32), zst), label
    for r in range(rows):
        if f64:
            tol, gr, gf = f64_params(None if w is None else w[r])
            check_row(y[r], out[r], blocks[r], z[r], zb[r], f"{label} row {r}", fit_tol=tol,
                      gap_rel=gr, gap_floor=gf)
        else:
            check_row(y[r], out[r], blocks[r], z[r], zb[r], f"{label} row {r}")
    # the backward over the GPU's own blocks
    ref = (oracle.backward_f64 if f64 else oracle.backward)(g, blocks, w)
    scale = np.abs(g).max() * (1.0 if w is None else float(np.max(w) / np.min(w)))
    assert np.abs(dy - ref).max() <= (1e-12 if f64 else 1e-5) * scale, label


@pytest.mark.parametrize("case", range(20))
def test_ragged(cuda_ok, case):
    import torch
    import convex_hull_pava_gb300 as chp
    rng = np.random.default_rng(20_000 + case)
    segs = int(rng.integers(1, 2000))
    max_len = int(np.exp(rng.uniform(0, np.log(60_000))))
    long_n = int(rng.integers(0, 4))
    lens = wl.ragged_lengths(segs, max_len, seed=case, long_segments=long_n,
                             long_len=int(rng.integers(8193, 40_000)))
    lens[rng.random(segs) < 0.05] = 0                      # some empty segments
    y, w, off = wl.ragged_calibration(lens, seed=case)
    if y.size == 0:
        return
    w = w if rng.integers(2) else None
    inc = bool(rng.integers(2))
    out, blocks, st = chp.iso_fit_ragged(torch.from_numpy(y).cuda(), torch.from_numpy(off).cuda(),
                                         None if w is None else torch.from_numpy(w).cuda(), inc)
    out, blocks, st = out.cpu().numpy(), blocks.cpu().numpy(), st.cpu().numpy().astype(np.uint32)
    z, zb, zst = oracle.pava_ragged(y, off, w, inc)
    assert np.array_equal(st, zst)
    for s in range(segs):
        a, b = int(off[s]), int(off[s + 1])
        if b > a:
            check_row(y[a:b], out[a:b], blocks[a:b], z[a:b], zb[a:b], f"case {case} segment {s}")
