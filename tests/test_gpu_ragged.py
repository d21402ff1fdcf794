"""Parity of the ragged-batch fit (iso_fit_ragged, through the C ABI) with the
oracle's per-segment fits, on seeded calibration-style batches: every lane
class of the whole-row kernels, long segments through the long-row path,
empty and rejected segments, the max_len hint, and the backward of the whole
array as one row."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import check_row

pytestmark = pytest.mark.gpu


def run_ragged(y, off, w=None, increasing=True, max_len=0, fill=None):
    import torch
    import convex_hull_pava_gb300 as chp
    yt = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    ot = torch.from_numpy(np.ascontiguousarray(off, dtype=np.int64)).cuda()
    wt = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).cuda()
    out = blocks = None
    if fill is not None:
        out = torch.full_like(yt, fill)
        blocks = torch.full(yt.shape, 7, dtype=torch.uint8, device=yt.device)
    out, blocks, st = chp.iso_fit_ragged(yt, ot, wt, increasing, max_len=max_len, out=out,
                                         blocks=blocks)
    torch.cuda.synchronize()
    return out.cpu().numpy(), blocks.cpu().numpy(), st.cpu().numpy().astype(np.uint32)


def check_ragged(y, off, w=None, increasing=True, max_len=0, label="", segs=None):
    out, blocks, st = run_ragged(y, off, w, increasing, max_len)
    z, zb, zst = oracle.pava_ragged(y, off, w, increasing, max_len)
    assert np.array_equal(st, zst), f"{label}: status {np.nonzero(st != zst)[0][:5]}"
    for s in (range(len(off) - 1) if segs is None else segs):
        a, b = int(off[s]), int(off[s + 1])
        if zst[s] or b <= a:
            continue
        check_row(y[a:b], out[a:b], blocks[a:b], z[a:b], zb[a:b], f"{label} segment {s} [{a},{b})")
    return out, blocks, st


@pytest.mark.parametrize("increasing", [True, False])
@pytest.mark.parametrize("weighted", [False, True])
def test_every_lane_class(cuda_ok, increasing, weighted):
    lengths = wl.ragged_lengths(3000, 8192, seed=11)
    lengths[:10] = [1, 2, 31, 32, 33, 1024, 1025, 4096, 8191, 8192]
    y, w, off = wl.ragged_calibration(lengths, seed=12)
    check_ragged(y, off, w if weighted else None, increasing, label="classes")


@pytest.mark.parametrize("weighted", [False, True])
def test_long_segments_with_short_ones(cuda_ok, weighted):
    lengths = wl.ragged_lengths(400, 3000, seed=21, long_segments=6, long_len=40_000)
    lengths[:4] = [8193, 12_289, 4097 * 3 + 1, 100_000]
    y, w, off = wl.ragged_calibration(lengths, seed=22)
    check_ragged(y, off, w if weighted else None, True, label="long")


@pytest.mark.parametrize("fam", ["noise", "increasing", "sawtooth", "cancellation", "offset"])
def test_long_and_short_families(cuda_ok, fam):
    """Segments cut from rows of the accuracy families, at odd offsets."""
    lengths = np.array([9000, 1, 70_000, 33, 8192, 20_001, 500], dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(lengths)])
    y = wl.family(fam, 1, int(off[-1]), seed=5).ravel()
    check_ragged(y, off, None, True, label=fam)
    check_ragged(y, off, None, False, label=fam + " decreasing")


def test_equal_lengths_match_the_dense_batch_bitwise(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    for rows, n in [(64, 700), (3, 20_000)]:
        y = wl.noisy_ramp(rows, n, 6)
        off = np.arange(0, rows * n + 1, n, dtype=np.int64)
        out, blocks, st = run_ragged(y.ravel(), off)
        d_out, d_blocks, d_st = chp.iso_fit(torch.from_numpy(y).cuda())
        assert np.array_equal(out, d_out.cpu().numpy().ravel())
        assert np.array_equal(blocks, d_blocks.cpu().numpy().ravel())


def test_empty_rejected_and_uncovered(cuda_ok):
    y = wl.noisy_ramp(1, 60_000, 7).ravel()
    y[30_010] = np.inf                      # a long segment with a bad value
    y[100] = np.nan                         # a short one
    # [0,10) [10,10) [10,200) [200,30000) [30000,50000) [50000,59000) and
    # [59000,61000), which ends past the array: rejected, left unwritten
    off = np.array([0, 10, 10, 200, 30_000, 50_000, 59_000, 61_000], dtype=np.int64)
    out, blocks, st = run_ragged(y, off, fill=-5.0)
    z, zb, zst = oracle.pava_ragged(y, off)
    assert list(st) == [0, 0, oracle.BAD_Y, 0, oracle.BAD_Y, 0, oracle.BAD_SHAPE]
    assert list(zst) == list(st)
    for s in (0, 3, 5):
        a, b = off[s], off[s + 1]
        check_row(y[a:b], out[a:b], blocks[a:b], z[a:b], zb[a:b], f"segment {s}")
    for s in (2, 4):
        a, b = off[s], off[s + 1]
        assert np.isnan(out[a:b]).all() and blocks[a] == 1 and not blocks[a + 1:b].any()
    assert (out[59_000:] == -5.0).all() and (blocks[59_000:] == 7).all()


def test_max_len_hint(cuda_ok):
    lengths = wl.ragged_lengths(500, 2000, seed=31)
    lengths[7] = 10_000
    y, w, off = wl.ragged_calibration(lengths, seed=32)
    check_ragged(y, off, w, True, max_len=10_000, label="exact hint")
    check_ragged(y, off, w, True, max_len=2000, label="short hint")   # segment 7 rejected
    out, _, st = run_ragged(y, off, w, True, max_len=2000)
    assert st[7] == oracle.BAD_SHAPE and (st[np.arange(500) != 7] == 0).all()


def test_out_of_range_offsets_rejected(cuda_ok):
    y = wl.noisy_ramp(1, 1000, 8).ravel()
    off = np.array([0, 300, -5, 400, 2000], dtype=np.int64)
    out, blocks, st = run_ragged(y, off)
    assert list(st) == [0, oracle.BAD_SHAPE, oracle.BAD_SHAPE, oracle.BAD_SHAPE]


@pytest.mark.parametrize("weighted", [False, True])
def test_backward_of_the_whole_array(cuda_ok, weighted):
    """Every segment's first element starts a block, so the backward of the
    concatenation as one row is each segment's own backward."""
    import torch
    import convex_hull_pava_gb300 as chp
    lengths = wl.ragged_lengths(300, 3000, seed=41, long_segments=2, long_len=30_000)
    y, w, off = wl.ragged_calibration(lengths, seed=42)
    w = w if weighted else None
    g = wl.normal(y.shape, 43)
    out, blocks, st = run_ragged(y, off, w)
    z, zb, _ = oracle.pava_ragged(y, off, w)
    gt = torch.from_numpy(g).cuda()
    bt = torch.from_numpy(blocks).cuda()
    wt = None if w is None else torch.from_numpy(w).cuda()
    dy = chp.iso_backward(gt.view(1, -1), bt.view(1, -1), None if wt is None else wt.view(1, -1))
    ref = np.concatenate([oracle.backward(g[a:b], zb[a:b], None if w is None else w[a:b])
                          for a, b in zip(off[:-1], off[1:])])
    np.testing.assert_allclose(dy.cpu().numpy().ravel(), ref, rtol=2e-5, atol=2e-5 * np.abs(g).max())
    yt = torch.from_numpy(y).cuda().requires_grad_(True)
    ot = torch.from_numpy(off).cuda()
    wq = None if w is None else torch.from_numpy(w).cuda().requires_grad_(True)
    fit = chp.isotonic_ragged(yt, ot, wq)
    fit.backward(gt)
    np.testing.assert_allclose(yt.grad.cpu().numpy(), ref, rtol=2e-5, atol=2e-5 * np.abs(g).max())
    if w is not None:
        refw = np.concatenate([oracle.backward_w(g[a:b], zb[a:b], w[a:b], y[a:b], z[a:b])
                               for a, b in zip(off[:-1], off[1:])])
        got = wq.grad.cpu().numpy()
        tol = 1e-4 * (1 + np.abs(refw).max())
        assert np.abs(got - refw).max() <= tol


def test_calibration_batch_full_size(cuda_ok):
    """The benchmark's ragged batch (65,536 curves of 1 to 8,192 points and 8
    curves of about 2^20 points): status of every segment, and parity on every
    long segment and on 300 sampled short ones."""
    lengths = wl.ragged_lengths(65_536, 8192, seed=0, long_segments=8, long_len=1 << 20)
    y, w, off = wl.ragged_calibration(lengths, seed=0)
    out, blocks, st = run_ragged(y, off, w, True)
    assert not st.any()
    rng = np.random.default_rng(1)
    segs = list(np.nonzero(lengths > 8192)[0]) + list(rng.choice(lengths.size, 300, replace=False))
    for s in segs:
        a, b = int(off[s]), int(off[s + 1])
        z, zb, zs = oracle.pava(y[a:b], w[a:b], True)
        assert zs == 0
        zb = zb.copy()
        check_row(y[a:b], out[a:b], blocks[a:b], z, zb, f"segment {s} (n={b - a})")
