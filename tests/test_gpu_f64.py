"""float64 I/O (the ABI's _f64 entry points, the paper's float64 working type of
Section 6): parity of the fit, the block starts and both gradients with the
double-double oracle, on float64 inputs that float32 cannot hold, for whole
rows, long rows and ragged batches; and on float32-representable inputs the
same block starts as the float32 path."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import check_row, f64_params

pytestmark = pytest.mark.gpu


def f64_rows(fam, rows, n, seed):
    """A data family in float64 with detail below float32 resolution."""
    rng = np.random.default_rng(seed + 31)
    y = wl.family(fam, rows, n, seed).astype(np.float64)
    return y + 1e-9 * (1.0 + np.abs(y)) * rng.standard_normal(y.shape)


def f64_weights(kind, rows, n, seed):
    w = wl.weights(kind, rows, n, seed)
    if w is None:
        return None
    rng = np.random.default_rng(seed + 77)
    return w.astype(np.float64) * (1.0 + 1e-9 * rng.standard_normal(w.shape))


def run(y, w=None, increasing=True):
    import torch
    import convex_hull_pava_gb300 as chp
    yt = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    wt = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).cuda()
    out, blocks, st = chp.iso_fit(yt, wt, increasing)
    assert out.dtype == torch.float64
    torch.cuda.synchronize()
    return out.cpu().numpy(), blocks.cpu().numpy(), st.cpu().numpy().astype(np.uint32)


def parity(y, w=None, increasing=True, label=""):
    y2 = np.atleast_2d(y)
    w2 = None if w is None else np.atleast_2d(w)
    out, blocks, st = run(y2, w2, increasing)
    z, zb, zst = oracle.pava_f64(y2, w2, increasing)
    assert np.array_equal(st, zst), label
    for r in range(y2.shape[0]):
        tol, gr, gf = f64_params(None if w2 is None else w2[r])
        check_row(y2[r], out[r], blocks[r], z[r], zb[r], f"{label} row {r}", fit_tol=tol,
                  gap_rel=gr, gap_floor=gf)
    return out, blocks


@pytest.mark.parametrize("n", [1, 2, 31, 33, 100, 1000, 1025, 4097, 8192])
@pytest.mark.parametrize("weighted", [False, True])
def test_whole_rows(cuda_ok, n, weighted):
    rows = max(1, 4096 // n)
    y = f64_rows("noise", rows, n, n)
    w = f64_weights("uniform", rows, n, n) if weighted else None
    parity(y, w, True, f"n={n}")
    parity(y, w, False, f"n={n} decreasing")


@pytest.mark.parametrize("n", [8193, 20_000, 100_003, 1_000_000])
@pytest.mark.parametrize("weighted", [False, True])
def test_long_rows(cuda_ok, n, weighted):
    y = f64_rows("noise", 2, n, 3)
    w = f64_weights("uniform", 2, n, 3) if weighted else None
    parity(y, w, True, f"long n={n}")


@pytest.mark.parametrize("fam", wl.FAMILIES)
@pytest.mark.parametrize("weighting", wl.WEIGHTINGS)
def test_families(cuda_ok, fam, weighting):
    for n in (3000, 40_000):
        y = f64_rows(fam, 2, n, 5)
        w = f64_weights(weighting, 2, n, 5)
        parity(y, w, True, f"{fam}/{weighting}/{n}")


def test_values_beyond_float32_range(cuda_ok):
    """Magnitudes float32 cannot hold (rows at 1e-300 .. 1e300; subnormal
    values below a normal row maximum).  A tile whose largest magnitude is
    itself subnormal is rounded to multiples of 2^-1071, coarser than the
    subnormal spacing: not tested here."""
    rng = np.random.default_rng(4)
    for scale in (1e-300, 1e-30, 1e30, 1e300):
        y = scale * (np.linspace(0, 3, 5000) + rng.standard_normal((3, 5000)))
        parity(y, None, True, f"scale {scale}")
        parity(y[:, :4000], None, False, f"scale {scale} decreasing")
    y = 1e-300 * rng.standard_normal((2, 3000))
    y[:, ::7] = 5e-324 * rng.integers(-50, 50, (2, 429))
    parity(y, None, True, "subnormal values")


def test_float32_inputs_give_the_float32_blocks(cuda_ok):
    """On float32-representable inputs the fixed-point geometry is the same, so
    the block starts equal the float32 path's and the fits agree to float32."""
    import torch
    import convex_hull_pava_gb300 as chp
    for rows, n, weighted in [(64, 1000, False), (8, 8192, True), (2, 100_000, False), (2, 50_000, True)]:
        y32 = wl.noisy_ramp(rows, n, 8)
        w32 = wl.weights("uniform", rows, n, 8) if weighted else None
        a = chp.iso_fit(torch.from_numpy(y32).cuda(), None if w32 is None else torch.from_numpy(w32).cuda())
        b = chp.iso_fit(torch.from_numpy(y32.astype(np.float64)).cuda(),
                        None if w32 is None else torch.from_numpy(w32.astype(np.float64)).cuda())
        assert torch.equal(a[1], b[1])
        np.testing.assert_allclose(b[0].cpu().numpy(), a[0].cpu().numpy().astype(np.float64),
                                   rtol=2e-7, atol=2e-7)


def test_bad_rows(cuda_ok):
    y = f64_rows("noise", 3, 20_000, 6)
    y[0, 5] = np.nan
    y[2, 19_999] = np.inf
    w = f64_weights("uniform", 3, 20_000, 6)
    w[1, 7] = 0.0
    out, blocks, st = run(y, w)
    assert list(st) == [oracle.BAD_Y, oracle.BAD_W, oracle.BAD_Y]
    assert np.isnan(out).all() and not blocks.any()


@pytest.mark.parametrize("n", [777, 8192, 30_000])
@pytest.mark.parametrize("weighted", [False, True])
def test_backward(cuda_ok, n, weighted):
    import torch
    import convex_hull_pava_gb300 as chp
    y = f64_rows("noise", 3, n, 9)
    w = f64_weights("uniform", 3, n, 9) if weighted else None
    g = np.random.default_rng(10).standard_normal((3, n))
    out, blocks, _ = run(y, w)
    z, zb, _ = oracle.pava_f64(y, w)
    gt = torch.from_numpy(g).cuda()
    bt = torch.from_numpy(blocks).cuda()
    wt = None if w is None else torch.from_numpy(w).cuda()
    dy = chp.iso_backward(gt, bt, wt).cpu().numpy()
    ref = oracle.backward_f64(g, zb, w)
    np.testing.assert_allclose(dy, ref, rtol=0, atol=1e-12 * np.abs(g).max())
    if weighted:
        yt = torch.from_numpy(y).cuda()
        ot = torch.from_numpy(out).cuda()
        gy, gw = chp.iso_backward_w(gt, bt, wt, yt, ot)
        refw = np.stack([oracle.backward_w_f64(g[r], zb[r], w[r], y[r], z[r]) for r in range(3)])
        np.testing.assert_allclose(gw.cpu().numpy(), refw, rtol=0,
                                   atol=1e-11 * (1 + np.abs(refw).max()))
        np.testing.assert_allclose(gy.cpu().numpy(), ref, rtol=0, atol=1e-12 * np.abs(g).max())


def test_autograd(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    y = torch.from_numpy(f64_rows("noise", 4, 3000, 11)).cuda().requires_grad_(True)
    w = torch.from_numpy(f64_weights("uniform", 4, 3000, 11)).cuda().requires_grad_(True)
    z = chp.isotonic(y, w)
    assert z.dtype == torch.float64
    g = torch.randn(z.shape, dtype=torch.float64, device=z.device)
    z.backward(g)
    _, zb, _ = oracle.pava_f64(y.detach().cpu().numpy(), w.detach().cpu().numpy())
    ref = oracle.backward_f64(g.cpu().numpy(), zb, w.detach().cpu().numpy())
    np.testing.assert_allclose(y.grad.cpu().numpy(), ref, rtol=0, atol=1e-12 * float(g.abs().max()))
    assert w.grad is not None and torch.isfinite(w.grad).all()


@pytest.mark.parametrize("weighted", [False, True])
def test_ragged(cuda_ok, weighted):
    import torch
    import convex_hull_pava_gb300 as chp
    lengths = wl.ragged_lengths(400, 3000, seed=13, long_segments=3, long_len=30_000)
    y32, w32, off = wl.ragged_calibration(lengths, seed=14)
    rng = np.random.default_rng(15)
    y = y32.astype(np.float64) + 1e-9 * rng.standard_normal(y32.size)
    w = w32.astype(np.float64) * (1 + 1e-9 * rng.standard_normal(y32.size)) if weighted else None
    out, blocks, st = chp.iso_fit_ragged(torch.from_numpy(y).cuda(), torch.from_numpy(off).cuda(),
                                         None if w is None else torch.from_numpy(w).cuda())
    out, blocks, st = out.cpu().numpy(), blocks.cpu().numpy(), st.cpu().numpy().astype(np.uint32)
    z, zb, zst = oracle.pava_ragged(y, off, w, True, f64=True)
    assert np.array_equal(st, zst)
    for s in range(lengths.size):
        a, b = int(off[s]), int(off[s + 1])
        tol, gr, gf = f64_params(None if w is None else w[a:b])
        check_row(y[a:b], out[a:b], blocks[a:b], z[a:b], zb[a:b], f"segment {s}", fit_tol=tol,
                  gap_rel=gr, gap_floor=gf)
