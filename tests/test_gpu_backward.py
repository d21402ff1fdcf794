"""Parity of the CUDA backward (block averaging, through the C ABI) with the
fp64 oracle, over the block starts the CUDA forward wrote."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 1e-5


def run(y, w, g, increasing=True):
    import torch
    import convex_hull_pava_gb300 as chp
    yt = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    wt = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).cuda()
    gt = torch.from_numpy(np.ascontiguousarray(g)).cuda()
    out, blocks, _ = chp.iso_fit(yt, wt, increasing)
    dy = chp.iso_backward(gt, blocks, wt)
    torch.cuda.synchronize()
    return blocks.cpu().numpy(), dy.cpu().numpy()


def check(y, w, g, increasing=True, label=""):
    blocks, dy = run(y, w, g, increasing)
    ref = oracle.backward(g, blocks, w)
    scale = 1.0 + np.abs(ref).max(axis=-1, keepdims=True)
    err = np.abs(dy.astype(np.float64) - ref)
    assert (err <= TOL * scale).all(), f"{label}: max err {err.max():.3e}"
    # the backward is constant on each block for unit weights
    return blocks, dy


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 100, 1000, 1024, 1025, 4096, 8192])
@pytest.mark.parametrize("weighting", ["none", "uniform", "extreme"])
def test_rows(cuda_ok, n, weighting):
    rows = 13
    y = wl.noisy_ramp(rows, n, seed=n)
    w = wl.weights(weighting, rows, n, seed=n)
    g = wl.normal((rows, n), seed=n + 1)
    check(y, w, g, True, f"rows n={n} {weighting}")


@pytest.mark.parametrize("n", [8193, 20000, 65536, 100003])
@pytest.mark.parametrize("fam", ["noise", "increasing", "constant", "sawtooth", "random_walk"])
@pytest.mark.parametrize("weighting", ["none", "uniform"])
def test_long_rows(cuda_ok, n, fam, weighting):
    y = wl.family(fam, 2, n, seed=3)
    w = wl.weights(weighting, 2, n, seed=3)
    g = wl.normal((2, n), seed=4)
    check(y, w, g, True, f"long n={n} {fam} {weighting}")


def test_soft_rank_one_block(cuda_ok):
    """Soft rank at eps = 1: each row pools into one block, so the backward is
    the row mean of the upstream gradient (paper Section 7.9)."""
    W = wl.make("softrank1024x8192")
    blocks, dy = check(W.y, None, W.grad, False, "softrank")
    assert (blocks.sum(axis=1) == 1).all()
    mean = W.grad.astype(np.float64).mean(axis=1, keepdims=True)
    assert np.allclose(dy, mean, rtol=0, atol=1e-6)


def test_long_soft_rank_row(cuda_ok):
    y = wl.soft_rank_rows(1, 1_000_000, 1.0, 5)
    g = wl.normal((1, 1_000_000), 6)
    blocks, dy = check(y, None, g, False, "long softrank")
    assert blocks.sum() == 1


def test_autograd_op(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    y = torch.from_numpy(wl.noisy_ramp(3, 3000, 11)).cuda().requires_grad_(True)
    z = chp.isotonic(y)
    g = torch.randn_like(z)
    z.backward(g)
    _, blocks, _ = chp.iso_fit(y.detach())
    ref = oracle.backward(g.cpu().numpy(), blocks.cpu().numpy())
    assert np.allclose(y.grad.cpu().numpy(), ref, atol=1e-5)


def test_host_tensors_round_trip(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    y = torch.from_numpy(wl.noisy_ramp(2, 5000, 12))
    z = chp.isotonic(y)
    assert not z.is_cuda
    zo, _, _ = oracle.pava(y.numpy())
    assert np.abs(z.numpy() - zo).max() <= 1e-5 * (1 + np.abs(y.numpy()).max())


# ---- the weight gradient, d/dw_i = (y_i - z_i) G / W (paper Section 6, "Gradient") ----
def run_w(y, w, g, increasing=True):
    import torch
    import convex_hull_pava_gb300 as chp
    yt = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    wt = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).cuda()
    gt = torch.from_numpy(np.ascontiguousarray(g)).cuda()
    z, blocks, _ = chp.iso_fit(yt, wt, increasing)
    dy, dw = chp.iso_backward_w(gt, blocks, wt, yt, z)
    torch.cuda.synchronize()
    return blocks.cpu().numpy(), z.cpu().numpy(), dy.cpu().numpy(), dw.cpu().numpy()


def check_w(y, w, g, increasing=True, label=""):
    """Both gradients against the oracle, over the CUDA forward's blocks and fit
    (the weight gradient's formula takes the fit as given)."""
    blocks, z, dy, dw = run_w(y, w, g, increasing)
    ref_dy = oracle.backward(g, blocks, w)
    for r in range(y.shape[0]):
        wr = None if w is None else w[r]
        ref = oracle.backward_w(g[r], blocks[r], wr, y[r], z[r].astype(np.float64))
        err = np.abs(dw[r].astype(np.float64) - ref)
        assert err.max() <= TOL * (1.0 + np.abs(ref).max()), f"{label} row {r}: dw err {err.max():.3e}"
        e2 = np.abs(dy[r].astype(np.float64) - ref_dy[r])
        assert e2.max() <= TOL * (1.0 + np.abs(ref_dy[r]).max()), f"{label} row {r}: dy err {e2.max():.3e}"
    return blocks, z, dy, dw


@pytest.mark.parametrize("n", [1, 2, 33, 1000, 4096, 8192])
@pytest.mark.parametrize("weighting", ["none", "uniform", "extreme"])
def test_weight_gradient_rows(cuda_ok, n, weighting):
    rows = 7
    y = wl.noisy_ramp(rows, n, seed=n + 7)
    w = wl.weights(weighting, rows, n, seed=n + 7)
    g = wl.normal((rows, n), seed=n + 8)
    for inc in (True, False):
        check_w(y, w, g, inc, f"dw rows n={n} {weighting} inc={inc}")


@pytest.mark.parametrize("n", [8193, 100003])
@pytest.mark.parametrize("fam", ["noise", "increasing", "sawtooth"])
@pytest.mark.parametrize("weighting", ["none", "uniform", "extreme"])
def test_weight_gradient_long_rows(cuda_ok, n, fam, weighting):
    y = wl.family(fam, 2, n, seed=13)
    w = wl.weights(weighting, 2, n, seed=13)
    g = wl.normal((2, n), seed=14)
    for inc in (True, False):
        check_w(y, w, g, inc, f"dw long n={n} {fam} {weighting} inc={inc}")


def test_weight_gradient_sums_to_zero_on_each_block(cuda_ok):
    """sum_B (y_i - z_i) = 0 for unit weights (z is the block mean), so the unit
    weight gradient sums to zero over every block."""
    y = wl.noisy_ramp(3, 20000, 21)
    g = wl.normal((3, 20000), 22)
    blocks, z, dy, dw = check_w(y, None, g, True, "dw block sums")
    for r in range(3):
        ids = np.cumsum(blocks[r].astype(np.int64)) - 1
        sums = np.bincount(ids, weights=dw[r].astype(np.float64))
        assert np.abs(sums).max() <= 1e-3 * (1 + np.abs(dw[r]).max())


def test_weight_gradient_bad_row_is_nan(cuda_ok):
    y = wl.noisy_ramp(3, 5000, 23)
    y[1, 17] = np.nan
    w = wl.weights("uniform", 3, 5000, 23)
    g = wl.normal((3, 5000), 24)
    blocks, z, dy, dw = run_w(y, w, g)
    assert np.isnan(dw[1]).all()
    assert np.isfinite(dw[[0, 2]]).all()


def test_autograd_weight_gradient(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    y0 = wl.noisy_ramp(2, 9000, 25)
    w0 = wl.weights("uniform", 2, 9000, 25)
    y = torch.from_numpy(y0).cuda().requires_grad_(True)
    w = torch.from_numpy(w0).cuda().requires_grad_(True)
    z = chp.isotonic(y, w)
    g = torch.randn_like(z)
    z.backward(g)
    zt, blocks, _ = chp.iso_fit(y.detach(), w.detach())
    gn, bn, zn = g.cpu().numpy(), blocks.cpu().numpy(), zt.cpu().numpy().astype(np.float64)
    for r in range(2):
        ref = oracle.backward_w(gn[r], bn[r], w0[r], y0[r], zn[r])
        assert np.abs(w.grad[r].cpu().numpy() - ref).max() <= TOL * (1 + np.abs(ref).max())
    ref_dy = oracle.backward(gn, bn, w0)
    assert np.abs(y.grad.cpu().numpy() - ref_dy).max() <= TOL * (1 + np.abs(ref_dy).max())
