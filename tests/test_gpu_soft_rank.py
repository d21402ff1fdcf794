"""The soft rank end to end (sort, non-increasing fit, gather; backward through
the block averaging) against the same composition on the fp64 oracle."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from soft_rank_ref import ref_soft_rank

pytestmark = pytest.mark.gpu


def soft_rank_cuda(x, eps, g=None):
    import torch
    from convex_hull_pava_gb300.soft_rank import soft_rank
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda().requires_grad_(g is not None)
    r = soft_rank(xt, eps)
    gx = None
    if g is not None:
        r.backward(torch.from_numpy(np.ascontiguousarray(g)).cuda())
        gx = xt.grad.cpu().numpy()
    return r.detach().cpu().numpy(), gx


@pytest.mark.parametrize("n", [5, 100, 3000, 8192, 20000])
@pytest.mark.parametrize("eps", [1.0, 0.1, "1/n"])
def test_soft_rank_values(cuda_ok, n, eps):
    e = 1.0 / n if eps == "1/n" else eps
    x = wl.normal((3, n), seed=n)
    r, _ = soft_rank_cuda(x, e)
    ref, _, _ = ref_soft_rank(x, e)
    scale = 1.0 + np.abs(ref).max()
    assert np.abs(r - ref).max() <= 1e-5 * scale


def test_small_eps_gives_hard_ranks(cuda_ok):
    """When every gap between the sorted values of theta = x / eps exceeds 1,
    every element is its own block and the soft ranks are the hard ones (up to
    float32 rounding of s minus the fit; s reaches 1e4 here)."""
    rng = np.random.default_rng(3)
    x = np.stack([rng.permutation(1000) for _ in range(4)]).astype(np.float32) * 0.01
    r, _ = soft_rank_cuda(x, 1e-3)
    hard = np.argsort(np.argsort(x, axis=1), axis=1) + 1
    assert np.abs(r - hard).max() <= 1e-2


def test_eps_one_pools_each_row(cuda_ok):
    """At eps = 1 on N(0,1) values each row is one block (Section 7.9): every
    soft rank is s_k minus the row's mean of z."""
    x = wl.normal((2, 8192), seed=5)
    r, _ = soft_rank_cuda(x, 1.0)
    ref, blocks, _ = ref_soft_rank(x, 1.0)
    assert (blocks.sum(axis=1) == 1).all()
    assert np.abs(r - ref).max() <= 1e-5 * (1 + np.abs(ref).max())


@pytest.mark.parametrize("n", [100, 8192, 20000])
@pytest.mark.parametrize("eps", [1.0, "1/n"])
def test_soft_rank_gradient(cuda_ok, n, eps):
    """d/dx = (g_s - A g_s) back through the sort, / eps, with A the block
    averaging of the oracle's fit."""
    e = 1.0 / n if eps == "1/n" else eps
    x = wl.normal((2, n), seed=n + 1)
    g = wl.normal((2, n), seed=n + 2)
    _, gx = soft_rank_cuda(x, e, g)
    _, blocks, perms = ref_soft_rank(x, e)
    ref = np.empty((2, n))
    for r in range(2):
        gs = g[r][perms[r]]
        gs = gs.astype(np.float64) - oracle.backward(gs[None, :], blocks[r][None, :])[0]
        ref[r, perms[r]] = gs / e
    assert np.abs(gx - ref).max() <= 1e-4 * (1 + np.abs(ref).max())
