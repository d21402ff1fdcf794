"""Differentiable soft ranks on top of the isotonic fit.

"Merge Hulls Without Copying Vertices: GPU Isotonic Regression", Section 7.9:
the L2-regularised soft rank of x with strength eps projects theta = x / eps
onto the permutahedron.  It sorts theta in decreasing order into s, fits the
non-increasing isotonic regression of z = s - (n, n-1, ..., 1), and returns s
minus that fit in the original order (1 for the smallest value when eps is
small).  The fit's Jacobian averages over the fit's blocks (A), so the soft
rank's vector-Jacobian product is (g - A g) taken back through the sort and
divided by eps.  The sort, gather and scatter are torch operations; the fit
and the block averaging run in this package's kernels.
"""
from __future__ import annotations

from . import iso_backward, iso_fit

_Fn = None


def _make():
    import torch

    class _SoftRank(torch.autograd.Function):
        @staticmethod
        def forward(ctx, x, eps):
            theta = x / eps
            s, perm = torch.sort(theta, dim=-1, descending=True)
            n = x.shape[-1]
            w = torch.arange(n, 0, -1, dtype=x.dtype, device=x.device)
            z = (s - w).contiguous()
            fit, blocks, _ = iso_fit(z, None, False)
            r = s - fit
            ranks = torch.empty_like(r).scatter_(-1, perm, r)
            ctx.save_for_backward(perm, blocks)
            ctx.eps = eps
            return ranks

        @staticmethod
        def backward(ctx, g):
            perm, blocks = ctx.saved_tensors
            gs = torch.gather(g, -1, perm).contiguous()
            gs = gs - iso_backward(gs, blocks, None)
            gx = torch.empty_like(gs).scatter_(-1, perm, gs)
            return gx / ctx.eps, None

    return _SoftRank


def soft_rank(x, eps: float = 1.0):
    """Soft ranks of every row of the float32 CUDA tensor x (2-D), with
    regularisation strength eps > 0; differentiable with respect to x."""
    global _Fn
    if not eps > 0:
        raise ValueError("eps must be > 0")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [rows, n]")
    if _Fn is None:
        _Fn = _make()
    return _Fn.apply(x.contiguous(), float(eps))
