"""The soft rank of "Merge Hulls Without Copying Vertices: GPU Isotonic
Regression", Section 7.9, composed on the host from numpy's sort and the fp64
oracle (test infrastructure)."""
import numpy as np

import oracle


def ref_soft_rank(x, eps):
    """The paper's Section 7.9 on the host: theta = x / eps sorted in
    decreasing order into s, the oracle's non-increasing fit of s - (n..1),
    s minus the fit, back in the original order."""
    x = x.astype(np.float64)
    rows, n = x.shape
    out = np.empty_like(x)
    blocks = np.empty(x.shape, np.uint8)
    perms = np.empty(x.shape, np.int64)
    for r in range(rows):
        theta = (x[r] / eps).astype(np.float32)     # the CUDA path divides in float32
        perm = np.argsort(-theta, kind="stable")
        s = theta[perm].astype(np.float32)
        z = (s - np.arange(n, 0, -1, dtype=np.float32)).astype(np.float32)
        fit, b, st = oracle.pava(z[None, :], None, False)
        rr = s.astype(np.float64) - fit[0]
        out[r, perm] = rr
        blocks[r] = b[0]
        perms[r] = perm
    return out, blocks, perms
