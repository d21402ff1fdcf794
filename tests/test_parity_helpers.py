"""The parity checkers themselves, on the CPU: they accept the oracle's own
results and reject planted errors (a fit off by more than the tolerance, a
missing required boundary, a non-constant block)."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import check_batch, check_row


def _case():
    y = wl.noisy_ramp(300, 16, seed=5)
    z, zb, _ = oracle.pava(y)
    return y, z.astype(np.float32), zb.copy(), z, zb


def test_batch_checker_accepts_oracle_output():
    y, out, blocks, z, zb = _case()
    check_batch(y, out, blocks, z, zb, "oracle")
    for r in range(0, 300, 37):
        check_row(y[r], out[r], blocks[r], z[r], zb[r], "oracle")


def test_batch_checker_rejects_planted_errors():
    y, out, blocks, z, zb = _case()
    bad = out.copy()
    bad[123, 7] += 1e-3
    with pytest.raises(AssertionError, match="fit error"):
        check_batch(y, bad, blocks, z, zb)
    r, c = next((r, c) for r in range(200, 300) for c in range(1, 16) if zb[r, c]
                and abs(z[r, c] - z[r, c - 1]) > 1e-3)
    b2 = blocks.copy()
    b2[r, c] = 0
    with pytest.raises(AssertionError):
        check_batch(y, out, b2, z, zb)
    b3 = blocks.copy()
    b3[:, 0] = 0
    with pytest.raises(AssertionError, match="element 0"):
        check_batch(y, out, b3, z, zb)
