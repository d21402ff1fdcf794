"""The floor of the block-boundary criterion (a gap of 2^-44 * max|y|, below
which neither the oracle's fp64 sums nor the 2^-50 grid decide the order of
two block means) exempts no boundary on the five named workloads: there, every
oracle boundary whose adjacent means differ by more than 1e-6 relative is
required of the CUDA path, exactly as the literal criterion asks."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import GAP_FLOOR, GAP_REL


def boundary_counts(W):
    z, zb, st = oracle.pava(W.y, W.w, W.increasing)
    assert not np.any(st)
    z = np.atleast_2d(z)
    zb = np.atleast_2d(zb).astype(bool)
    y = np.atleast_2d(W.y)
    gap = np.abs(z[:, 1:] - z[:, :-1])
    scale = np.maximum(np.abs(z[:, 1:]), np.abs(z[:, :-1]))
    ymax = np.abs(y).max(axis=1, keepdims=True).astype(np.float64)
    literal = zb[:, 1:] & (gap > GAP_REL * scale)
    exempt = literal & ~(gap > GAP_FLOOR * ymax)
    return int(zb[:, 1:].sum()), int(literal.sum()), int(exempt.sum())


@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_gap_floor_exempts_nothing_on_named_workloads(name):
    W = wl.make(name)
    boundaries, required, exempt = boundary_counts(W)
    print(f"{name}: {boundaries} oracle boundaries, {required} required by the 1e-6 rule, "
          f"{exempt} exempted by the floor")
    assert exempt == 0
