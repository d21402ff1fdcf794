"""The largest shapes the tests run: a 2^28-element row (1 GB of input; the
row-level sums exceed 64 bits), a weighted 2^27-element row, and 2^20 rows of
16 elements (the paper's 10^6 x 16 batch shape).  Parity with the oracle over
every element (the C oracle runs at about 10^8 elements per second)."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import check_batch, check_row

pytestmark = pytest.mark.gpu


def fit(y, w=None, increasing=True):
    import torch
    import convex_hull_pava_gb300 as chp
    yt = torch.from_numpy(y).cuda()
    wt = None if w is None else torch.from_numpy(w).cuda()
    out, blocks, st = chp.iso_fit(yt, wt, increasing)
    torch.cuda.synchronize()
    r = out.cpu().numpy(), blocks.cpu().numpy(), st.cpu().numpy()
    del yt, wt, out, blocks, st
    torch.cuda.empty_cache()
    return r


def test_row_of_2_pow_28(cuda_ok):
    n = 1 << 28
    y = wl.noisy_ramp(1, n, seed=21)[0]
    out, blocks, st = fit(y)
    assert int(st[0]) == 0
    z, zb, _ = oracle.pava(y)
    check_row(y, out, blocks, z, zb, "n=2^28")


def test_weighted_row_of_2_pow_27(cuda_ok):
    n = 1 << 27
    y = wl.noisy_ramp(1, n, seed=22)[0]
    w = wl.weights("uniform", 1, n, seed=22)[0]
    out, blocks, st = fit(y, w, False)
    assert int(st[0]) == 0
    z, zb, _ = oracle.pava(y, w, False)
    check_row(y, out, blocks, z, zb, "weighted n=2^27")


def test_2_pow_20_rows_of_16(cuda_ok):
    y = wl.noisy_ramp(1 << 20, 16, seed=23)
    out, blocks, st = fit(y, None, False)
    assert not st.any()
    z, zb, _ = oracle.pava(y, None, False)
    # every row: fit, block starts and ties (vectorised over the 2^20 rows)
    check_batch(y, out, blocks, z, zb, "16-element rows")
