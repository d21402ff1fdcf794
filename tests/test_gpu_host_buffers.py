"""Pinned host buffers passed straight to the calls (unified addressing: the
kernels read inputs and write outputs in place over the host link): the results
are those of device buffers, bit for bit."""
import numpy as np
import pytest

from convex_hull_pava_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,n,weighted", [(64, 1000, False), (3, 8192, True), (2, 100_003, False),
                                             (2, 50_000, True)])
def test_fit_and_backward(cuda_ok, rows, n, weighted):
    import torch
    import convex_hull_pava_gb300 as chp
    y = wl.noisy_ramp(rows, n, 3)
    w = wl.weights("uniform", rows, n, 3) if weighted else None
    g = wl.normal((rows, n), 4)
    yd = torch.from_numpy(y).cuda()
    wd = None if w is None else torch.from_numpy(w).cuda()
    od, bd, sd = chp.iso_fit(yd, wd, False)
    yh = torch.from_numpy(y).pin_memory()
    wh = None if w is None else torch.from_numpy(w).pin_memory()
    oh, bh, sh = chp.iso_fit(yh, wh, False)
    assert not oh.is_cuda and oh.is_pinned()
    torch.cuda.synchronize()
    assert torch.equal(od.cpu(), oh) and torch.equal(bd.cpu(), bh) and torch.equal(sd.cpu(), sh)
    dd = chp.iso_backward(torch.from_numpy(g).cuda(), bd, wd)
    dh = chp.iso_backward(torch.from_numpy(g).pin_memory(), bh, wh)
    torch.cuda.synchronize()
    assert torch.equal(dd.cpu(), dh)


def test_ragged(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    lens = wl.ragged_lengths(300, 3000, seed=5, long_segments=2, long_len=20_000)
    y, w, off = wl.ragged_calibration(lens, seed=5)
    od, bd, sd = chp.iso_fit_ragged(torch.from_numpy(y).cuda(), torch.from_numpy(off).cuda(),
                                    torch.from_numpy(w).cuda())
    oh, bh, sh = chp.iso_fit_ragged(torch.from_numpy(y).pin_memory(), torch.from_numpy(off).pin_memory(),
                                    torch.from_numpy(w).pin_memory())
    torch.cuda.synchronize()
    assert torch.equal(od.cpu(), oh) and torch.equal(bd.cpu(), bh) and torch.equal(sd.cpu(), sh)
