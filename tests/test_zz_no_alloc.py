"""iso_backward_noalloc against iso_backward and the oracle (collected last on
purpose).

The entry point serves callers that cannot allocate device memory; it keeps
the long-row scratch in a fixed array inside the library.  Two calls in a row
must each agree with the workspace-taking entry point and with the oracle's
block averaging (the array keeps the previous call's contents, which must not
leak into the next result).  The size limit is tested on both sides with real
buffers of the full size, so that a regression of the check computes a result
instead of touching memory that is not there."""
import ctypes

import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 1e-5   # the backward parity tolerance, relative to 1 + max |reference|
SCRATCH = 2 << 20          # bytes of the fixed scratch array
TILE = 8192                # elements per tile record of the long-row backward


def _close(a, b):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    return np.abs(a - b).max() <= TOL * (1.0 + np.abs(b).max())


def test_noalloc_matches_backward_twice(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    cases = [
        (wl.noisy_ramp(2, 100_003, 31), None, 41),                         # long rows, unit weights
        (wl.family("sawtooth", 3, 50_000, 32), wl.weights("uniform", 3, 50_000, 32), 42),
        (wl.noisy_ramp(5, 3000, 33), None, 43),                            # whole rows: no scratch
    ]
    for y, w, seed in cases:
        yt = torch.from_numpy(y).cuda()
        wt = None if w is None else torch.from_numpy(w).cuda()
        _, blocks, _ = chp.iso_fit(yt, wt, True)
        bh = blocks.cpu().numpy()
        for call in range(2):
            gh = wl.normal(y.shape, seed + call)
            g = torch.from_numpy(gh).cuda()
            ref = chp.iso_backward(g, blocks, wt)
            got = chp.iso_backward_noalloc(g, blocks, wt)
            torch.cuda.synchronize()
            got = got.cpu().numpy()
            assert _close(got, ref.cpu().numpy()), (y.shape, call)
            assert _close(got, oracle.backward(gh, bh, w)), (y.shape, call, "oracle")


def _tiles(rows, n):
    return rows * ((n + TILE - 1) // TILE)


def test_noalloc_limit_both_sides(cuda_ok):
    import torch
    import convex_hull_pava_gb300 as chp
    lib = chp.load_library()
    # 21,845 tiles (85 rows of 257 tiles) fill the array exactly; 21,846
    # tiles (331 rows of 66 tiles) need more than it holds
    fit_rows, fit_n = 85, 257 * TILE
    over_rows, over_n = 331, 65 * TILE + 1
    assert _tiles(fit_rows, fit_n) == 21_845 and _tiles(over_rows, over_n) == 21_846
    assert chp.iso_backward_workspace_bytes(fit_rows, fit_n, False) == SCRATCH
    assert chp.iso_backward_workspace_bytes(over_rows, over_n, False) > SCRATCH

    # just over the limit: refused before any launch (real buffers of the full size)
    g = torch.zeros((over_rows, over_n), dtype=torch.float32, device="cuda")
    b = torch.zeros((over_rows, over_n), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(g)
    st = lib.iso_backward_noalloc(ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(b.data_ptr()), None,
                                  over_rows, over_n, ctypes.c_void_p(o.data_ptr()), None)
    torch.cuda.synchronize()
    assert st == chp.ISO_ERR_WORKSPACE
    del g, b, o

    # exactly at the limit: accepted, and equal to the oracle's block averaging
    rng = np.random.default_rng(44)
    gh = wl.normal((fit_rows, fit_n), 45)
    bh = (rng.random((fit_rows, fit_n)) < 1e-3).astype(np.uint8)
    bh[:, 0] = 1
    g = torch.from_numpy(gh).cuda()
    b = torch.from_numpy(bh).cuda()
    got = chp.iso_backward_noalloc(g, b, None)
    ref = chp.iso_backward(g, b, None)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert _close(got, ref.cpu().numpy())
    assert _close(got, oracle.backward(gh, bh, None))
