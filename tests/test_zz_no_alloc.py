"""iso_backward_noalloc against iso_backward (collected last on purpose).

The entry point serves callers that cannot allocate device memory; it keeps
the long-row scratch in a fixed array inside the library.  Two calls in a row
must each agree with the workspace-taking entry point (the array keeps the
previous call's contents, which must not leak into the next result)."""
import ctypes

import numpy as np
import pytest

from convex_hull_pava_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 1e-5   # the backward parity tolerance, relative to 1 + max |reference|


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
        for call in range(2):
            g = torch.from_numpy(wl.normal(y.shape, seed + call)).cuda()
            ref = chp.iso_backward(g, blocks, wt)
            got = chp.iso_backward_noalloc(g, blocks, wt)
            torch.cuda.synchronize()
            assert _close(got.cpu().numpy(), ref.cpu().numpy()), (y.shape, call)


def test_noalloc_rejects_calls_beyond_its_scratch(cuda_ok):
    import convex_hull_pava_gb300 as chp
    lib = chp.load_library()
    fake = ctypes.c_void_p(0x1000)
    # 21,846 tiles of 8,192 elements: one tile more than the fixed scratch holds
    st = lib.iso_backward_noalloc(fake, fake, None, 21_846, 8193, fake, None)
    assert st == chp.ISO_ERR_WORKSPACE
