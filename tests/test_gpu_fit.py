"""Parity of the CUDA fit (through the C ABI) with the fp64 oracle on the same
seeded float32 inputs.  Shapes span the whole-row kernels (one lane to 256
lanes, several rows per CTA), the long-row path (several chunks and a ragged
tail), and the named workloads at full size."""
import numpy as np
import pytest

import oracle
from convex_hull_pava_gb300 import workloads as wl
from parity import check_rows

pytestmark = pytest.mark.gpu


def run_fit(y, w=None, increasing=True, want_blocks=True):
    import torch
    import convex_hull_pava_gb300 as chp
    yt = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    wt = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).cuda()
    out, blocks, st = chp.iso_fit(yt, wt, increasing, want_blocks=want_blocks)
    torch.cuda.synchronize()
    return (out.cpu().numpy(), None if blocks is None else blocks.cpu().numpy(),
            st.cpu().numpy())


def parity(y, w=None, increasing=True, label=""):
    out, blocks, st = run_fit(y, w, increasing)
    z, zb, zst = oracle.pava(y, w, increasing)
    assert np.array_equal(np.atleast_1d(st).astype(np.uint32), np.atleast_1d(zst)), label
    check_rows(y, out, blocks, z, zb, label)
    return out, blocks


# ---- whole rows: every lane count, ragged lanes, several rows per CTA ----
SHORT_N = [1, 2, 3, 5, 17, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129, 255, 256, 257, 511, 512,
           513, 1000, 1023, 1024, 1025, 2047, 2048, 2049, 4095, 4096, 4097, 6000, 8191, 8192]


@pytest.mark.parametrize("n", SHORT_N)
def test_short_rows_noise(cuda_ok, n):
    rows = 37
    y = wl.noisy_ramp(rows, n, seed=n)
    parity(y, None, True, f"noise n={n}")


@pytest.mark.parametrize("fam", wl.FAMILIES)
@pytest.mark.parametrize("weighting", wl.WEIGHTINGS)
@pytest.mark.parametrize("n", [40, 1000, 5000])
def test_short_rows_families(cuda_ok, fam, weighting, n):
    rows = 9
    y = wl.family(fam, rows, n, seed=n)
    w = wl.weights(weighting, rows, n, seed=n)
    for inc in (True, False):
        parity(y, w, inc, f"{fam}/{weighting} n={n} inc={inc}")


@pytest.mark.parametrize("n", [1, 7, 32, 333, 1024, 3000, 8192])
def test_short_rows_weighted_noise(cuda_ok, n):
    rows = 21
    y = wl.noisy_ramp(rows, n, seed=3)
    w = wl.weights("uniform", rows, n, seed=3)
    parity(y, w, True, f"weighted noise n={n}")


# ---- long rows: several chunks, ragged tails, bridges across chunks ----
LONG_N = [8193, 12000, 16384, 16385, 40000, 65536, 100003, 262144 + 77]


@pytest.mark.parametrize("n", LONG_N)
def test_long_rows_noise(cuda_ok, n):
    y = wl.noisy_ramp(2, n, seed=n % 1000)
    parity(y, None, True, f"long noise n={n}")


@pytest.mark.parametrize("fam", wl.FAMILIES)
@pytest.mark.parametrize("weighting", ["none", "uniform", "extreme"])
def test_long_rows_families(cuda_ok, fam, weighting):
    n = 50_000
    y = wl.family(fam, 2, n, seed=5)
    w = wl.weights(weighting, 2, n, seed=5)
    for inc in (True, False):
        parity(y, w, inc, f"long {fam}/{weighting} inc={inc}")


@pytest.mark.parametrize("n", [20_000, 300_000])
def test_long_rows_cliff_search(cuda_ok, n):
    """A cliff at the end pulls the top bridge across the whole row: the walks
    give up and bisection over the lists finds the tangents (paper Section
    5.2; test_gpu_bridge counts the searches)."""
    y = wl.family("cliff", 1, n, seed=1)
    parity(y, None, True, f"cliff n={n}")
    w = wl.weights("extreme", 1, n, seed=1)
    parity(y, w, True, f"cliff weighted n={n}")


def test_long_rows_sawtooth_many_rows(cuda_ok):
    y = wl.family("sawtooth", 5, 70_001, seed=9)
    parity(y, None, True, "sawtooth rows=5")


# ---- degenerate cases ----
def test_constant_and_monotone(cuda_ok):
    for n in (1, 50, 5000, 30000):
        y = np.full((3, n), 1.25, np.float32)
        out, blocks = parity(y, None, True, f"constant n={n}")
        assert np.all(out == 1.25)
        y = np.tile(np.arange(n, dtype=np.float32), (2, 1))
        out, _ = parity(y, None, True, f"increasing n={n}")
        assert np.array_equal(out, y)          # idempotent on monotone data


def test_single_element_blocks_are_exact(cuda_ok):
    """A block of one element is fitted by its own value: exactly on the
    whole-row path, to within one float32 rounding of the slope on long rows."""
    for n, exact in ((8000, True), (20000, False)):
        y = wl.family("increasing", 4, n, 3)
        w = wl.weights("extreme", 4, n, 3)
        out, blocks, _ = run_fit(y, w)
        b = blocks.astype(bool)
        single = b & np.concatenate([b[:, 1:], np.ones((4, 1), bool)], 1)
        assert single.mean() > 0.5
        if exact:
            assert np.array_equal(out[single], y[single])
        else:
            rel = np.abs(out[single].astype(np.float64) - y[single]) / np.abs(y[single])
            assert rel.max() <= 2.5e-7


def test_bad_rows(cuda_ok):
    for n in (100, 20000):
        y = wl.noisy_ramp(4, n, 2)
        w = np.ones_like(y)
        y[1, n // 2] = np.nan
        y[2, 3] = np.inf
        w[3, 0] = 0.0
        out, blocks, st = run_fit(y, w)
        assert list(st) == [0, 1, 1, 2]
        assert np.isnan(out[1:]).all() and (blocks[1:] == 0).all()
        z, zb, _ = oracle.pava(y[:1], w[:1])
        check_rows(y[:1], out[:1], blocks[:1], z, zb, f"bad rows n={n}")


def test_without_blocks_output(cuda_ok):
    y = wl.noisy_ramp(3, 20000, 4)
    out, blocks, _ = run_fit(y, None, True, want_blocks=False)
    assert blocks is None
    z, zb, _ = oracle.pava(y)
    check_rows(y, out, None, z, zb, "no blocks")


def test_stream_order_and_repeat(cuda_ok):
    """Two calls in a row on one workspace give identical results."""
    import torch
    import convex_hull_pava_gb300 as chp
    y = torch.from_numpy(wl.noisy_ramp(1, 100_000, 8)).cuda()
    nb = chp.iso_fit_workspace_bytes(1, 100_000, False)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    a, ba, _ = chp.iso_fit(y, workspace=ws)
    a = a.clone(); ba = ba.clone()
    b, bb, _ = chp.iso_fit(y, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(ba, bb)


# ---- the named workloads at full size ----
@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_named_workloads_full_size(cuda_ok, name):
    W = wl.make(name)
    parity(W.y, W.w, W.increasing, name)


# ---- chunks whose points are all locally convex but at lane boundaries: the
# all-vertex test must look across lanes (a shuffle inside a warp, shared
# memory across warps) ----
@pytest.mark.parametrize("drop_at", [32, 31 * 32, 32 * 32, 64 * 32, 127 * 32, "every_lane"])
@pytest.mark.parametrize("weighting", ["none", "uniform"])
def test_long_rows_increasing_with_lane_boundary_drops(cuda_ok, drop_at, weighting):
    C = 4096
    n = 3 * C + 77
    rng = np.random.default_rng(11)
    base = np.sort(rng.random((2, n)), axis=1) + 1e-6 * np.arange(n)[None, :]
    y = base.copy()
    for c0 in range(0, n, C):
        if drop_at == "every_lane":
            for l in range(32, min(C, n - c0), 32):
                y[:, c0 + l:] -= 0.25          # each lane starts below the last one's end
        elif c0 + drop_at < n:
            y[:, c0 + drop_at:] -= 0.5         # one drop at a lane (or warp) boundary
    y = np.ascontiguousarray(y, dtype=np.float32)
    w = wl.weights(weighting, 2, n, seed=12)
    for inc in (True, False):
        parity(y if inc else -y, w, inc, f"drops at {drop_at} {weighting} inc={inc}")
    # and the plain increasing rows (every chunk all vertices) beside them
    parity(np.ascontiguousarray(base, dtype=np.float32), w, True, f"all vertices {weighting}")
