"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws random numbers and lays them out; it holds none of the
isotonic-regression arithmetic.  Every generator is deterministic in its seed
(numpy ``default_rng``), draws in float64 and casts to float32 once, so the
same float32 bytes go to the GPU path and to the oracle.

The five named workloads follow the shapes and value distributions of the
isotonic-regression paper's data families ("Merge Hulls Without Copying
Vertices: GPU Isotonic Regression", Section 7.1: "noise" is a ramp from 0 to 3
plus standard normal noise, "increasing" data keeps every point as a vertex;
Section 7.9: the soft-rank problem z = s - w with w = (n, ..., 1)).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Workload:
    name: str
    rows: int
    n: int
    increasing: bool
    weighted: bool
    y: np.ndarray                      # float32 [rows, n]
    w: np.ndarray | None = None        # float32 [rows, n] or None (unit weights)
    grad: np.ndarray | None = None     # float32 [rows, n] upstream gradient, if the workload has one
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def elements(self) -> int:
        return self.rows * self.n


def noisy_ramp(rows: int, n: int, seed: int = 0) -> np.ndarray:
    """``linspace(0, 3, n) + N(0, 1)``: one draw of shape ``[rows, n]``."""
    rng = np.random.default_rng(seed)
    noise = rng.standard_normal((rows, n))
    return (np.linspace(0.0, 3.0, n)[None, :] + noise).astype(np.float32)


def dense_increasing(rows: int, n: int, seed: int = 0):
    """``sort(U(0,1)) + 1e-7*i`` per row (fp64, then fp32) and ``w ~ U(0.5, 2)``."""
    rng = np.random.default_rng(seed)
    y = np.empty((rows, n), dtype=np.float32)
    ramp = 1e-7 * np.arange(n, dtype=np.float64)
    for r in range(rows):
        u = np.sort(rng.random(n))
        y[r] = (u + ramp).astype(np.float32)
    w = rng.uniform(0.5, 2.0, size=(rows, n)).astype(np.float32)
    return y, w


def soft_rank_rows(rows: int, n: int, eps: float = 1.0, seed: int = 0) -> np.ndarray:
    """Isotonic input of an L2 soft rank: theta ~ N(0,1) per row sorted in
    decreasing order, ``y[k] = theta[k] / eps - (n - k)`` (0-based k), to be fit
    non-increasing."""
    rng = np.random.default_rng(seed)
    theta = -np.sort(-rng.standard_normal((rows, n)), axis=1) / eps
    return (theta - (n - np.arange(n, dtype=np.float64))[None, :]).astype(np.float32)


def ragged_lengths(segments: int, max_len: int, seed: int = 0, long_segments: int = 0,
                   long_len: int = 0) -> np.ndarray:
    """Segment lengths of a many-curve batch: log-uniform in [1, max_len] (many
    short curves, few long ones), then ``long_segments`` lengths of
    ``long_len`` +- 25% placed at seeded positions."""
    rng = np.random.default_rng(seed)
    lens = np.exp(rng.uniform(0.0, np.log(max_len + 1.0), segments)).astype(np.int64)
    lens = np.clip(lens, 1, max_len)
    if long_segments:
        pos = rng.choice(segments, size=min(long_segments, segments), replace=False)
        lens[pos] = (long_len * rng.uniform(0.75, 1.25, pos.size)).astype(np.int64)
    return lens


def ragged_calibration(lengths, seed: int = 0):
    """Per-segment calibration curves laid end to end (the paper's Section 7.7
    fits one curve per segment of scored events): in a segment of n points,
    scores u sorted from U(0, 1), each point a group of c = 1, 2 or 3 events
    (probabilities 0.7, 0.22, 0.08) with floor(c u^g + U(0, 1)) positives (c
    u^g on average), g ~ U(0.5, 2) per segment; the target is the group's
    positive rate, its weight the count c.  Returns
    ``(y, w, offsets)``: float32 [total] twice and int64 [segments + 1]."""
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    offsets = np.zeros(lengths.size + 1, dtype=np.int64)
    np.cumsum(lengths, out=offsets[1:])
    total = int(offsets[-1])
    seg = np.repeat(np.arange(lengths.size), lengths)
    g = rng.uniform(0.5, 2.0, lengths.size)[seg]
    # sorted U(0, 1) scores per segment, without a sort: the k-th of n sorted
    # uniforms is the k-th of n + 1 partial sums of Exp(1) draws over the last
    e = rng.exponential(size=total)
    cs = np.cumsum(e)
    base = np.concatenate([[0.0], cs])[offsets[:-1]]
    span = np.concatenate([[0.0], cs])[offsets[1:]] - base + rng.exponential(size=lengths.size)
    u = (cs - base[seg]) / span[seg]
    v = rng.random(total)
    c = 1 + (v < 0.3) + (v < 0.08)
    pos = np.floor(c * np.clip(u, 0.0, 1.0) ** g + rng.random(total))
    y = (pos / c).astype(np.float32)
    return y, c.astype(np.float32), offsets


def normal(shape, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


CONFIG_NAMES = ("row65k", "batch4096x1024", "row1e7", "dense16x4m", "softrank1024x8192")


def make(name: str) -> Workload:
    """The five named workloads.

    * ``row65k``: 1 x 65,536 noisy ramp, unit weights, non-decreasing fit.
    * ``batch4096x1024``: 4,096 x 1,024 noisy ramp (many short rows).
    * ``row1e7``: 1 x 10,000,000 noisy ramp (few hull vertices survive).
    * ``dense16x4m``: 16 x 4,194,304 strictly increasing data with weights in
      U(0.5, 2) (dense hull: nearly every point is a vertex).
    * ``softrank1024x8192``: 1,024 x 8,192 soft-rank rows at eps = 1, fit
      non-increasing, with an upstream gradient ~ N(0,1) (seed 1).
    """
    if name == "row65k":
        return Workload(name, 1, 65536, True, False, noisy_ramp(1, 65536, 0))
    if name == "batch4096x1024":
        return Workload(name, 4096, 1024, True, False, noisy_ramp(4096, 1024, 0))
    if name == "row1e7":
        return Workload(name, 1, 10_000_000, True, False, noisy_ramp(1, 10_000_000, 0))
    if name == "dense16x4m":
        y, w = dense_increasing(16, 4_194_304, 0)
        return Workload(name, 16, 4_194_304, True, True, y, w)
    if name == "softrank1024x8192":
        y = soft_rank_rows(1024, 8192, 1.0, 0)
        g = normal((1024, 8192), 1)
        return Workload(name, 1024, 8192, False, False, y, None, g)
    raise KeyError(name)


# ---------------------------------------------------------------------------
# Data families of the paper's accuracy study (Section 7.6) and weightings.
# ---------------------------------------------------------------------------
FAMILIES = ("increasing", "decreasing", "constant", "piecewise", "gaussian", "random_walk",
            "sawtooth", "cliff", "collinear", "offset", "noise", "cancellation", "ties")
WEIGHTINGS = ("none", "uniform", "extreme")


def family(name: str, rows: int, n: int, seed: int = 0) -> np.ndarray:
    """float32 ``[rows, n]`` rows of one data family."""
    rng = np.random.default_rng(seed)
    i = np.arange(n, dtype=np.float64)[None, :]
    shape = (rows, n)
    if name == "increasing":
        y = np.sort(rng.random(shape), axis=1) + 1e-7 * i
    elif name == "decreasing":
        y = -np.sort(rng.random(shape), axis=1) - 1e-7 * i
    elif name == "constant":
        y = np.broadcast_to(rng.standard_normal((rows, 1)), shape).copy()
    elif name == "piecewise":
        k = max(1, n // 64)
        levels = np.sort(rng.standard_normal((rows, k)), axis=1)
        idx = np.minimum((i * k / max(n, 1)).astype(np.int64), k - 1)
        y = np.take_along_axis(levels, np.broadcast_to(idx, shape), axis=1)
        y = y + 0.1 * rng.standard_normal(shape)
    elif name == "gaussian":
        y = rng.standard_normal(shape)
    elif name == "random_walk":
        y = np.cumsum(rng.standard_normal(shape), axis=1)
    elif name == "sawtooth":
        period = max(2, n // 8)
        y = (i % period) / period + 0.01 * rng.standard_normal(shape)
    elif name == "cliff":
        y = np.sort(rng.random(shape), axis=1) + 1e-7 * i
        y[:, -1] = -1e3
    elif name == "collinear":
        y = 1.0 + 1e-6 * rng.standard_normal(shape)
    elif name == "offset":
        y = 1e6 + np.linspace(0.0, 3.0, n)[None, :] + rng.standard_normal(shape)
    elif name == "noise":
        y = np.linspace(0.0, 3.0, n)[None, :] + rng.standard_normal(shape)
    elif name == "cancellation":
        # per 64 elements: 32 x (+B), one -32B and 31 small, nearly collinear values
        B = 1e6
        y = np.empty(shape)
        for start in range(0, n, 64):
            seg = y[:, start:start + 64]
            m = seg.shape[1]
            blk = np.concatenate([np.full(32, B), [-32 * B], 1e-3 * np.arange(31)
                                  + 1e-9 * rng.standard_normal(31)])
            seg[:] = blk[:m][None, :]
    elif name == "ties":
        y = rng.integers(0, 4, size=shape).astype(np.float64)
    else:
        raise KeyError(name)
    return np.ascontiguousarray(y, dtype=np.float32)


def weights(kind: str, rows: int, n: int, seed: int = 0):
    """None (unit), U[0.1, 1.1], or exp(U[0, 8]) (dynamic range ~3e3)."""
    rng = np.random.default_rng(seed + 7919)
    if kind == "none":
        return None
    if kind == "uniform":
        return rng.uniform(0.1, 1.1, size=(rows, n)).astype(np.float32)
    if kind == "extreme":
        return np.exp(rng.uniform(0.0, 8.0, size=(rows, n))).astype(np.float32)
    raise KeyError(kind)
