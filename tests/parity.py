"""Shared helpers for the GPU parity tests: device copies, NaN-poisoned
outputs and the error bound every comparison with the oracle uses.

Tolerance (stated for this path): bf16 output within max-abs 2e-2 and
mean-abs 2e-3 of the unrounded fp64 oracle for N(0,1) inputs; for the
large-magnitude stress inputs (q,k x8, v x100) both bounds are multiplied by
max|v| of that input.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def tolerance_scale(v: torch.Tensor, stress: bool) -> float:
    return float(v.float().abs().max()) if stress else 1.0


def poisoned(shape, device="cuda"):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device=device)


def assert_close(got: torch.Tensor, want: np.ndarray, scale: float = 1.0, what: str = ""):
    g = got.detach().double().cpu().numpy().reshape(want.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output (unwritten rows?)"
    err = np.abs(g - want)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS * scale, f"{what}: max abs err {mx:.3e} > {MAX_ABS * scale:.3e}"
    assert mean <= MEAN_ABS * scale, f"{what}: mean abs err {mean:.3e} > {MEAN_ABS * scale:.3e}"
    return mx, mean


def sample_rows(S: int, n_random: int = 24, seed: int = 0):
    """Query rows for a sampled comparison: both ends, tile boundaries, random."""
    rows = {0, 1, 2, S - 1, S - 2, S - 3}
    for b in (127, 128, 255, 256, 257):
        if b < S:
            rows.add(b)
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, S, size=n_random))
    return sorted(r for r in rows if 0 <= r < S)


TILE = 128  # query rows per tile of the prefill kernel (two tiles per work item)


def tile_rows(S: int, seed: int = 0):
    """Rows that put every 128-row query tile under comparison: its first
    row, its last row and one random row inside it.  Every 256-row work item
    (both of its tiles) and, with all heads compared, every (item, head)
    pair of a single-sequence prefill is then checked element by element."""
    rng = np.random.default_rng(seed)
    rows = set()
    for t0 in range(0, S, TILE):
        t1 = min(S, t0 + TILE) - 1
        rows.update((t0, t1, int(rng.integers(t0, t1 + 1))))
    return sorted(rows)


def covered_tiles(rows, S: int) -> int:
    """Number of distinct 128-row query tiles that contain one of `rows`."""
    return len({r // TILE for r in rows if 0 <= r < S})


def bf16_ulp_distance(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """Distance in bf16 units in the last place between two bf16 tensors of one
    shape (neighbouring representable values are 1 apart; +0 and -0 coincide)."""
    def order(x):
        i = x.contiguous().view(torch.int16).to(torch.int32)
        mag = i & 0x7FFF
        return torch.where(i < 0, -mag, mag)
    return (order(a) - order(b)).abs()
