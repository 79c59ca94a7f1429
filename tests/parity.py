"""Helpers shared by the GPU parity tests: run the oracle on the same seeded
bf16 inputs and compare element by element within the stated tolerances."""
import numpy as np
import torch

import oracle
from workloads import to_f64

# Tolerances (absolute, over every valid element): O within 2e-2, LSE within
# 5e-3, gradients within 5e-2.  Empty rows must match exactly.
TOL_O = 2e-2
TOL_LSE = 5e-3
TOL_GRAD = 5e-2


def tile_edge_rows(L, n_random=64, seed=0):
    """Rows at every 128-tile boundary neighbourhood of a long sequence (first
    and last tiles in full) plus random rows."""
    rows = set(range(min(L, 130)))
    rows |= set(range(max(0, L - 130), L))
    rng = np.random.default_rng(seed)
    rows |= set(int(x) for x in rng.integers(0, L, size=n_random))
    for t in range(0, L, 128 * max(1, L // (128 * 16))):
        for r in (t - 1, t, t + 1, t + 127):
            if 0 <= r < L:
                rows.add(r)
    return np.array(sorted(rows))


def compare_forward(o_gpu, lse_gpu, O_ref, lse_ref, what=""):
    """Element-wise check: finite rows within tolerance, empty rows exact."""
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.float().cpu().numpy().astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: empty-row pattern differs"
    assert np.all(o[empty] == 0.0), f"{what}: empty rows must give O == 0"
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    fin = ~empty
    do = np.abs(o - O_ref).max() if o.size else 0.0
    dl = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert do <= TOL_O, f"{what}: max|dO| = {do:.3e}"
    assert dl <= TOL_LSE, f"{what}: max|dLSE| = {dl:.3e}"
    return do, dl


def oracle_forward(inp, scale, rows=None, heads=None, **kw):
    q, k, v = (to_f64(inp[n]) for n in ("q", "k", "v"))
    return oracle.attention_forward(q, k, v, scale, rows=rows, heads=heads, **kw)


def to_cuda(inp):
    return {n: t.cuda() for n, t in inp.items()}
