"""The bench's work accounting against brute force: allowed pairs of a causal
mask with offsets, and (logical pairs, executed tiles) of block lists with
duplicates, empty rows and a partial last block.  Every TFLOP/s and pairs/s
figure the bench reports divides these counts by a time."""
import numpy as np
import pytest

import bench
import oracle
from workloads import local_global_random_blocklist, random_blocklist


@pytest.mark.parametrize("Lq,Lk,q0,k0", [(1, 1, 0, 0), (130, 300, 0, 0), (257, 129, 5, 300),
                                         (64, 1000, 936, 0), (300, 260, 0, 100), (17, 40, 0, 50)])
def test_causal_pairs_is_the_mask_count(Lq, Lk, q0, k0):
    M = oracle.allowed_rows(np.arange(Lq), Lk, causal=True, q_offset=q0, k_offset=k0)
    assert bench.causal_pairs(Lq, Lk, q0=q0, k0=k0) == int(M.sum())


def _brute_sparse(L, rp, ci, causal, block=128):
    M = oracle.allowed_rows(np.arange(L), L, causal=causal, block=block, row_ptr=rp, col_idx=ci)
    n = (L + block - 1) // block
    tiles = 0
    for a in range(n):
        for c in range(n):
            if M[a * block:(a + 1) * block, c * block:(c + 1) * block].any():
                tiles += 1
    return int(M.sum()), tiles


@pytest.mark.parametrize("L,causal,seed", [(1000, True, 0), (1000, False, 1), (640, True, 2),
                                           (129, True, 3)])
def test_sparse_counts_match_the_mask(L, causal, seed):
    n = (L + 127) // 128
    rp, ci = random_blocklist(n, n, seed=seed)
    assert bench.sparse_counts(L, rp, ci, causal) == _brute_sparse(L, rp, ci, causal)


def test_sparse_counts_local_global_pattern_with_duplicates_and_an_empty_row():
    L = 2000
    n = (L + 127) // 128
    rp, ci = local_global_random_blocklist(n, seed=5)
    assert bench.sparse_counts(L, rp, ci, True) == _brute_sparse(L, rp, ci, True)


def test_block_sparse_workload_counts_per_head():
    """L' = 16320, the local + global + random pattern of seed 2: about 1.261e7
    allowed pairs and 836 executed tiles per head (the study's figures)."""
    L = 16320
    rp, ci = local_global_random_blocklist((L + 127) // 128, seed=2)
    pairs, tiles = bench.sparse_counts(L, rp, ci, True)
    assert tiles == 836
    assert abs(pairs - 1.261e7) <= 0.0005e7


@pytest.mark.parametrize("L,seed", [(1000, 7), (16320, 2)])
def test_sparse_counts_equal_the_oracles_pinned_counts(L, seed):
    n = (L + 127) // 128
    rp, ci = local_global_random_blocklist(n, seed=seed)
    s = oracle.blocklist_stats(rp, ci, L, causal=True)
    assert bench.sparse_counts(L, rp, ci, True) == (s["pairs"], s["executed"])
