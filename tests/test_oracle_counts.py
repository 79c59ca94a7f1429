"""Pins for the oracle's work counts: logical allowed pairs, executed tiles and
the block-list accounting (listed, executed, causal-future blocks).

The block-sparse attention patterns page ("Count active blocks and acknowledge
the changed operator") asks that a sparse run report both the logical allowed
token pairs and the executed tile work, and says the causal element rule
applies inside every listed block, so a listed block wholly in the causal future
contributes nothing.  These counts are checked here against scalar loops over
(query, key) written from that definition (no oracle helper involved) and
against closed forms of the dense and causal cases.
"""
import numpy as np
import pytest

import oracle
from workloads import local_global_random_blocklist, random_blocklist


def _brute(L, rp, ci, causal, block):
    """Scalar loops straight from the definition: key j is visible to query i
    when (not causal or j <= i) and block(j) appears in the raw list of
    block(i) (membership, so a duplicate cannot count twice)."""
    n = (L + block - 1) // block
    rows = [list(ci[rp[a]:rp[a + 1]]) for a in range(n)]
    pairs = 0
    tile_hit = set()
    for i in range(L):
        for j in range(L):
            if causal and j > i:
                continue
            if (j // block) not in rows[i // block]:
                continue
            pairs += 1
            tile_hit.add((i // block, j // block))
    listed = set()
    future = 0
    for a in range(n):
        for c in rows[a]:
            if (a, c) in listed:
                continue
            listed.add((a, c))
            qs = range(a * block, min(L, (a + 1) * block))
            ks = range(c * block, min(L, (c + 1) * block))
            if causal and all(j > i for i in qs for j in ks):
                future += 1
    return {"listed": len(listed), "executed": len(tile_hit), "future": future, "pairs": pairs}


@pytest.mark.parametrize("L,block,causal,seed", [(37, 8, True, 0), (37, 8, False, 1),
                                                 (64, 8, True, 2), (29, 4, True, 3),
                                                 (29, 4, False, 4), (9, 8, True, 5)])
def test_blocklist_stats_match_scalar_loops_on_random_lists(L, block, causal, seed):
    n = (L + block - 1) // block
    rp, ci = random_blocklist(n, n, seed=seed)       # random order, duplicates, empty rows
    got = oracle.blocklist_stats(rp, ci, L, causal=causal, block=block)
    assert got == _brute(L, rp, ci, causal, block)


def test_blocklist_stats_hand_example_with_future_duplicates_and_empty_row():
    # L = 20, blocks of 8: rows 0..7 | 8..15 | 16..19 (partial last block)
    rp = np.array([0, 3, 3, 8], np.int32)
    ci = np.array([2, 0, 0,          # row 0: block 2 is in the future, 0 listed twice
                   # row 1: empty
                   2, 1, 0, 2, 1],   # row 2: blocks 0, 1, 2 (2 and 1 listed twice)
                  np.int32)
    got = oracle.blocklist_stats(rp, ci, 20, causal=True, block=8)
    # row 0: block 0 -> 8*9/2 = 36 pairs; block 2 -> none (future)
    # row 2: 4 queries x 8 keys of block 0 and of block 1, plus the partial
    #        diagonal block 4*5/2 = 10
    assert got == {"listed": 5, "executed": 4, "future": 1, "pairs": 36 + 32 + 32 + 10}
    assert got == _brute(20, rp, ci, True, 8)


@pytest.mark.parametrize("L,block", [(1, 4), (8, 4), (30, 4), (129, 16), (200, 128)])
def test_causal_and_dense_closed_forms(L, block):
    n = (L + block - 1) // block
    full_rp = np.arange(n + 1, dtype=np.int32) * n
    full_ci = np.tile(np.arange(n, dtype=np.int32), n)
    tri_rp = np.concatenate([[0], np.cumsum(np.arange(1, n + 1))]).astype(np.int32)
    tri_ci = np.concatenate([np.arange(a + 1) for a in range(n)]).astype(np.int32)
    # every block listed, no mask: L^2 pairs, n^2 tiles
    assert oracle.blocklist_stats(full_rp, full_ci, L, causal=False, block=block) == {
        "listed": n * n, "executed": n * n, "future": 0, "pairs": L * L}
    # every block listed, causal: the upper triangle of blocks is future
    assert oracle.blocklist_stats(full_rp, full_ci, L, causal=True, block=block) == {
        "listed": n * n, "executed": n * (n + 1) // 2, "future": n * (n - 1) // 2,
        "pairs": L * (L + 1) // 2}
    # lower-triangular list, causal: exactly the causal dense work
    assert oracle.blocklist_stats(tri_rp, tri_ci, L, causal=True, block=block) == {
        "listed": n * (n + 1) // 2, "executed": n * (n + 1) // 2, "future": 0,
        "pairs": L * (L + 1) // 2}


@pytest.mark.parametrize("Lq,Lk,q0,k0,tile", [(20, 20, 0, 0, 8), (17, 40, 0, 9, 8),
                                              (33, 12, 5, 0, 4), (12, 30, 20, 3, 4)])
def test_logical_pairs_and_executed_tiles_of_causal_masks_with_offsets(Lq, Lk, q0, k0, tile):
    M = oracle.allowed_rows(np.arange(Lq), Lk, causal=True, q_offset=q0, k_offset=k0)
    pairs = sum(1 for i in range(Lq) for j in range(Lk) if j + k0 <= i + q0)
    tiles = len({(i // tile, j // tile) for i in range(Lq) for j in range(Lk) if j + k0 <= i + q0})
    assert oracle.logical_pairs(M) == pairs
    assert oracle.executed_tiles(M, tile) == tiles


def test_executed_tiles_ignores_tiles_with_only_masked_lanes():
    M = np.zeros((10, 10), dtype=bool)
    M[9, 0] = True          # tile (2, 0) of 4x4 tiles, in the partial last row of tiles
    M[0, 9] = True          # tile (0, 2)
    assert oracle.executed_tiles(M, 4) == 2
    assert oracle.logical_pairs(M) == 2
    assert oracle.executed_tiles(np.zeros((10, 10), dtype=bool), 4) == 0


def test_listed_equals_executed_plus_future_on_square_causal_lists():
    """On a square causal problem a listed block either holds the diagonal or
    earlier keys (executed) or lies wholly after the block's queries (future)."""
    for seed in range(4):
        L = 300 + 37 * seed
        n = (L + 127) // 128
        rp, ci = random_blocklist(n, n, seed=10 + seed)
        s = oracle.blocklist_stats(rp, ci, L, causal=True)
        assert s["listed"] == s["executed"] + s["future"]


def test_block_sparse_workload_counts():
    """L' = 16320, the local + global + random pattern of seed 2, one list:
    the generator only draws earlier blocks, so nothing is in the future;
    836 executed tiles and about 1.261e7 allowed pairs per head."""
    L = 16320
    rp, ci = local_global_random_blocklist((L + 127) // 128, seed=2)
    s = oracle.blocklist_stats(rp, ci, L, causal=True)
    assert s["future"] == 0
    assert s["listed"] == s["executed"] == 836
    assert abs(s["pairs"] - 1.261e7) <= 0.0005e7
