"""Pins of the mean-pooled block selector oracle (CPU).

Each pin ties oracle.select to something other than its own formula: the
brute-force mean of the full logit matrix, the exact block mass for the
homogeneous blocks where the pages say pooling ranks correctly, the pages'
stated failure mode (a block with one very relevant token), and direct
enumeration of the window, causal and top-r rules.
"""
import itertools

import numpy as np
import pytest

from oracle import select as sel


def test_pooled_score_is_the_mean_logit_of_the_block_pair():
    rng = np.random.default_rng(0)
    L, d, blk, scale = 300, 16, 64, 0.25                 # partial last block (44 rows)
    q = rng.standard_normal((L, d))
    k = rng.standard_normal((L, d))
    S = scale * (q @ k.T)
    got = sel.pooled_scores(q, k, scale, blk, dtype=np.float64)
    n = (L + blk - 1) // blk
    for a, c in itertools.product(range(n), range(n)):
        ref = S[a * blk:(a + 1) * blk, c * blk:(c + 1) * blk].mean()
        assert abs(got[a, c] - ref) <= 1e-12


def test_homogeneous_blocks_rank_like_the_block_mass():
    """Identical rows inside each block: every logit of a block pair equals the
    pooled score, so pooling ranks exactly like log sum exp (same-size blocks)."""
    rng = np.random.default_rng(1)
    n, blk, d, scale = 6, 32, 8, 0.5
    qb = rng.standard_normal((n, d))
    kb = rng.standard_normal((n, d))
    q = np.repeat(qb, blk, axis=0)
    k = np.repeat(kb, blk, axis=0)
    pooled = sel.pooled_scores(q, k, scale, blk, dtype=np.float64)
    mass = sel.block_mass(q, k, scale, blk)
    for a in range(n):
        assert list(np.argsort(-pooled[a], kind="stable")) == list(np.argsort(-mass[a], kind="stable"))
        # and the mass is the pooled score plus log(block pair size)
        assert np.allclose(mass[a], pooled[a] + np.log(blk * blk), atol=1e-9)


def test_pooling_can_miss_a_block_with_one_relevant_token():
    """The pages' failure mode: one key aligned with the query makes block 1's
    mass the larger, but its other keys pull block 1's mean below block 0's."""
    d, blk, scale = 4, 8, 1.0
    q = np.tile(np.array([1.0, 0, 0, 0]), (blk, 1))
    k0 = np.tile(np.array([1.0, 0, 0, 0]), (blk, 1))               # uniformly moderate
    k1 = np.tile(np.array([-1.0, 0, 0, 0]), (blk, 1))
    k1[3] = [12.0, 0, 0, 0]                                        # one very relevant key
    k = np.concatenate([k0, k1])
    pooled = sel.pooled_scores(q, k, scale, blk, dtype=np.float64)[0]
    mass = sel.block_mass(q, k, scale, blk)[0]
    assert pooled[0] > pooled[1]          # pooling prefers block 0 ...
    assert mass[1] > mass[0]              # ... though block 1 holds more attention mass


@pytest.mark.parametrize("causal", [True, False])
def test_rows_hold_window_and_best_candidates(causal):
    rng = np.random.default_rng(2)
    n, top_r, local = 9, 3, 2
    S = rng.standard_normal((n, n)).astype(np.float32)
    for a in range(n):
        row = sel.select_row(S[a], a, n, top_r, local, causal)
        last = a if causal else n - 1
        window = {c for c in (a, a - 1) if c >= 0}
        assert row == sorted(set(row))                       # ascending, no duplicates
        assert window <= set(row)                            # mandatory local window
        assert all(c <= last for c in row)                   # nothing in the causal future
        others = [c for c in range(last + 1) if c not in window]
        picked = [c for c in row if c not in window]
        assert len(picked) == min(top_r, len(others))
        rest = [c for c in others if c not in picked]
        if picked and rest:                                  # picked are the best candidates
            assert min(S[a][picked]) >= max(S[a][rest])


def test_ties_prefer_the_lower_block_index():
    S = np.zeros(6, dtype=np.float32)
    assert sel.select_row(S, 5, 6, 2, 1, causal=True) == [0, 1, 5]


def test_shared_lists_add_the_heads_scores():
    rng = np.random.default_rng(3)
    B, H, L, d, scale = 1, 2, 512, 16, 0.25
    q = rng.standard_normal((B, H, L, d)).astype(np.float32)
    k = rng.standard_normal((B, H, L, d)).astype(np.float32)
    rp, ci, lists = sel.select_blocks(q, k, scale, top_r=1, local=1, causal=True, n_lists=1)
    S = sel.pooled_scores(q[0, 0], k[0, 0], scale) + sel.pooled_scores(q[0, 1], k[0, 1], scale)
    n = (L + 127) // 128
    assert lists[0] == [sel.select_row(S[a], a, n, 1, 1, True) for a in range(n)]
    assert rp.shape == (1, n + 1) and rp[0, -1] == len(ci)
    # one list per head: each head its own scores
    _, _, per_head = sel.select_blocks(q, k, scale, top_r=1, local=1, causal=True, n_lists=2)
    S1 = sel.pooled_scores(q[0, 1], k[0, 1], scale)
    assert per_head[1] == [sel.select_row(S1[a], a, n, 1, 1, True) for a in range(n)]


def test_grouped_heads_pool_their_shared_key_head():
    """Query heads 0, 1 share key head 0 and heads 2, 3 key head 1: a list over
    each pair adds the two query heads' scores against that pair's key head."""
    rng = np.random.default_rng(4)
    B, H, Hkv, L, d, scale = 1, 4, 2, 640, 8, 0.3
    q = rng.standard_normal((B, H, L, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    _, _, lists = sel.select_blocks(q, k, scale, top_r=2, local=1, causal=False, n_lists=2)
    n = (L + 127) // 128
    for lst, kh in ((0, 0), (1, 1)):
        S = (sel.pooled_scores(q[0, 2 * lst], k[0, kh], scale)
             + sel.pooled_scores(q[0, 2 * lst + 1], k[0, kh], scale))
        assert lists[lst] == [sel.select_row(S[a], a, n, 2, 1, False) for a in range(n)]
