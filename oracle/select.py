"""CPU oracle for the mean-pooled block selector (test infrastructure only).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the product library
never imports, links or calls it, and it shares no code with the CUDA path.

It follows "Exact Blocks, Rings, and Sparsity" (g-u-n.github.io blog):
  * section 5 ("Why the sparse unit is usually a block"): the selector picks,
    per query tile, the key tiles C_a the block-sparse kernel visits, and it
    must score something cheaper than the full QK^T matrix;
  * section 5 ("Fixed pooling: a cheap proxy, not the true block mass"): a key
    block is summarised by the mean of its keys, and the block's score is the
    mean logit, which ranks blocks like the exact block mass
    log sum_j exp(s_ij) when the logits inside a block are close;
  * section 5 (the selector chooses an exact set: selected blocks united with
    a mandatory local window);
  * section 6 (under grouped heads, query heads that share a KV head share the
    block choice).

Readings where the pages are silent, each taken here as stated:
  * the score of query block a against key block c is the mean logit over the
    pair of blocks, scale * qbar_a . kbar_c, with qbar and kbar the means of
    the block's query and key rows (the mean of the per-query pooled scores of
    the pages over the queries of the block);
  * heads that share a list add their pooled scores;
  * the local window is the `local` most recent key blocks a, a-1, ...,
    a-local+1 (those >= 0); the top-r are chosen among the other candidate
    blocks (under a causal mask, blocks 0..a; otherwise all), larger score
    first, the lower block index first on equal scores;
  * the row lists local and selected blocks together in ascending order.

Precision: the pooled means and scores are computed in the dtype given
(float32 by default, the kernel's precision, because the scores decide which
integers are selected).
"""
from __future__ import annotations

import numpy as np


def pool_blocks(x, block: int = 128, dtype=np.float32):
    """Mean of each block of rows of x [..., L, d]: [..., ceil(L/block), d]
    (the last block averages only its L - (n-1)*block rows)."""
    x = np.asarray(x, dtype=dtype)
    L = x.shape[-2]
    n = (L + block - 1) // block
    out = np.zeros(x.shape[:-2] + (n, x.shape[-1]), dtype=dtype)
    for c in range(n):
        out[..., c, :] = x[..., c * block:min(L, (c + 1) * block), :].mean(axis=-2, dtype=dtype)
    return out


def pooled_scores(q, k, scale, block: int = 128, dtype=np.float32):
    """scale * qbar_a . kbar_c for one head: [n_qblk, n_kblk]."""
    qb = pool_blocks(q, block, dtype)
    kb = pool_blocks(k, block, dtype)
    return (dtype(scale) * (qb @ kb.T)).astype(dtype)


def select_row(scores_row, a: int, n_kblk: int, top_r: int, local: int, causal: bool):
    """Blocks kept for query block a: the local window united with the top_r
    highest-scoring other candidates (ties: lower index first), ascending."""
    last = a if causal else n_kblk - 1
    window = set(c for c in range(a - local + 1, a + 1) if 0 <= c <= last)
    cand = [c for c in range(last + 1) if c not in window]
    cand.sort(key=lambda c: (-float(scores_row[c]), c))
    return sorted(window | set(cand[:top_r]))


def select_blocks(q, k, scale, *, top_r: int, local: int, causal: bool, n_lists: int,
                  block: int = 128, dtype=np.float32):
    """Block lists for q [B,H,L,d] and k [B,H_kv,L,d]: ``n_lists`` lists over the
    B*H query heads in consecutive groups (head b*H + h uses list
    (b*H + h) // (B*H // n_lists)); query head h pools the keys of key head
    h // (H / H_kv).
    Returns (row_ptr [n_lists, n+1], col_idx, lists) where row_ptr holds
    offsets into the one col_idx array and ``lists`` the per-list rows."""
    B, H, L, _ = q.shape
    G = H // k.shape[1]
    n = (L + block - 1) // block
    hpl = B * H // n_lists
    lists = []
    for lst in range(n_lists):
        S = np.zeros((n, n), dtype=dtype)
        for x in range(lst * hpl, (lst + 1) * hpl):
            b, h = divmod(x, H)
            S = (S + pooled_scores(q[b, h], k[b, h // G], scale, block, dtype)).astype(dtype)
        lists.append([select_row(S[a], a, n, top_r, local, causal) for a in range(n)])
    rps, cols, off = [], [], 0
    for rows in lists:
        rp = [off]
        for r in rows:
            cols.extend(r)
            off += len(r)
            rp.append(off)
        rps.append(rp)
    return np.array(rps, dtype=np.int32), np.array(cols, dtype=np.int32), lists


def block_mass(q, k, scale, block: int = 128):
    """Exact block mass of one head, log sum_{i in a, j in c} exp(s_ij), in
    float64: the quantity pooling stands in for."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    Lq, Lk = q.shape[0], k.shape[0]
    nq, nk = (Lq + block - 1) // block, (Lk + block - 1) // block
    S = scale * (q @ k.T)
    out = np.zeros((nq, nk))
    for a in range(nq):
        for c in range(nk):
            blk = S[a * block:min(Lq, (a + 1) * block), c * block:min(Lk, (c + 1) * block)]
            m = blk.max()
            out[a, c] = m + np.log(np.exp(blk - m).sum())
    return out
