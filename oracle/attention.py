"""fp64 CPU oracle for exact, causal, block-sparse and chunk-merged softmax attention.

TEST INFRASTRUCTURE ONLY.  The product library never imports, links or calls
anything in this package; only the tests, the smoke check and the CPU-baseline
leg of the benchmark use it.  It shares no code with the CUDA path.

It follows the definitions on these web pages (cited by title and section):

  [EBRS] "Exact Blocks, Rings, and Sparsity" (g-u-n.github.io blog):
         §1 dense attention, §2 online softmax state and merge invariant,
         §3 backward by recomputation, §4 Ring-Attention merge,
         §5-6 block-sparse schedule and drop-and-renormalise semantics.
  [FA]   "FlashAttention: Fast and Memory Efficient Exact Attention with IO
         Awareness" (reading notes): §5.1 online softmax statistics, §5.3
         backward recomputation (D_i = dO_i . O_i, dS = P o (dP - D)),
         Theorem 1 (the tiled algorithm returns exactly softmax(QK^T)V).
  [BSP]  block-sparse attention patterns page, "Count active blocks and
         acknowledge the changed operator": renormalise over the sparse
         domain, triangular element mask inside diagonal blocks, duplicates
         never counted twice, empty rows, build the reference from logical
         token pairs.

Like the conventional three-stage computation ([EBRS] §1) it materialises the
score matrix S and the probability matrix P for the rows it evaluates.  Rows are
processed in groups only to bound memory; every row is computed from its full
definition.

Readings where the pages are silent, each taken here as stated:
  * masked pairs contribute exactly zero (mask value -inf, not a large finite
    number);
  * a row with no allowed key has O = 0 and LSE = -inf and gets zero gradient;
  * causal visibility with offsets is ``j + k_offset <= i + q_offset``;
  * LSE is the natural log of the normaliser of the *scaled* logits;
  * grouped key/value heads ([EBRS] §6: under grouped-query attention several
    query heads share one physical KV head): with H query heads and H_kv key/
    value heads, H_kv dividing H, query head h reads key/value head
    h // (H / H_kv) (consecutive groups), and the gradient of a shared key/
    value head is the sum of the gradients its query heads send it.

Parity status: every function here is pinned by tests against closed forms,
the pages' worked examples, invariants, a library routine and brute force.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# Allowed pairs  ([BSP]; causal element mask [EBRS] §4 / [BSP])
# ---------------------------------------------------------------------------

def blocklist_sets(row_ptr: np.ndarray, col_idx: np.ndarray, n_kblk: int) -> list:
    """Set of active key blocks per query block.

    Set semantics: a block listed twice is the same block ([BSP]: duplicate
    entries must not count a key twice).  Raises ValueError on malformed CSR.
    """
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    col_idx = np.asarray(col_idx, dtype=np.int64)
    if row_ptr.ndim != 1 or len(row_ptr) < 1 or row_ptr[0] != 0:
        raise ValueError("row_ptr must be 1-D and start at 0")
    if np.any(np.diff(row_ptr) < 0):
        raise ValueError("row_ptr must be non-decreasing")
    if row_ptr[-1] != len(col_idx):
        raise ValueError("row_ptr[-1] must equal the number of column entries")
    if len(col_idx) and (col_idx.min() < 0 or col_idx.max() >= n_kblk):
        raise ValueError("block index out of range")
    return [set(int(c) for c in col_idx[row_ptr[a]:row_ptr[a + 1]])
            for a in range(len(row_ptr) - 1)]


def blocklist_normalize(row_ptr: np.ndarray, col_idx: np.ndarray, n_kblk: int
                        ) -> Tuple[np.ndarray, np.ndarray]:
    """Canonical CSR: each row's set of blocks in ascending order."""
    sets = blocklist_sets(row_ptr, col_idx, n_kblk)
    out_ptr = np.zeros(len(sets) + 1, dtype=np.int32)
    cols = []
    for a, s in enumerate(sets):
        out_ptr[a + 1] = out_ptr[a] + len(s)
        cols.extend(sorted(s))
    return out_ptr, np.array(cols, dtype=np.int32)


def allowed_rows(rows: Sequence[int], Lk: int, *, causal: bool = False,
                 q_offset: int = 0, k_offset: int = 0, block: Optional[int] = None,
                 row_ptr=None, col_idx=None) -> np.ndarray:
    """Boolean [len(rows), Lk]: which (query row, key) pairs are allowed.

    Built from logical token pairs ([BSP]): key j is visible to query i when
      * causal is off, or j + k_offset <= i + q_offset, and
      * block-sparse is off, or block(j) is in the set listed for block(i).
    """
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(Lk, dtype=np.int64)[None, :]
    M = np.ones((i.shape[0], Lk), dtype=bool)
    if causal:
        M &= (j + k_offset) <= (i + q_offset)
    if row_ptr is not None:
        assert block is not None
        n_kblk = (Lk + block - 1) // block
        sets = blocklist_sets(row_ptr, col_idx, n_kblk)
        blk = np.zeros((len(sets), n_kblk), dtype=bool)
        for a, s in enumerate(sets):
            for c in s:
                blk[a, c] = True
        M &= blk[i // block, j // block]
    return M


def allowed_mask(Lq: int, Lk: int, **kw) -> np.ndarray:
    return allowed_rows(np.arange(Lq), Lk, **kw)


# ---------------------------------------------------------------------------
# Forward  ([EBRS] §1, [FA] Theorem 1: the method returns exactly this)
# ---------------------------------------------------------------------------

def _rows_forward(q_rows, k, v, scale, M):
    """O and LSE for a group of query rows of one head, from the definition."""
    S = scale * (q_rows @ k.T)                       # scores, scaled logits
    Sm = np.where(M, S, NEG_INF)
    has = M.any(axis=1)
    m = np.where(has, Sm.max(axis=1, initial=NEG_INF), 0.0)
    E = np.where(M, np.exp(Sm - m[:, None]), 0.0)
    ell = E.sum(axis=1)
    O = np.zeros((q_rows.shape[0], v.shape[1]))
    lse = np.full(q_rows.shape[0], NEG_INF)
    P = np.zeros_like(E)
    P[has] = E[has] / ell[has, None]                 # renormalised over allowed keys
    O[has] = P[has] @ v
    lse[has] = m[has] + np.log(ell[has])
    return O, lse, P


def forward_head(q, k, v, scale, mask_fn, rows=None, group=256):
    """One head.  ``mask_fn(rows) -> bool[len(rows), Lk]``.  Returns (O, LSE)
    for ``rows`` (default: all rows)."""
    Lq = q.shape[0]
    rows = np.arange(Lq) if rows is None else np.asarray(rows)
    O = np.zeros((len(rows), v.shape[1]))
    lse = np.full(len(rows), NEG_INF)
    for s in range(0, len(rows), group):
        r = rows[s:s + group]
        o_, l_, _ = _rows_forward(q[r], k, v, scale, mask_fn(r))
        O[s:s + group] = o_
        lse[s:s + group] = l_
    return O, lse


def kv_group(H: int, H_kv: int) -> int:
    """Query heads per key/value head; H_kv must divide H ([EBRS] §6)."""
    if H_kv < 1 or H % H_kv:
        raise ValueError(f"{H_kv} key/value heads do not divide {H} query heads")
    return H // H_kv


def attention_forward(q, k, v, scale, *, causal=False, q_offset=0, k_offset=0,
                      block=None, row_ptr=None, col_idx=None, rows=None,
                      heads=None):
    """O [B,H,R,d] and LSE [B,H,R] for arrays q [B,H,Lq,d], k/v [B,H_kv,Lk,d].

    Query head h reads key/value head h // (H / H_kv).  ``rows`` restricts the
    evaluation to a subset of query rows (all heads); ``heads`` to a list of
    (b, h) query heads (the result then has shape [n, R, ...]).
    """
    Lk = k.shape[-2]
    G = kv_group(q.shape[1], k.shape[1])

    def mask_fn(r):
        return allowed_rows(r, Lk, causal=causal, q_offset=q_offset, k_offset=k_offset,
                            block=block, row_ptr=row_ptr, col_idx=col_idx)

    if heads is not None:
        outs = [forward_head(q[b, h], k[b, h // G], v[b, h // G], scale, mask_fn, rows)
                for b, h in heads]
        return np.stack([o for o, _ in outs]), np.stack([l for _, l in outs])
    B, H = q.shape[:2]
    R = q.shape[2] if rows is None else len(rows)
    O = np.zeros((B, H, R, v.shape[-1]))
    lse = np.zeros((B, H, R))
    for b in range(B):
        for h in range(H):
            O[b, h], lse[b, h] = forward_head(q[b, h], k[b, h // G], v[b, h // G], scale,
                                              mask_fn, rows)
    return O, lse


def probabilities(q, k, scale, M):
    """The full probability matrix P of one head (rows with no allowed key are 0)."""
    _, _, P = _rows_forward(q, k, np.zeros((k.shape[0], 1)), scale, M)
    return P


# ---------------------------------------------------------------------------
# Partial states and their merge  ([EBRS] §2 merge invariant, §4 Ring merge;
# [FA] §5.1 block-wise combination of m and l)
# ---------------------------------------------------------------------------

def partial_state(q, k, v, scale, M):
    """(m, l, A) of one head over the keys of ``k``/``v`` allowed by ``M``.

    m = max allowed scaled logit, l = sum exp(s - m), A = sum exp(s - m) V.
    A row with no allowed key has the empty state (-inf, 0, 0).
    """
    S = scale * (q @ k.T)
    has = M.any(axis=1)
    Sm = np.where(M, S, NEG_INF)
    m = Sm.max(axis=1, initial=NEG_INF)
    mm = np.where(has, m, 0.0)
    E = np.where(M, np.exp(Sm - mm[:, None]), 0.0)
    return m, E.sum(axis=1), E @ v


def merge_states(m, l, A):
    """Combine C partial states over disjoint key sets (leading axis C).

    m* = max_c m_c; each state is rescaled by exp(m_c - m*) and the l and A
    terms are added.  States with m_c = -inf are empty and weigh nothing.
    Returns (O = A*/l*, LSE = m* + ln l*), with O = 0, LSE = -inf for rows
    whose every state is empty.
    """
    m = np.asarray(m, dtype=np.float64)
    mstar = m.max(axis=0)
    has = np.isfinite(mstar)
    ms = np.where(has, mstar, 0.0)
    w = np.where(np.isfinite(m), np.exp(np.where(np.isfinite(m), m, 0.0) - ms), 0.0)
    lstar = (w * l).sum(axis=0)
    Astar = (w[..., None] * A).sum(axis=0)
    O = np.zeros_like(Astar)
    O[has] = Astar[has] / lstar[has][..., None]
    lse = np.full(mstar.shape, NEG_INF)
    lse[has] = mstar[has] + np.log(lstar[has])
    return O, lse


def merge_pair(sa, sb):
    """Associative merge of two states (m, l, A) into one state ([EBRS] §4)."""
    (ma, la, Aa), (mb, lb, Ab) = sa, sb
    mn = np.maximum(ma, mb)
    fin = np.isfinite(mn)
    mref = np.where(fin, mn, 0.0)
    wa = np.where(np.isfinite(ma), np.exp(np.where(np.isfinite(ma), ma, 0.0) - mref), 0.0)
    wb = np.where(np.isfinite(mb), np.exp(np.where(np.isfinite(mb), mb, 0.0) - mref), 0.0)
    return mn, wa * la + wb * lb, wa[..., None] * Aa + wb[..., None] * Ab


def finalize_state(m, l, A):
    """O = A / l and LSE = m + ln l; empty rows give O = 0, LSE = -inf."""
    has = l > 0
    O = np.zeros_like(A)
    O[has] = A[has] / l[has][..., None]
    lse = np.full(np.shape(m), NEG_INF)
    lse[has] = np.asarray(m)[has] + np.log(l[has])
    return O, lse


# ---------------------------------------------------------------------------
# Backward  ([EBRS] §3; [FA] §5.3)
# ---------------------------------------------------------------------------

def backward_head(q, k, v, do, scale, M):
    """Gradients of one head for upstream dO, with P recomputed from scratch.

    dV = P^T dO;  dP = dO V^T;  D_i = sum_j P_ij dP_ij;  dS = P o (dP - D);
    dQ = scale dS K;  dK = scale dS^T Q.  Returns (dq, dk, dv, D).
    """
    P = probabilities(q, k, scale, M)
    dv = P.T @ do
    dP = do @ v.T
    D = (P * dP).sum(axis=1)
    dS = P * (dP - D[:, None])
    dq = scale * (dS @ k)
    dk = scale * (dS.T @ q)
    return dq, dk, dv, D


def attention_backward(q, k, v, do, scale, *, causal=False, block=None, row_ptr=None,
                       col_idx=None, heads=None):
    """(dq, dk, dv, D) for q/do [B,H,L,d] and k/v [B,H_kv,L,d] (square, offsets 0).

    dk and dv of key/value head g add the gradients of its query heads
    g*G .. g*G+G-1 (G = H / H_kv).  With ``heads`` (a list of (b, h) query
    heads) the per-query-head terms are returned unsummed, shape [n, L, d].
    """
    Lq, Lk = q.shape[-2], k.shape[-2]
    G = kv_group(q.shape[1], k.shape[1])
    M = allowed_mask(Lq, Lk, causal=causal, block=block, row_ptr=row_ptr, col_idx=col_idx)
    if heads is not None:
        outs = [backward_head(q[b, h], k[b, h // G], v[b, h // G], do[b, h], scale, M)
                for b, h in heads]
        return tuple(np.stack([o[i] for o in outs]) for i in range(4))
    B, H = q.shape[:2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(H):
            dq[b, h], dk_h, dv_h, D[b, h] = backward_head(
                q[b, h], k[b, h // G], v[b, h // G], do[b, h], scale, M)
            dk[b, h // G] += dk_h
            dv[b, h // G] += dv_h
    return dq, dk, dv, D


# ---------------------------------------------------------------------------
# Work counts ([BSP]: report logical allowed pairs and executed tile work)
# ---------------------------------------------------------------------------

def logical_pairs(M: np.ndarray) -> int:
    """Number of allowed (query, key) token pairs of a realised mask: the
    logical work of the operator ([BSP]: build the count from logical token
    pairs, not from the padded tiles)."""
    return int(M.sum())


def executed_tiles(M: np.ndarray, tile: int = 128) -> int:
    """Number of (query tile, key tile) pairs with at least one allowed pair:
    the tile work a kernel that skips empty tiles executes ([BSP]: executed
    lanes differ from logical pairs)."""
    Lq, Lk = M.shape
    nq, nk = (Lq + tile - 1) // tile, (Lk + tile - 1) // tile
    pad = np.zeros((nq * tile, nk * tile), dtype=bool)
    pad[:Lq, :Lk] = M
    return int(pad.reshape(nq, tile, nk, tile).any(axis=(1, 3)).sum())


def blocklist_stats(row_ptr, col_idx, L: int, *, causal: bool, block: int = 128) -> dict:
    """What a block list asks for on a square sequence of L tokens ([BSP],
    "Count active blocks and acknowledge the changed operator": report the
    logical allowed pairs and the executed tile work; under a causal mask the
    token-level rule applies inside every listed block, so a listed block that
    lies wholly in the causal future contributes nothing).

      listed    listed (query block, key block) pairs, duplicates counted once
      executed  listed pairs whose tile holds at least one allowed token pair
      future    listed pairs with no allowed token pair under the causal mask
                (every key of the block after every query of the block)
      pairs     allowed token pairs of the realised mask
    """
    n = (L + block - 1) // block
    sets = blocklist_sets(row_ptr, col_idx, n)
    M = allowed_mask(L, L, causal=causal, block=block, row_ptr=row_ptr, col_idx=col_idx)
    future = 0
    if causal:
        for a, s in enumerate(sets):
            last_query = min(L, (a + 1) * block) - 1
            future += sum(1 for c in s if c * block > last_query)
    return {"listed": sum(len(s) for s in sets), "executed": executed_tiles(M, block),
            "future": future, "pairs": logical_pairs(M)}
