"""Pins for the fp64 oracle: it is checked against what the pages and the
mathematics fix, never against itself.

* worked examples printed on the pages (tests/golden/*.json);
* closed forms (uniform keys, one dominant key, equal value rows);
* invariants (rows of P sum to 1, shift invariance, merge in any order and at any
  split, all-blocks-active sparse == dense, D_i = dO_i . O_i, constant dP row);
* a library routine (torch scaled_dot_product_attention in fp64 with the same
  boolean mask, and torch autograd for the gradients);
* brute force on tiny inputs (scalar loops, central finite differences).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import local_global_random_blocklist, random_blocklist

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, scale, M):
    """torch SDPA (fp64, CPU) with the boolean mask; rows must be non-empty."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    out = torch.nn.functional.scaled_dot_product_attention(
        t(q)[None, None], t(k)[None, None], t(v)[None, None],
        attn_mask=t(M)[None, None], scale=scale)
    return out[0, 0].numpy()


def _lse_lib(q, k, scale, M):
    s = torch.from_numpy(scale * (q @ k.T))
    s = s.masked_fill(~torch.from_numpy(M), float("-inf"))
    return torch.logsumexp(s, dim=-1).numpy()


# ---------------------------------------------------------------------------
# Worked examples from the pages
# ---------------------------------------------------------------------------

def test_three_logit_example_states_and_output():
    g = _golden("three_logit.json")
    q = np.ones((1, 1))
    k1 = np.array(g["tile1"]["logits"])[:, None]
    v1 = np.array(g["tile1"]["values"])[:, None]
    k2 = np.array(g["tile2"]["logits"])[:, None]
    v2 = np.array(g["tile2"]["values"])[:, None]
    M1 = np.ones((1, 2), bool)
    M2 = np.ones((1, 1), bool)
    m1, l1, A1 = oracle.partial_state(q, k1, v1, 1.0, M1)
    assert m1[0] == g["after_tile1"]["m"]
    assert abs(l1[0] - g["after_tile1"]["l"]) < 1e-13
    assert abs(A1[0, 0] - g["after_tile1"]["A"]) < 1e-13
    s2 = oracle.partial_state(q, k2, v2, 1.0, M2)
    m, l, A = oracle.merge_pair((m1, l1, A1), s2)
    assert m[0] == g["after_tile2"]["m"]
    assert abs(l[0] - g["after_tile2"]["l"]) < 1e-13
    assert abs(A[0, 0] - g["after_tile2"]["A"]) < 1e-12
    O, lse = oracle.finalize_state(m, l, A)
    assert abs(O[0, 0] - g["output"]) < 1e-13
    assert abs(lse[0] - g["lse"]) < 1e-12
    # the unsplit forward over the three keys gives the same numbers
    kk = np.concatenate([k1, k2])
    vv = np.concatenate([v1, v2])
    Of, lf = oracle.attention_forward(q[None, None], kk[None, None], vv[None, None], 1.0)
    assert abs(Of[0, 0, 0, 0] - g["output"]) < 1e-13
    assert abs(lf[0, 0, 0] - g["lse"]) < 1e-12
    # and the fixture itself matches the closed form written in it
    e1, e2 = math.exp(-1), math.exp(-2)
    assert abs(g["output"] - (2 * e1 + 4 * e2 + 10) / (1 + e1 + e2)) < 1e-15


def test_drop_and_renormalise_example():
    g = _golden("drop_renormalise.json")
    logits = np.array(g["logits"])
    q = np.ones((1, 1))
    k = logits[:, None]
    v = np.array(g["values"])[:, None]
    O, _ = oracle.attention_forward(q[None, None], k[None, None], v[None, None], 1.0)
    assert O[0, 0, 0, 0] == pytest.approx(g["dense_output"], abs=1e-14)
    # block size 1: selecting key blocks {0, 1} for the single query block
    row_ptr = np.array([0, len(g["selected"])], np.int32)
    col_idx = np.array(g["selected"], np.int32)
    Os, _ = oracle.attention_forward(q[None, None], k[None, None], v[None, None], 1.0,
                                     block=1, row_ptr=row_ptr, col_idx=col_idx)
    assert Os[0, 0, 0, 0] == pytest.approx(g["selected_output"], abs=1e-14)
    M = oracle.allowed_mask(1, 3, block=1, row_ptr=row_ptr, col_idx=col_idx)
    P = oracle.probabilities(q, k, 1.0, M)
    assert np.allclose(P[0, :2], g["selected_probability_each"], atol=1e-15)
    assert P[0, 2] == 0.0
    Pd = oracle.probabilities(q, k, 1.0, np.ones((1, 3), bool))
    assert np.allclose(Pd, g["dense_probability_each"], atol=1e-15)


# ---------------------------------------------------------------------------
# Invariants and closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one_and_lse_normalises(causal):
    q, k = _rand((40, 8), 1), _rand((40, 8), 2)
    scale = 0.7
    M = oracle.allowed_mask(40, 40, causal=causal)
    P = oracle.probabilities(q, k, scale, M)
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(P[~M] == 0)
    _, lse = oracle.attention_forward(q[None, None], k[None, None], _rand((40, 3), 3)[None, None],
                                      scale, causal=causal)
    S = scale * q @ k.T
    tot = np.where(M, np.exp(S - lse[0, 0][:, None]), 0.0).sum(axis=1)
    assert np.allclose(tot, 1.0, atol=1e-12)


def test_shift_invariance():
    """Adding c_i to every logit of row i leaves O unchanged and adds c_i to LSE.
    The shift is built into the inputs: one extra dimension with K == 1 and
    Q == c_i / scale."""
    L, d = 33, 5
    q, k, v = _rand((L, d), 4), _rand((L, d), 5), _rand((L, 3), 6)
    scale = 1 / math.sqrt(d)
    c = _rand((L,), 7) * 50
    q2 = np.concatenate([q, (c / scale)[:, None]], axis=1)
    k2 = np.concatenate([k, np.ones((L, 1))], axis=1)
    for causal in (False, True):
        O1, l1 = oracle.attention_forward(q[None, None], k[None, None], v[None, None], scale, causal=causal)
        O2, l2 = oracle.attention_forward(q2[None, None], k2[None, None], v[None, None], scale, causal=causal)
        assert np.allclose(O1, O2, atol=1e-12)
        assert np.allclose(l2 - l1, c[None, None], atol=1e-10)


@pytest.mark.parametrize("kind", ["dense", "causal", "sparse"])
def test_uniform_keys_give_mean_of_allowed_values(kind):
    L, d, blk = 48, 4, 8
    q = _rand((L, d), 8)
    krow = _rand((1, d), 9)
    k = np.repeat(krow, L, axis=0)
    v = _rand((L, 6), 10)
    scale = 0.9
    kw = {}
    if kind == "causal":
        kw = dict(causal=True)
    if kind == "sparse":
        rp, ci = random_blocklist(L // blk, L // blk, seed=11, p_empty=0.0)
        kw = dict(block=blk, row_ptr=rp, col_idx=ci, causal=True)
    M = oracle.allowed_mask(L, L, **kw)
    O, lse = oracle.attention_forward(q[None, None], k[None, None], v[None, None], scale, **kw)
    for i in range(L):
        n = M[i].sum()
        if n == 0:
            assert np.all(O[0, 0, i] == 0) and lse[0, 0, i] == -np.inf
            continue
        assert np.allclose(O[0, 0, i], v[M[i]].mean(axis=0), atol=1e-12)
        s = scale * float(q[i] @ krow[0])
        assert lse[0, 0, i] == pytest.approx(s + math.log(n), abs=1e-12)


def test_dominant_key_closed_form():
    """K_{j*} = u, every other key 0, q_i = t u: O_i = (e^{t s |u|^2} V_{j*} + sum_{j!=j*} V_j)
    / (e^{t s |u|^2} + n - 1), and a large t gives V_{j*}."""
    L, d = 20, 4
    u = np.array([0.5, -1.0, 0.25, 2.0])
    jstar = 13
    k = np.zeros((L, d))
    k[jstar] = u
    v = _rand((L, 3), 12)
    scale = 0.5
    for t in (0.3, 2.0, 40.0):
        q = np.tile(t * u, (L, 1))
        O, lse = oracle.attention_forward(q[None, None], k[None, None], v[None, None], scale)
        w = math.exp(t * scale * float(u @ u))
        expect = (w * v[jstar] + (v.sum(axis=0) - v[jstar])) / (w + L - 1)
        assert np.allclose(O[0, 0], expect[None], atol=1e-12)
        assert np.allclose(lse[0, 0], math.log(w + L - 1), atol=1e-12)
    assert np.allclose(O[0, 0], v[jstar][None], atol=1e-12)


def test_all_blocks_active_equals_dense_and_lower_triangle_equals_causal():
    L, d, blk = 70, 8, 16           # partial last block of 6 tokens
    q, k, v = (_rand((1, 2, L, d), s) for s in (13, 14, 15))
    n = (L + blk - 1) // blk
    scale = 1 / math.sqrt(d)
    full_ptr = np.arange(0, n * n + 1, n, dtype=np.int32)
    full_col = np.tile(np.arange(n, dtype=np.int32)[::-1], n)   # reversed order
    Od, ld = oracle.attention_forward(q, k, v, scale)
    Os, ls = oracle.attention_forward(q, k, v, scale, block=blk, row_ptr=full_ptr, col_idx=full_col)
    assert np.array_equal(Od, Os) and np.array_equal(ld, ls)
    tri = [list(range(a + 1)) for a in range(n)]
    tri_ptr = np.cumsum([0] + [len(r) for r in tri]).astype(np.int32)
    tri_col = np.array([c for r in tri for c in r], np.int32)
    Oc, lc = oracle.attention_forward(q, k, v, scale, causal=True)
    Ot, lt = oracle.attention_forward(q, k, v, scale, causal=True, block=blk,
                                      row_ptr=tri_ptr, col_idx=tri_col)
    assert np.array_equal(Oc, Ot) and np.array_equal(lc, lt)
    # a lower-triangular block list without the element mask is NOT causal ([BSP])
    On, _ = oracle.attention_forward(q, k, v, scale, block=blk, row_ptr=tri_ptr, col_idx=tri_col)
    assert not np.allclose(On, Oc)


def test_duplicates_and_order_do_not_change_the_result():
    L, d, blk = 64, 4, 8
    q, k, v = (_rand((1, 1, L, d), s) for s in (16, 17, 18))
    rp, ci = random_blocklist(L // blk, L // blk, seed=19)
    cp, cc = oracle.blocklist_normalize(rp, ci, L // blk)
    O1, l1 = oracle.attention_forward(q, k, v, 0.5, block=blk, row_ptr=rp, col_idx=ci)
    O2, l2 = oracle.attention_forward(q, k, v, 0.5, block=blk, row_ptr=cp, col_idx=cc)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)
    # doubling every entry changes nothing
    rp2 = (rp * 2).astype(np.int32)
    ci2 = np.concatenate([np.repeat(ci[rp[a]:rp[a + 1]], 2) for a in range(len(rp) - 1)]).astype(np.int32)
    O3, l3 = oracle.attention_forward(q, k, v, 0.5, block=blk, row_ptr=rp2, col_idx=ci2)
    assert np.array_equal(O1, O3) and np.array_equal(l1, l3)


def test_empty_rows_give_zero_output_and_minus_inf_lse():
    L, d, blk = 32, 4, 8
    q, k, v = (_rand((1, 1, L, d), s) for s in (20, 21, 22))
    rp = np.array([0, 1, 1, 3, 3], np.int32)       # rows 1 and 3 empty
    ci = np.array([0, 2, 1], np.int32)
    O, lse = oracle.attention_forward(q, k, v, 0.5, block=blk, row_ptr=rp, col_idx=ci, causal=True)
    for a in (1, 3):
        assert np.all(O[0, 0, a * blk:(a + 1) * blk] == 0)
        assert np.all(lse[0, 0, a * blk:(a + 1) * blk] == -np.inf)
    do = _rand((1, 1, L, d), 23)
    dq, dk, dv, D = oracle.attention_backward(q, k, v, do, 0.5, block=blk, row_ptr=rp,
                                              col_idx=ci, causal=True)
    assert np.all(dq[0, 0, blk:2 * blk] == 0)
    # key block 3 is never listed: no gradient reaches its keys or values
    assert np.all(dk[0, 0, 3 * blk:] == 0) and np.all(dv[0, 0, 3 * blk:] == 0)


def test_causal_offsets_with_empty_leading_rows():
    Lq, Lk, d = 20, 12, 3
    q, k, v = _rand((1, 1, Lq, d), 24), _rand((1, 1, Lk, d), 25), _rand((1, 1, Lk, d), 26)
    O, lse = oracle.attention_forward(q, k, v, 1.0, causal=True, q_offset=0, k_offset=8)
    assert np.all(lse[0, 0, :8] == -np.inf) and np.all(O[0, 0, :8] == 0)
    assert np.isfinite(lse[0, 0, 8:]).all()
    # row 8 sees exactly key 0 (absolute position 8): O = V_0
    assert np.allclose(O[0, 0, 8], v[0, 0, 0], atol=1e-15)


# ---------------------------------------------------------------------------
# Merge of partial states ([EBRS] §2, §4)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_chunked_merge_equals_unchunked_in_any_order(seed):
    rng = np.random.default_rng(100 + seed)
    L, d = 57, 6
    q, k, v = _rand((L, d), 30 + seed), _rand((L, d), 40 + seed) * 3, _rand((L, d), 50 + seed)
    scale = 0.8
    cuts = np.sort(rng.choice(np.arange(1, L), size=3, replace=False))
    bounds = list(zip([0, *cuts], [*cuts, L]))
    states = []
    for s, e in bounds:
        M = oracle.allowed_rows(np.arange(L), e - s, causal=True, k_offset=s)
        states.append(oracle.partial_state(q, k[s:e], v[s:e], scale, M))
    Oref, lref = oracle.attention_forward(q[None, None], k[None, None], v[None, None], scale, causal=True)
    for perm in itertools.permutations(range(len(states))):
        m = np.stack([states[p][0] for p in perm])
        l = np.stack([states[p][1] for p in perm])
        A = np.stack([states[p][2] for p in perm])
        O, lse = oracle.merge_states(m, l, A)
        assert np.allclose(O, Oref[0, 0], atol=1e-12)
        assert np.array_equal(np.isinf(lse), np.isinf(lref[0, 0]))
        fin = np.isfinite(lse)
        assert np.allclose(lse[fin], lref[0, 0][fin], atol=1e-12)
    # pairwise merges associate
    sa, sb, sc = states[0], states[1], states[2]
    left = oracle.merge_pair(oracle.merge_pair(sa, sb), sc)
    right = oracle.merge_pair(sa, oracle.merge_pair(sb, sc))
    for x, y in zip(left, right):
        assert np.allclose(x, y, atol=1e-12)


def test_merge_of_all_empty_states_stays_empty():
    m = np.full((3, 4), -np.inf)
    l = np.zeros((3, 4))
    A = np.zeros((3, 4, 2))
    O, lse = oracle.merge_states(m, l, A)
    assert np.all(O == 0) and np.all(lse == -np.inf)


# ---------------------------------------------------------------------------
# A library routine
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["dense", "causal", "offset", "sparse"])
def test_forward_matches_torch_sdpa(kind):
    Lq, Lk, d, blk = 45, 37, 7, 8
    q, k, v = _rand((Lq, d), 60), _rand((Lk, d), 61), _rand((Lk, 5), 62)
    scale = 0.37
    kw = {}
    if kind == "causal":
        kw = dict(causal=True, q_offset=Lk - Lq + 10)
    if kind == "offset":
        kw = dict(causal=True, q_offset=3, k_offset=1)
    if kind == "sparse":
        rp, ci = random_blocklist((Lq + blk - 1) // blk, (Lk + blk - 1) // blk, seed=63, p_empty=0.0)
        kw = dict(block=blk, row_ptr=rp, col_idx=ci)
    M = oracle.allowed_mask(Lq, Lk, **kw)
    rows = np.nonzero(M.any(axis=1))[0]
    assert len(rows) > 10
    O, lse = oracle.attention_forward(q[None, None], k[None, None], v[None, None], scale, **kw)
    ref = _sdpa(q[rows], k, v, scale, M[rows])
    assert np.allclose(O[0, 0, rows], ref, atol=1e-12)
    assert np.allclose(lse[0, 0, rows], _lse_lib(q[rows], k, scale, M[rows]), atol=1e-12)


@pytest.mark.parametrize("kind", ["dense", "causal", "sparse"])
def test_backward_matches_torch_autograd(kind):
    L, d, blk = 40, 6, 8
    q, k, v, do = (_rand((L, d), s) for s in (70, 71, 72, 73))
    scale = 1 / math.sqrt(d)
    kw = {}
    if kind == "causal":
        kw = dict(causal=True)
    if kind == "sparse":
        rp, ci = random_blocklist(L // blk, L // blk, seed=74, p_empty=0.0)
        kw = dict(block=blk, row_ptr=rp, col_idx=ci, causal=True)
        if not oracle.allowed_mask(L, L, **kw).any(axis=1).all():
            kw["causal"] = False
    M = oracle.allowed_mask(L, L, **kw)
    assert M.any(axis=1).all()
    dq, dk, dv, D = oracle.attention_backward(q[None, None], k[None, None], v[None, None],
                                              do[None, None], scale, **kw)
    tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_() for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None],
        attn_mask=torch.from_numpy(M)[None, None], scale=scale)[0, 0]
    out.backward(torch.from_numpy(do))
    assert np.allclose(dq[0, 0], tq.grad.numpy(), atol=1e-11)
    assert np.allclose(dk[0, 0], tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dv[0, 0], tv.grad.numpy(), atol=1e-11)
    # D_i = dO_i . O_i ([FA] §5.3; [EBRS] §3)
    assert np.allclose(D[0, 0], (do * out.detach().numpy()).sum(axis=1), atol=1e-12)


def test_constant_dP_row_gives_zero_dS():
    """Every V row equal => dP_ij = dO_i . u is constant along j => dS = 0, so
    dQ = dK = 0 ([EBRS] §3, the constant-c example)."""
    L, d = 24, 5
    q, k, do = _rand((L, d), 80), _rand((L, d), 81), _rand((L, d), 82)
    v = np.tile(_rand((1, d), 83), (L, 1))
    M = oracle.allowed_mask(L, L, causal=True)
    dq, dk, dv, D = oracle.backward_head(q, k, v, do, 0.6, M)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    assert np.allclose(D, do @ v[0], atol=1e-13)


# ---------------------------------------------------------------------------
# Brute force on tiny inputs
# ---------------------------------------------------------------------------

def _scalar_attention(q, k, v, scale, M):
    Lq, Lk = len(M), len(M[0])
    O = [[0.0] * len(v[0]) for _ in range(Lq)]
    lse = [-math.inf] * Lq
    for i in range(Lq):
        logits = [scale * sum(q[i][t] * k[j][t] for t in range(len(q[i]))) if M[i][j] else None
                  for j in range(Lk)]
        vis = [x for x in logits if x is not None]
        if not vis:
            continue
        mx = max(vis)
        w = [math.exp(x - mx) if x is not None else 0.0 for x in logits]
        z = sum(w)
        for c in range(len(v[0])):
            O[i][c] = sum(w[j] * v[j][c] for j in range(Lk)) / z
        lse[i] = mx + math.log(z)
    return np.array(O), np.array(lse)


@pytest.mark.parametrize("kind", ["dense", "causal", "sparse", "offset"])
def test_brute_force_tiny_forward(kind):
    Lq, Lk, d, blk = 7, 8, 3, 2
    q, k, v = _rand((Lq, d), 90), _rand((Lk, d), 91), _rand((Lk, 4), 92)
    kw = {}
    if kind == "causal":
        kw = dict(causal=True)
    if kind == "offset":
        kw = dict(causal=True, q_offset=1, k_offset=2)
    if kind == "sparse":
        kw = dict(block=blk, row_ptr=np.array([0, 1, 1, 4, 6], np.int32),
                  col_idx=np.array([0, 3, 1, 3, 2, 2], np.int32))
    M = oracle.allowed_mask(Lq, Lk, **kw)
    O, lse = oracle.attention_forward(q[None, None], k[None, None], v[None, None], 0.8, **kw)
    Ob, lb = _scalar_attention(q.tolist(), k.tolist(), v.tolist(), 0.8, M.tolist())
    assert np.allclose(O[0, 0], Ob, atol=1e-13)
    assert np.array_equal(np.isinf(lse[0, 0]), np.isinf(lb))
    assert np.allclose(lse[0, 0][np.isfinite(lb)], lb[np.isfinite(lb)], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny_gradients_by_finite_differences(causal):
    L, d, h = 6, 3, 1e-6
    q, k, v, do = (_rand((L, d), s) for s in (93, 94, 95, 96))
    M = oracle.allowed_mask(L, L, causal=causal)
    scale = 0.7

    def loss(q_, k_, v_):
        O, _ = _scalar_attention(q_.tolist(), k_.tolist(), v_.tolist(), scale, M.tolist())
        return float((O * do).sum())

    dq, dk, dv, _ = oracle.backward_head(q, k, v, do, scale, M)
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            fp = loss(*args)
            args[which][idx] -= 2 * h
            fm = loss(*args)
            num[idx] = (fp - fm) / (2 * h)
        assert np.allclose(grad, num, atol=1e-7), which


# ---------------------------------------------------------------------------
# Block lists
# ---------------------------------------------------------------------------

def test_blocklist_normalize_sorts_and_dedupes():
    rp = np.array([0, 3, 3, 7], np.int32)
    ci = np.array([2, 0, 2, 1, 1, 3, 0], np.int32)
    p, c = oracle.blocklist_normalize(rp, ci, 4)
    assert p.tolist() == [0, 2, 2, 5]
    assert c.tolist() == [0, 2, 0, 1, 3]


@pytest.mark.parametrize("rp,ci", [
    ([0, 2, 1], [0, 1]),          # decreasing row_ptr
    ([0, 1], [4]),                # index out of range
    ([0, 1], [-1]),               # negative index
    ([0, 3], [0, 1]),             # nnz mismatch
    ([1, 2], [0, 1]),             # does not start at 0
])
def test_blocklist_normalize_rejects_malformed(rp, ci):
    with pytest.raises(ValueError):
        oracle.blocklist_normalize(np.array(rp, np.int32), np.array(ci, np.int32), 4)


def test_local_global_random_pattern_counts():
    """The generator's realised block list: 128 rows, raw entries with
    duplicates, row 64 empty; the realised set is what the oracle uses."""
    rp, ci = local_global_random_blocklist(128, seed=2)
    sets = oracle.blocklist_sets(rp, ci, 128)
    assert len(sets) == 128 and sets[64] == set()
    assert sets[0] == {0} and sets[1] == {0, 1}
    for a, s in enumerate(sets):
        if a != 64:
            assert set(range(max(0, a - 3), a + 1)) | {0} <= s
            assert max(s) == a
    raw, uniq = len(ci), sum(len(s) for s in sets)
    assert raw > uniq     # duplicates present in the raw list
    assert 800 < uniq < 900 and 850 < raw < 900


# ---------------------------------------------------------------------------
# Grouped key/value heads ([EBRS] §6: query heads sharing one KV head)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,Hkv", [(4, 2), (6, 1), (3, 3)])
def test_grouped_heads_match_torch_sdpa_with_gqa(H, Hkv):
    """Library routine: torch SDPA with enable_gqa (query head h reads KV head
    h // (H / H_kv)), forward and autograd gradients; the shared head's dK/dV
    is the sum over its query heads."""
    B, L, d = 2, 33, 5
    q, do = _rand((B, H, L, d), 100), _rand((B, H, L, d), 101)
    k, v = _rand((B, Hkv, L, d), 102), _rand((B, Hkv, L, d), 103)
    scale = 0.45
    M = oracle.allowed_mask(L, L, causal=True)
    O, lse = oracle.attention_forward(q, k, v, scale, causal=True)
    dq, dk, dv, D = oracle.attention_backward(q, k, v, do, scale, causal=True)
    tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_() for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=torch.from_numpy(M), scale=scale, enable_gqa=True)
    out.backward(torch.from_numpy(do))
    assert np.allclose(O, out.detach().numpy(), atol=1e-12)
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-11)
    G = H // Hkv
    for b, h in itertools.product(range(B), range(H)):
        assert np.allclose(lse[b, h], _lse_lib(q[b, h], k[b, h // G], scale, M), atol=1e-12)


def test_grouped_heads_gradient_by_finite_differences():
    """Brute force: a shared key/value head perturbed once moves the outputs of
    every query head of its group, so its gradient is the group's sum."""
    B, H, Hkv, L, d, h = 1, 2, 1, 5, 2, 1e-6
    q, do = _rand((B, H, L, d), 110), _rand((B, H, L, d), 111)
    k, v = _rand((B, Hkv, L, d), 112), _rand((B, Hkv, L, d), 113)
    M = oracle.allowed_mask(L, L, causal=True).tolist()
    scale = 0.9

    def loss(k_, v_):
        tot = 0.0
        for hq in range(H):
            O, _ = _scalar_attention(q[0, hq].tolist(), k_[0, 0].tolist(), v_[0, 0].tolist(),
                                     scale, M)
            tot += float((O * do[0, hq]).sum())
        return tot

    _, dk, dv, _ = oracle.attention_backward(q, k, v, do, scale, causal=True)
    for arr, grad, which in ((k, dk, 0), (v, dv, 1)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = [k.copy(), v.copy()]
            args[which][idx] += h
            fp = loss(*args)
            args[which][idx] -= 2 * h
            fm = loss(*args)
            num[idx] = (fp - fm) / (2 * h)
        assert np.allclose(grad, num, atol=1e-7), which


def test_kv_heads_must_divide_query_heads():
    with pytest.raises(ValueError):
        oracle.kv_group(6, 4)
    with pytest.raises(ValueError):
        oracle.kv_group(2, 0)
