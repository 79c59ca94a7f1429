"""Block-sparse backward parity on the GPU (attn_bwd_blocksparse through the C
ABI): gradients over the kept blocks only, with the local + global + random
pattern (duplicates, an empty query block, a partial last block), unstructured
lists, set semantics, key blocks no query block lists, equivalence with the
dense backward when every block is listed, bad entries reported, and the
B=2 H=16 L=16320 d=128 workload checked on sampled key blocks and rows."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import TOL_GRAD, TOL_LSE, TOL_O, to_cuda
from workloads import (SPARSE_16K, Workload, local_global_random_blocklist, make_inputs,
                       random_blocklist, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


def _fwd_bwd(bss, inp, rp, ci, causal, scale):
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal,
                                      scale=scale)
    dq, dk, dv, delta = bss.attn_bwd_blocksparse(inp["q"], inp["k"], inp["v"], o, lse, inp["do"],
                                                 rp, ci, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv, delta


def _check_grads(got, ref, what):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        gn = g.double().cpu().numpy()
        assert np.isfinite(gn).all(), f"{what}: {name} not finite"
        err = np.abs(gn - r).max()
        assert err <= TOL_GRAD, f"{what}: max|d{name}| = {err:.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_local_global_random_pattern_gradients(bss, d, causal):
    L = 2048 - 64                                   # 16 blocks, the last one half full
    n = (L + 127) // 128
    rp, ci = local_global_random_blocklist(n, seed=2)
    w = Workload("sb", 1, 2, L, d, causal, seed=70 + d, backward=True)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    _, _, dq, dk, dv, _ = _fwd_bwd(bss, inp, rp, ci, causal, w.scale)
    assert bss.attn_poll_status() == 0
    q, k, v, do = (to_f64(cpu[x]) for x in ("q", "k", "v", "do"))
    ref = oracle.attention_backward(q, k, v, do, w.scale, causal=causal, block=128, row_ptr=rp,
                                    col_idx=ci)
    _check_grads((dq, dk, dv), ref[:3], f"pattern d={d} causal={causal}")
    # the emptied query block has no allowed pair: its dQ is exactly zero
    e = n // 2
    assert torch.all(dq[:, :, e * 128:(e + 1) * 128] == 0)


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_unstructured_lists_gradients(bss, seed):
    L, d = 1000, 64 if seed % 2 else 128
    n = (L + 127) // 128
    rp, ci = random_blocklist(n, n, seed=seed, max_per_row=5, p_empty=0.15)
    causal = seed <= 2
    w = Workload("su", 2, 1, L, d, causal, seed=80 + seed, backward=True)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    _, _, dq, dk, dv, _ = _fwd_bwd(bss, inp, rp, ci, causal, w.scale)
    assert bss.attn_poll_status() == 0
    q, k, v, do = (to_f64(cpu[x]) for x in ("q", "k", "v", "do"))
    ref = oracle.attention_backward(q, k, v, do, w.scale, causal=causal, block=128, row_ptr=rp,
                                    col_idx=ci)
    _check_grads((dq, dk, dv), ref[:3], f"random list seed={seed}")


def test_unlisted_key_blocks_get_zero_gradients(bss):
    """Key blocks 2 and 5 appear in no list: their dK and dV rows are exactly 0."""
    L, d = 900, 128
    n = (L + 127) // 128                            # 8 blocks
    lists = [[0], [0, 1], [1, 0, 1], [3], [3, 4], [4, 3], [6, 0], [7, 6]]
    rp = np.cumsum([0] + [len(x) for x in lists]).astype(np.int32)
    ci = np.array([c for x in lists for c in x], np.int32)
    w = Workload("sz", 1, 2, L, d, True, seed=91, backward=True)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    _, _, dq, dk, dv, _ = _fwd_bwd(bss, inp, rp, ci, True, w.scale)
    assert bss.attn_poll_status() == 0
    for j in (2, 5):
        assert torch.all(dk[:, :, j * 128:(j + 1) * 128] == 0)
        assert torch.all(dv[:, :, j * 128:(j + 1) * 128] == 0)
    q, k, v, do = (to_f64(cpu[x]) for x in ("q", "k", "v", "do"))
    ref = oracle.attention_backward(q, k, v, do, w.scale, causal=True, block=128, row_ptr=rp,
                                    col_idx=ci)
    _check_grads((dq, dk, dv), ref[:3], "unlisted key blocks")


def test_every_block_listed_equals_dense_backward(bss):
    """With every block listed the sparse walk visits the dense causal tiles in
    the same order: given the same O and LSE, dK, dV and D are identical to
    attn_bwd's; dQ (added in by reduce operations whose order is not fixed)
    agrees within the tolerance.  The two forwards agree within the tolerance:
    at d=128 the dense one scores pairs of key blocks (its reference max moves
    per pair), so their roundings differ."""
    L, d = 1100, 128
    n = (L + 127) // 128
    rp = (np.arange(n + 1) * n).astype(np.int32)
    ci = np.tile(np.arange(n, dtype=np.int32), n)
    w = Workload("sd", 1, 3, L, d, True, seed=92, backward=True)
    inp = to_cuda(make_inputs(w))
    o, lse, dq, dk, dv, delta = _fwd_bwd(bss, inp, rp, ci, True, w.scale)
    o2, lse2 = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale)
    ref = bss.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True,
                       scale=w.scale)
    torch.cuda.synchronize()
    assert (o.float() - o2.float()).abs().max().item() <= TOL_O
    assert (lse - lse2).abs().max().item() <= TOL_LSE
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]) and torch.equal(delta, ref[3])
    assert (dq.float() - ref[0].float()).abs().max().item() <= TOL_GRAD


def test_order_and_duplicates_do_not_change_gradients(bss):
    L, d = 1500, 64
    n = (L + 127) // 128
    rp, ci = random_blocklist(n, n, seed=19, max_per_row=6, p_empty=0.1)
    cp, cc = bss.attn_blocklist_normalize(rp, ci, n)
    rng = np.random.default_rng(1)
    perm_ci = np.concatenate([rng.permutation(np.repeat(cc[cp[a]:cp[a + 1]], 2))
                              for a in range(n)]).astype(np.int32)
    perm_rp = (cp * 2).astype(np.int32)
    w = Workload("sp", 1, 2, L, d, True, seed=93, backward=True)
    inp = to_cuda(make_inputs(w))
    runs = [_fwd_bwd(bss, inp, a, b, True, w.scale) for a, b in ((rp, ci), (cp, cc),
                                                                  (perm_rp, perm_ci))]
    for r in runs[1:]:
        assert torch.equal(r[3], runs[0][3]) and torch.equal(r[4], runs[0][4])   # dk, dv
        assert (r[2].float() - runs[0][2].float()).abs().max().item() <= 1e-2    # dq


def test_bad_entry_is_reported(bss):
    L, d = 512, 64
    n = 4
    rp = np.array([0, 1, 3, 4, 6], np.int32)
    ci = np.array([0, 1, 99, 2, 3, 1], np.int32)     # 99 is out of range
    w = Workload("se", 1, 1, L, d, True, seed=94, backward=True)
    inp = to_cuda(make_inputs(w))
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True)
    bss.attn_poll_status()
    bss.attn_bwd_blocksparse(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], rp, ci, causal=True)
    assert bss.attn_poll_status() == bss.ERR_BAD_BLOCKLIST


def _sampled_reference(q, k, v, do, scale, rp, ci, n, L, key_blocks):
    """Oracle gradients for whole key blocks of one head.  dK_j and dV_j depend
    only on the query rows whose lists hold block j, and those rows' dQ only on
    their own allowed keys, so the oracle's backward over that sub-problem (the
    rows, and every key any of them may see) is exact for them."""
    sets = oracle.blocklist_sets(rp, ci, n)
    out = []
    for j in key_blocks:
        qb = [a for a in range(n) if j in sets[a] and j <= a]
        rows = np.concatenate([np.arange(a * 128, min((a + 1) * 128, L)) for a in qb])
        kb = sorted(set().union(*(sets[a] for a in qb)))
        keys = np.concatenate([np.arange(c * 128, min((c + 1) * 128, L)) for c in kb])
        M = oracle.allowed_rows(rows, L, causal=True, block=128, row_ptr=rp, col_idx=ci)[:, keys]
        gq, gk, gv, _ = oracle.backward_head(q[rows], k[keys], v[keys], do[rows], scale, M)
        sel = np.searchsorted(keys, np.arange(j * 128, min((j + 1) * 128, L)))
        out.append((j, rows, gq, gk[sel], gv[sel]))
    return out


def test_sparse_16k_full_size_sampled(bss):
    """B=2 H=16 L=16320 d=128 causal with the local + global + random lists
    (the block-sparse benchmark's launch configuration): every gradient finite,
    emptied query block's dQ exactly 0, and for two heads the oracle on whole
    key blocks (their dK, dV and the dQ rows that see them)."""
    w = Workload(SPARSE_16K.name, SPARSE_16K.B, SPARSE_16K.H, SPARSE_16K.L, SPARSE_16K.d, True,
                 SPARSE_16K.seed, backward=True)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    n = (w.L + 127) // 128
    rp, ci = local_global_random_blocklist(n, seed=2)
    _, _, dq, dk, dv, _ = _fwd_bwd(bss, inp, rp, ci, True, w.scale)
    assert bss.attn_poll_status() == 0
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    e = n // 2
    assert torch.all(dq[:, :, e * 128:(e + 1) * 128] == 0)
    for b, h in ((0, 3), (1, 15)):
        q, k, v, do = (to_f64(cpu[x][b:b + 1, h:h + 1])[0, 0] for x in ("q", "k", "v", "do"))
        for j, rows, gq, gk, gv in _sampled_reference(q, k, v, do, w.scale, rp, ci, n, w.L,
                                                       key_blocks=(60, 100, n - 1)):
            sl = slice(j * 128, min((j + 1) * 128, w.L))
            assert np.abs(dk[b, h, sl].double().cpu().numpy() - gk).max() <= TOL_GRAD
            assert np.abs(dv[b, h, sl].double().cpu().numpy() - gv).max() <= TOL_GRAD
            assert np.abs(dq[b, h, rows].double().cpu().numpy() - gq).max() <= TOL_GRAD


def _global_at(n, g, seed):
    """Raw CSR of the local + global + random pattern with the global block at
    g instead of 0 (rows before g list it too: under a causal mask it lies in
    their future and contributes nothing)."""
    rng = np.random.default_rng(seed)
    rows = []
    for a in range(n):
        row = [a - t for t in range(4) if a - t >= 0] + [g]
        if a >= 1:
            row += [int(rng.integers(0, a)) for _ in range(2)]
        rows.append(row)
    rp = np.zeros(n + 1, np.int32)
    for a, r in enumerate(rows):
        rp[a + 1] = rp[a] + len(r)
    return rp, np.array([c for r in rows for c in r], np.int32)


def test_long_columns_first_with_per_group_lists(bss):
    """Lists per K/V head whose global block (listed by every row) differs, so
    that each list has one key column far longer than the mean: the backward
    launches those key tiles first.  B=1, H=4 query heads over 2 K/V heads,
    L=4096 (32 blocks), causal, d=64; every gradient against the oracle with
    each head's own list, dK and dV summed over the heads of a group."""
    L, d, H, Hkv = 4096, 64, 4, 2
    n = L // 128
    lists = [_global_at(n, 0, seed=5), _global_at(n, 9, seed=6)]
    rp = np.zeros((2, n + 1), np.int32)
    rp[0] = lists[0][0]
    rp[1] = lists[1][0] + len(lists[0][1])
    ci = np.concatenate([lists[0][1], lists[1][1]]).astype(np.int32)
    w = Workload("lc", 1, H, L, d, True, seed=77, backward=True, Hkv=Hkv)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    _, _, dq, dk, dv, _ = _fwd_bwd(bss, inp, rp, ci, True, w.scale)
    stats = bss.attn_blocklist_stats(rp, ci, L, causal=True).cpu().tolist()
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    for li, (r, c) in enumerate(lists):
        s = oracle.blocklist_stats(r, c, L, causal=True)
        assert stats[li] == [s["listed"], s["executed"], s["future"], s["pairs"]]
    assert stats[1][2] == 9                       # rows 0..8 list the future block 9
    q, k, v, do = (to_f64(cpu[x]) for x in ("q", "k", "v", "do"))
    G = H // Hkv
    dk_ref = np.zeros_like(k)
    dv_ref = np.zeros_like(v)
    for h in range(H):
        r, c = lists[h // G]
        M = oracle.allowed_mask(L, L, causal=True, block=128, row_ptr=r, col_idx=c)
        gq, gk, gv, _ = oracle.backward_head(q[0, h], k[0, h // G], v[0, h // G], do[0, h],
                                             w.scale, M)
        err = np.abs(dq[0, h].double().cpu().numpy() - gq).max()
        assert err <= TOL_GRAD, f"head {h}: max|ddq| = {err:.3e}"
        dk_ref[0, h // G] += gk
        dv_ref[0, h // G] += gv
    for name, g, ref in (("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        err = np.abs(g.double().cpu().numpy() - ref).max()
        assert err <= TOL_GRAD, f"max|d{name}| = {err:.3e}"
