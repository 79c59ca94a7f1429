"""Grouped key/value heads on the GPU (H_kv < H through the C ABI): query head h
reads key/value head h // (H / H_kv) in the dense, causal, split-KV and
block-sparse forwards and in both backwards, whose dK/dV of a shared head add
the gradients of its query heads; block lists shared by a KV head's query heads
and the mean-pooled selector over grouped heads.  Every case against the oracle
on the same seeded inputs; the forward also against the same kernel run on
K/V repeated per query head (bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import select as sel
from tests.parity import TOL_GRAD, compare_forward, oracle_forward, to_cuda
from workloads import Workload, make_inputs, random_blocklist, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


def gqa_inputs(w: Workload, Hkv: int):
    """q (and do) with w.H heads, k and v with Hkv heads, drawn in that order."""
    return make_inputs(w, Hkv=Hkv)


def _repeat(t, G):
    return t.repeat_interleave(G, dim=1).contiguous()


def _check_grads(got, ref, what, names=("dq", "dk", "dv")):
    for name, g, r in zip(names, got, ref):
        gn = g.double().cpu().numpy()
        assert np.isfinite(gn).all(), f"{what}: {name} not finite"
        err = np.abs(gn - r).max()
        assert err <= TOL_GRAD, f"{what}: max|{name}| = {err:.3e}"


@pytest.mark.parametrize("B,H,Hkv,L,d,causal", [
    (1, 4, 2, 1000, 128, True),
    (2, 8, 1, 700, 64, True),        # one KV head for every query head
    (1, 6, 3, 1300, 64, False),
    (2, 4, 4, 384, 128, True),       # H_kv = H: plain multi-head
])
def test_forward_matches_oracle_and_repeated_kv(bss, B, H, Hkv, L, d, causal):
    w = Workload("gf", B, H, L, d, causal, seed=L + H + Hkv)
    cpu = gqa_inputs(w, Hkv)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=causal, scale=w.scale)
    G = H // Hkv
    o_r, lse_r = bss.attn_fwd(inp["q"], _repeat(inp["k"], G), _repeat(inp["v"], G),
                              causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.equal(o, o_r) and torch.equal(lse, lse_r)
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=causal)
    compare_forward(o, lse, O_ref, l_ref, f"gqa H={H} Hkv={Hkv}")


@pytest.mark.parametrize("B,H,Hkv,Lq,Lk,d,chunks", [
    (2, 8, 2, 16, 3000, 128, 8),      # decode-shaped
    (1, 4, 1, 300, 1100, 64, 3),
])
def test_splitkv_matches_oracle(bss, B, H, Hkv, Lq, Lk, d, chunks):
    w = Workload("gs", B, H, Lk, d, True, seed=Lq + Lk, Lq=Lq)
    cpu = gqa_inputs(w, Hkv)
    inp = to_cuda(cpu)
    q_off = Lk - Lq
    o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], chunks, causal=True,
                                  scale=w.scale, q_offset=q_off)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=True, q_offset=q_off)
    compare_forward(o, lse, O_ref, l_ref, f"gqa splitkv H={H} Hkv={Hkv}")


@pytest.mark.parametrize("B,H,Hkv,L,d,causal", [
    (1, 4, 2, 1000, 128, True),
    (2, 4, 1, 640, 64, False),
    (1, 8, 2, 1500, 64, True),
])
def test_backward_sums_the_group_gradients(bss, B, H, Hkv, L, d, causal):
    w = Workload("gb", B, H, L, d, causal, seed=3 * L + Hkv, backward=True)
    cpu = gqa_inputs(w, Hkv)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=causal, scale=w.scale)
    dq, dk, dv, delta = bss.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"],
                                     causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert dk.shape == inp["k"].shape and dv.shape == inp["v"].shape
    q, k, v, do = (to_f64(cpu[x]) for x in ("q", "k", "v", "do"))
    ref = oracle.attention_backward(q, k, v, do, w.scale, causal=causal)
    _check_grads((dq, dk, dv), ref[:3], f"gqa bwd H={H} Hkv={Hkv}")
    # delta is D_i = dO_i . O_i from the saved bf16 O, near the oracle's fp64 D
    d_def = (o.double() * inp["do"].double()).sum(-1).cpu().numpy()
    assert np.abs(delta.double().cpu().numpy() - d_def).max() <= 1e-3
    assert np.abs(delta.double().cpu().numpy() - ref[3]).max() <= TOL_GRAD


def _group_lists(n_lists, n, seed):
    lists = [random_blocklist(n, n, seed=seed + 13 * x, max_per_row=5, p_empty=0.1)
             for x in range(n_lists)]
    rps, cis, off = [], [], 0
    for rp, ci in lists:
        rps.append(rp + off)
        cis.append(ci)
        off += len(ci)
    return np.stack(rps).astype(np.int32), np.concatenate(cis).astype(np.int32), lists


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("per", ["kv_head", "batch"])
def test_blocksparse_lists_per_kv_head(bss, causal, per):
    """One list per KV head (shared by its G query heads) or per batch entry:
    forward and backward against the oracle, list by list."""
    B, H, Hkv, L, d = 2, 4, 2, 900, 64
    G = H // Hkv
    n = (L + 127) // 128
    n_lists = B * Hkv if per == "kv_head" else B
    hpl = B * H // n_lists
    rp, ci, lists = _group_lists(n_lists, n, seed=7 if causal else 8)
    w = Workload("gl", B, H, L, d, causal, seed=96, backward=True)
    cpu = gqa_inputs(w, Hkv)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal,
                                      scale=w.scale)
    dq, dk, dv, _ = bss.attn_bwd_blocksparse(inp["q"], inp["k"], inp["v"], o, lse, inp["do"],
                                             rp, ci, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    q, k, v, do = (to_f64(cpu[x]) for x in ("q", "k", "v", "do"))
    dk_ref = np.zeros_like(k)
    dv_ref = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            lrp, lci = lists[(b * H + h) // hpl]
            kw = dict(causal=causal, block=128, row_ptr=lrp, col_idx=lci)
            O_ref, l_ref = oracle_forward(cpu, w.scale, heads=[(b, h)], **kw)
            compare_forward(o[b, h], lse[b, h], O_ref[0], l_ref[0], f"head {(b, h)}")
            gq, gk, gv, _ = oracle.attention_backward(q, k, v, do, w.scale, heads=[(b, h)], **kw)
            err = np.abs(dq[b, h].double().cpu().numpy() - gq[0]).max()
            assert err <= TOL_GRAD, f"dq head {(b, h)}: {err:.3e}"
            dk_ref[b, h // G] += gk[0]
            dv_ref[b, h // G] += gv[0]
    _check_grads((dk, dv), (dk_ref, dv_ref), f"gqa sparse per={per}", ("dk", "dv"))


def test_per_query_head_lists_forward_only(bss):
    """Lists per query head are fine for the forward; the backward, which walks a
    KV head's query heads with one list, rejects lists that split a group."""
    B, H, Hkv, L, d = 1, 4, 2, 700, 128
    n = (L + 127) // 128
    rp, ci, lists = _group_lists(B * H, n, seed=9)
    w = Workload("gq", B, H, L, d, True, seed=97, backward=True)
    cpu = gqa_inputs(w, Hkv)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    for h in range(H):
        lrp, lci = lists[h]
        O_ref, l_ref = oracle_forward(cpu, w.scale, heads=[(0, h)], causal=True, block=128,
                                      row_ptr=lrp, col_idx=lci)
        compare_forward(o[0, h], lse[0, h], O_ref[0], l_ref[0], f"head {h}")
    with pytest.raises(bss.AttnError):
        bss.attn_bwd_blocksparse(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], rp, ci,
                                 causal=True, scale=w.scale)


@pytest.mark.parametrize("causal", [True, False])
def test_selector_over_grouped_heads(bss, causal):
    """Lists per KV head from the mean-pooled scores of its query heads against
    the shared keys, then the sparse forward and backward on them."""
    B, H, Hkv, L, d = 2, 4, 2, 1400, 128
    G = H // Hkv
    w = Workload("gsel", B, H, L, d, causal, seed=98, backward=True)
    cpu = gqa_inputs(w, Hkv)
    inp = to_cuda(cpu)
    n_lists = B * Hkv
    rp, ci = bss.attn_select_blocks(inp["q"], inp["k"], 3, local_blocks=2, causal=causal,
                                    n_lists=n_lists, scale=w.scale)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal,
                                      scale=w.scale)
    dq, dk, dv, _ = bss.attn_bwd_blocksparse(inp["q"], inp["k"], inp["v"], o, lse, inp["do"],
                                             rp, ci, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    # the selection, against the oracle's (grouped heads pool their shared key head)
    q32, k32 = (cpu[x].float().numpy() for x in ("q", "k"))
    rp_o, ci_o, lists_o = sel.select_blocks(q32, k32, w.scale, top_r=3, local=2, causal=causal,
                                            n_lists=n_lists)
    assert np.array_equal(rp.cpu().numpy(), rp_o)
    got = ci.cpu().numpy()
    if not np.array_equal(got, ci_o):
        # only near-ties may differ: compare the pooled score of what each side kept
        n = rp_o.shape[1] - 1
        q64, k64 = to_f64(cpu["q"]), to_f64(cpu["k"])
        for lst in range(n_lists):
            b, kh = divmod(lst, Hkv)
            S = sum(sel.pooled_scores(q64[b, kh * G + x], k64[b, kh], w.scale, dtype=np.float64)
                    for x in range(G))
            for a in range(n):
                g = set(got[rp_o[lst, a]:rp_o[lst, a + 1]])
                o_ = set(lists_o[lst][a])
                for cg, co in zip(sorted(g - o_, key=lambda c: -S[a, c]),
                                  sorted(o_ - g, key=lambda c: -S[a, c])):
                    assert abs(S[a, cg] - S[a, co]) <= 1e-4 * (1 + abs(S[a, co]))
    # the sparse forward and backward on the GPU's own lists
    rp_h, ci_h = rp.cpu().numpy(), got
    q, k, v, do = (to_f64(cpu[x]) for x in ("q", "k", "v", "do"))
    dk_ref = np.zeros_like(k)
    dv_ref = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            lst = b * Hkv + h // G
            lrp = rp_h[lst] - rp_h[lst, 0]
            lci = ci_h[rp_h[lst, 0]:rp_h[lst, -1]]
            kw = dict(causal=causal, block=128, row_ptr=lrp, col_idx=lci)
            O_ref, l_ref = oracle_forward(cpu, w.scale, heads=[(b, h)], **kw)
            compare_forward(o[b, h], lse[b, h], O_ref[0], l_ref[0], f"head {(b, h)}")
            gq, gk, gv, _ = oracle.attention_backward(q, k, v, do, w.scale, heads=[(b, h)], **kw)
            assert np.abs(dq[b, h].double().cpu().numpy() - gq[0]).max() <= TOL_GRAD
            dk_ref[b, h // G] += gk[0]
            dv_ref[b, h // G] += gv[0]
    _check_grads((dk, dv), (dk_ref, dv_ref), "gqa selected lists", ("dk", "dv"))
