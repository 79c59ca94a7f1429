"""Block-sparse forward and backward with several block lists (attn_fwd_blocksparse
and attn_bwd_blocksparse with n_lists > 1): lists shared by consecutive groups of
heads, one per head and one per batch, each head checked against the oracle
with its own list, and a multi-list launch against per-list single launches."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import TOL_GRAD, compare_forward, oracle_forward, to_cuda
from workloads import Workload, make_inputs, random_blocklist, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


def stacked_lists(n_lists, n, seed):
    """n_lists raw CSR lists as one [n_lists, n+1] row_ptr (offsets into one
    col_idx) plus the individual lists."""
    lists = [random_blocklist(n, n, seed=seed + 17 * x, max_per_row=5, p_empty=0.1)
             for x in range(n_lists)]
    rps, cis, off = [], [], 0
    for rp, ci in lists:
        rps.append(rp + off)
        cis.append(ci)
        off += len(ci)
    return np.stack(rps).astype(np.int32), np.concatenate(cis).astype(np.int32), lists


@pytest.mark.parametrize("per", ["head", "batch"])
@pytest.mark.parametrize("causal", [True, False])
def test_lists_forward_and_backward_match_oracle(bss, per, causal):
    B, H, L, d = 2, 3, 900, 64
    n = (L + 127) // 128
    n_lists = B * H if per == "head" else B
    hpl = B * H // n_lists
    rp, ci, lists = stacked_lists(n_lists, n, seed=5 if causal else 6)
    w = Workload("ml", B, H, L, d, causal, seed=95, backward=True)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal,
                                      scale=w.scale)
    dq, dk, dv, _ = bss.attn_bwd_blocksparse(inp["q"], inp["k"], inp["v"], o, lse, inp["do"],
                                             rp, ci, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    q, k, v, do = (to_f64(cpu[x]) for x in ("q", "k", "v", "do"))
    for b in range(B):
        for h in range(H):
            lrp, lci = lists[(b * H + h) // hpl]
            kw = dict(causal=causal, block=128, row_ptr=lrp, col_idx=lci)
            O_ref, l_ref = oracle_forward(cpu, w.scale, heads=[(b, h)], **kw)
            compare_forward(o[b, h], lse[b, h], O_ref[0], l_ref[0], f"head {(b, h)}")
            gq, gk, gv, _ = oracle.attention_backward(q, k, v, do, w.scale, heads=[(b, h)], **kw)
            for name, g, r in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
                err = np.abs(g[b, h].double().cpu().numpy() - r[0]).max()
                assert err <= TOL_GRAD, f"head {(b, h)}: max|d{name}| = {err:.3e}"


def test_one_launch_equals_per_list_launches(bss):
    """Lists per batch in one launch give the same bits as one launch per batch
    with that batch's list alone."""
    B, H, L, d = 3, 2, 700, 128
    n = (L + 127) // 128
    rp, ci, lists = stacked_lists(B, n, seed=21)
    w = Workload("ml1", B, H, L, d, True, seed=96, backward=True)
    inp = to_cuda(make_inputs(w))
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True)
    dq, dk, dv, _ = bss.attn_bwd_blocksparse(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], rp,
                                             ci, causal=True)
    for b in range(B):
        x = {n_: t[b:b + 1].contiguous() for n_, t in inp.items()}
        ob, lb = bss.attn_fwd_blocksparse(x["q"], x["k"], x["v"], *lists[b], causal=True)
        _, dkb, dvb, _ = bss.attn_bwd_blocksparse(x["q"], x["k"], x["v"], ob, lb, x["do"],
                                                  *lists[b], causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o[b], ob[0]) and torch.equal(lse[b], lb[0])
        assert torch.equal(dk[b], dkb[0]) and torch.equal(dv[b], dvb[0])


def test_list_count_must_divide_heads(bss):
    B, H, L, d = 2, 3, 256, 64
    w = Workload("mlx", B, H, L, d, True, seed=97)
    inp = to_cuda(make_inputs(w))
    rp, ci, _ = stacked_lists(4, 2, seed=1)
    with pytest.raises(bss.AttnError):
        bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True)
