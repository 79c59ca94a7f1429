"""Mean-pooled block selector on the GPU (attn_select_blocks through the C ABI):
the lists against the oracle's selection (row offsets exactly; rows exactly up
to the order of candidates whose pooled scores tie within float32 rounding),
lists shared by head groups, and the selected lists driving the block-sparse
forward against the oracle, up to the L=16320 block-sparse workload."""
import numpy as np
import pytest
import torch

from oracle import select as sel
from tests.parity import compare_forward, oracle_forward, to_cuda
from workloads import SPARSE_16K, Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


def _list_scores(q64, k64, scale, lst, hpl, H):
    """Pooled scores of one list in float64 (sum over its heads)."""
    S = None
    for x in range(lst * hpl, (lst + 1) * hpl):
        b, h = divmod(x, H)
        s = sel.pooled_scores(q64[b, h], k64[b, h], scale, dtype=np.float64)
        S = s if S is None else S + s
    return S


def check_lists(rp_gpu, ci_gpu, cpu, scale, top_r, local, causal, n_lists):
    """GPU lists against the oracle's: row offsets exactly; each row exactly, or
    differing only in candidates whose float64 scores tie within 1e-4."""
    q32, k32 = (cpu[n].float().numpy() for n in ("q", "k"))
    rp_o, ci_o, lists_o = sel.select_blocks(q32, k32, scale, top_r=top_r, local=local,
                                            causal=causal, n_lists=n_lists)
    rp_g = rp_gpu.cpu().numpy()
    ci_g = ci_gpu.cpu().numpy()
    assert np.array_equal(rp_g, rp_o)
    B, H = q32.shape[:2]
    hpl = B * H // n_lists
    q64, k64 = (to_f64(cpu[n]) for n in ("q", "k"))
    n = rp_o.shape[1] - 1
    for lst in range(n_lists):
        S = None
        for a in range(n):
            got = list(ci_g[rp_g[lst, a]:rp_g[lst, a + 1]])
            want = lists_o[lst][a]
            assert got == sorted(set(got))
            if got == want:
                continue
            S = _list_scores(q64, k64, scale, lst, hpl, H) if S is None else S
            only_g = sorted(set(got) - set(want), key=lambda c: -S[a, c])
            only_o = sorted(set(want) - set(got), key=lambda c: -S[a, c])
            assert len(only_g) == len(only_o)
            for cg, co in zip(only_g, only_o):
                assert abs(S[a, cg] - S[a, co]) <= 1e-4 * (1 + abs(S[a, co])), (lst, a, cg, co)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,L,d,top_r,local,per_head", [
    (1, 2, 1000, 64, 2, 1, True),
    (2, 2, 2048, 128, 5, 3, False),
    (1, 3, 700, 128, 0, 2, True),          # window only
    (1, 1, 900, 64, 9, 0, True),           # more picks asked than candidates
])
def test_lists_match_oracle(bss, causal, B, H, L, d, top_r, local, per_head):
    w = Workload("sel", B, H, L, d, causal, seed=L + top_r)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    n_lists = B * H if per_head else 1
    rp, ci = bss.attn_select_blocks(inp["q"], inp["k"], top_r, local_blocks=local, causal=causal,
                                    n_lists=n_lists, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    check_lists(rp, ci, cpu, w.scale, top_r, local, causal, n_lists)


@pytest.mark.parametrize("n_lists", [1, 2, 4])
def test_selected_lists_drive_the_sparse_forward(bss, n_lists):
    B, H, L, d = 2, 2, 1500, 128
    w = Workload("sfw", B, H, L, d, True, seed=33 + n_lists)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    rp, ci = bss.attn_select_blocks(inp["q"], inp["k"], 3, local_blocks=2, causal=True,
                                    n_lists=n_lists, scale=w.scale)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    check_lists(rp, ci, cpu, w.scale, 3, 2, True, n_lists)
    rp_h, ci_h = rp.cpu().numpy(), ci.cpu().numpy()
    hpl = B * H // n_lists
    for b in range(B):
        for h in range(H):
            lst = (b * H + h) // hpl
            lrp = rp_h[lst] - rp_h[lst, 0]
            lci = ci_h[rp_h[lst, 0]:rp_h[lst, -1]]
            O_ref, l_ref = oracle_forward(cpu, w.scale, heads=[(b, h)], causal=True, block=128,
                                          row_ptr=lrp, col_idx=lci)
            compare_forward(o[b, h], lse[b, h], O_ref[0], l_ref[0], f"head {(b, h)}")


def test_sparse_16k_workload_selection(bss):
    """B=2 H=16 L=16320 d=128: per-head lists of the 4 local and 4 best-scoring
    blocks, against the oracle's selection; the sparse forward on them runs clean."""
    w = SPARSE_16K
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    n_lists = w.B * w.H
    rp, ci = bss.attn_select_blocks(inp["q"], inp["k"], 4, local_blocks=4, causal=True,
                                    n_lists=n_lists, scale=w.scale)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    check_lists(rp, ci, cpu, w.scale, 4, 4, True, n_lists)
