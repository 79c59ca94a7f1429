"""Block-sparse forward, backward and list accounting at the largest key range
the library addresses: 4096 key blocks of 128 (L = 524288), so that the
bitmaps of the forward, the key-major columns of the backward and the
accounting kernel's per-warp bitmaps use every word up to the last.  One head,
d=64, causal, with the local + global + random list (duplicates, the empty
middle row); the oracle on sampled rows and on whole sampled key blocks
("Exact Blocks, Rings, and Sparsity", section 5; block-sparse attention
patterns page, 'Count active blocks and acknowledge the changed operator')."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import TOL_GRAD, compare_forward, oracle_forward, to_cuda
from tests.test_gpu_sparse_bwd import _sampled_reference
from workloads import Workload, local_global_random_blocklist, make_inputs, to_f64

pytestmark = pytest.mark.gpu

N_MAX = 4096                    # key blocks a launch can address
L_MAX = N_MAX * 128


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


@pytest.fixture(scope="module")
def case():
    w = Workload("sparse_max", 1, 1, L_MAX, 64, True, seed=13, backward=True)
    cpu = make_inputs(w)
    rp, ci = local_global_random_blocklist(N_MAX, seed=13)
    return w, cpu, rp, ci


def test_forward_and_backward_at_the_largest_key_range(bss, case):
    w, cpu, rp, ci = case
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    dq, dk, dv, _ = bss.attn_bwd_blocksparse(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], rp,
                                             ci, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    e = N_MAX // 2                                  # the emptied query block
    assert torch.all(torch.isneginf(lse[0, 0, e * 128:(e + 1) * 128]))
    assert torch.all(o[0, 0, e * 128:(e + 1) * 128] == 0)
    assert torch.all(dq[0, 0, e * 128:(e + 1) * 128] == 0)
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t).all()
    # forward: rows in the first, middle and last query blocks (the last rows
    # scan every bitmap word) and random rows
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([np.arange(0, 4), np.arange(e * 128 - 2, e * 128 + 2),
                                     np.arange(L_MAX - 130, L_MAX, 7),
                                     rng.integers(0, L_MAX, size=24)]))
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, causal=True, block=128, row_ptr=rp,
                                  col_idx=ci)
    compare_forward(o[0, 0, rows], lse[0, 0, rows], O_ref[0, 0], l_ref[0, 0], "L=524288")
    # backward: whole key blocks, including the last one, against the oracle
    q, k, v, do = (to_f64(cpu[x])[0, 0] for x in ("q", "k", "v", "do"))
    for j, rows_j, gq, gk, gv in _sampled_reference(q, k, v, do, w.scale, rp, ci, N_MAX, L_MAX,
                                                    key_blocks=(100, 2047, 3000, N_MAX - 1)):
        sl = slice(j * 128, (j + 1) * 128)
        assert np.abs(dk[0, 0, sl].double().cpu().numpy() - gk).max() <= TOL_GRAD, j
        assert np.abs(dv[0, 0, sl].double().cpu().numpy() - gv).max() <= TOL_GRAD, j
        assert np.abs(dq[0, 0, rows_j].double().cpu().numpy() - gq).max() <= TOL_GRAD, j


def test_accounting_at_the_largest_key_range(bss, case):
    """Every sequence block is full here, so under the causal mask a listed
    block before its query block holds 128 x 128 allowed pairs, the diagonal
    block 128 * 129 / 2, and a later block none (counted as future); the
    lists are read through the oracle's CSR reading."""
    w, _, rp, ci = case
    got = bss.attn_blocklist_stats(rp, ci, L_MAX, causal=True).cpu().tolist()[0]
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    sets = oracle.blocklist_sets(rp, ci, N_MAX)
    listed = sum(len(s) for s in sets)
    future = sum(1 for a, s in enumerate(sets) for c in s if c > a)
    pairs = sum(128 * 128 * sum(1 for c in s if c < a) + (128 * 129 // 2 if a in s else 0)
                for a, s in enumerate(sets))
    assert got == [listed, listed - future, future, pairs]


def test_selector_at_the_largest_key_range(bss, case):
    """The mean-pooled selector over 4096 blocks (4 local and 4 best-scoring
    blocks per row): its lists against the oracle's selection, and the sparse
    forward on them runs clean."""
    from tests.test_gpu_select import check_lists
    w, cpu, _, _ = case
    inp = to_cuda(cpu)
    rp, ci = bss.attn_select_blocks(inp["q"], inp["k"], 4, local_blocks=4, causal=True,
                                    n_lists=1, scale=w.scale)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    check_lists(rp, ci, cpu, w.scale, 4, 4, True, 1)
