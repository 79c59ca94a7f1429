"""The bench step's rows at their full size (causal B=4 H=16 L=4096 d=128), in
the benchmark's launch configuration, against the oracle on sampled heads and
rows: the backward (every element of two heads), the 8-chunk split-KV forward
and the block-sparse forward on the step's list."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import TOL_GRAD, compare_forward, oracle_forward, tile_edge_rows, to_cuda
from workloads import CAUSAL_4K, Workload, local_global_random_blocklist, make_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


@pytest.fixture(scope="module")
def step_inputs():
    w = CAUSAL_4K
    w = Workload(w.name, w.B, w.H, w.L, w.d, True, w.seed, backward=True)
    cpu = make_inputs(w)
    return w, cpu, to_cuda(cpu)


def test_step_backward_full_size(bss, step_inputs):
    w, cpu, inp = step_inputs
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale)
    dq, dk, dv, _ = bss.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True,
                                 scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    q, k, v, do = (to_f64(cpu[n]) for n in ("q", "k", "v", "do"))
    heads = [(0, 0), (3, 15)]
    gq, gk, gv, _ = oracle.attention_backward(q, k, v, do, w.scale, causal=True, heads=heads)
    for n_, (b, h) in enumerate(heads):
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]),
                              (gq[n_], gk[n_], gv[n_])):
            err = np.abs(g.double().cpu().numpy() - r).max()
            assert err <= TOL_GRAD, f"head {(b, h)}: max|d{name}| = {err:.3e}"


def test_step_splitkv_full_size_sampled(bss, step_inputs):
    w, cpu, inp = step_inputs
    o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], 8, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    rows = tile_edge_rows(w.L, seed=3)
    heads = [(0, 1), (2, 9)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=heads, causal=True)
    for n_, (b, h) in enumerate(heads):
        compare_forward(o[b, h, rows], lse[b, h, rows], O_ref[n_], l_ref[n_], f"head {(b, h)}")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_step_blocksparse_full_size_sampled(bss, step_inputs):
    w, cpu, inp = step_inputs
    rp, ci = local_global_random_blocklist((w.L + 127) // 128, seed=2)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    rows = tile_edge_rows(w.L, seed=4)
    heads = [(1, 4), (3, 13)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=heads, causal=True, block=128,
                                  row_ptr=rp, col_idx=ci)
    for n_, (b, h) in enumerate(heads):
        compare_forward(o[b, h, rows], lse[b, h, rows], O_ref[n_], l_ref[n_], f"head {(b, h)}")
