"""Backward parity on the GPU through the C ABI: dQ, dK, dV (bf16) and the
row statistic D against the oracle's analytic gradients."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import TOL_GRAD, to_cuda
from workloads import BWD_8K, Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


def _check_grads(got, ref, what):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        gn = g.double().cpu().numpy()
        assert np.isfinite(gn).all(), f"{what}: {name} not finite"
        err = np.abs(gn - r).max()
        assert err <= TOL_GRAD, f"{what}: max|d{name}| = {err:.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("L", [128, 300, 513])
def test_backward_matches_oracle(bss, d, causal, L):
    w = Workload("b", 1, 2, L, d, causal, seed=500 + L + d, backward=True)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=causal, scale=w.scale)
    dq, dk, dv, delta = bss.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"],
                                     causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    q, k, v, do = (to_f64(cpu[n]) for n in ("q", "k", "v", "do"))
    gq, gk, gv, D = oracle.attention_backward(q, k, v, do, w.scale, causal=causal)
    _check_grads((dq, dk, dv), (gq, gk, gv), f"L={L} d={d} causal={causal}")
    # delta is D_i = dO_i . O_i from the saved bf16 O
    d_def = (inp["do"].double() * o.double()).sum(-1).cpu().numpy()
    assert np.abs(delta.double().cpu().numpy() - d_def).max() <= 1e-3
    assert np.abs(delta.double().cpu().numpy() - D).max() <= TOL_GRAD


def test_equal_value_rows_give_zero_dq_dk(bss):
    """Every V row equal: dP is constant along each row, so dS = 0 and dQ = dK = 0
    (Exact Blocks, Rings, and Sparsity, section 3, the constant-gradient example)."""
    L, d = 400, 64
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, 1, L, d, generator=g).bfloat16().cuda()
    k = torch.randn(1, 1, L, d, generator=g).bfloat16().cuda()
    v = torch.randn(1, 1, 1, d, generator=g).bfloat16().expand(1, 1, L, d).contiguous().cuda()
    do = torch.randn(1, 1, L, d, generator=g).bfloat16().cuda()
    o, lse = bss.attn_fwd(q, k, v, causal=True)
    dq, dk, dv, _ = bss.attn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert dq.abs().max().item() <= 1e-2 and dk.abs().max().item() <= 1e-2
    assert dv.abs().max().item() > 0.1


def test_backward_8k_full_size(bss):
    """B=8 H=16 L=8192 d=64 causal forward + backward (the benchmark's launch
    configuration); two heads checked against the oracle on every element."""
    w = BWD_8K
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale)
    dq, dk, dv, delta = bss.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True,
                                     scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    q, k, v, do = (to_f64(cpu[n]) for n in ("q", "k", "v", "do"))
    heads = [(0, 0), (7, 15)]
    gq, gk, gv, _ = oracle.attention_backward(q, k, v, do, w.scale, causal=True, heads=heads)
    for n_, (b, h) in enumerate(heads):
        _check_grads((dq[b, h], dk[b, h], dv[b, h]), (gq[n_], gk[n_], gv[n_]), f"head {(b, h)}")


def test_main_kernel_timing_events(bss):
    """attn_bwd_time_main: the events bracket the main kernel alone, so their
    interval is positive and shorter than the whole call's; clearing stops the
    recording, and setting only one event is refused."""
    import torch
    w = Workload("tm", 1, 4, 2048, 128, True, seed=8, backward=True)
    inp = to_cuda(make_inputs(w))
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    bss.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True, scale=w.scale)
    bss.attn_bwd_time_main(ev[1], ev[2])
    ev[0].record()
    bss.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True, scale=w.scale)
    ev[3].record()
    bss.attn_bwd_time_main()
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    main_ms, call_ms = ev[1].elapsed_time(ev[2]), ev[0].elapsed_time(ev[3])
    assert 0 < main_ms < call_ms
    # cleared: a later call leaves the events where they were
    t_before = ev[1].elapsed_time(ev[2])
    bss.attn_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert ev[1].elapsed_time(ev[2]) == t_before
    from block_sparse_softmax_gb300 import _lib
    assert _lib.load().attn_bwd_time_main(ev[1].cuda_event, None) == bss.ERR_INVALID_ARG
