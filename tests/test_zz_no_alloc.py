"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers may not call cudaMalloc or keep a workspace buffer of their own
(an allocator that forbids new device allocations, a host that hands out
none).  attn_bwd_noalloc serves them by keeping the fp32 dQ accumulator in a
static device array inside the library.  These tests call it through the C
ABI, twice in a row on different problems, and compare every output with the
regular attn_bwd (which takes a caller-provided workspace): dK, dV and D must
be identical, dQ (accumulated with atomics in a different order) within the
gradient tolerance of the other tests.  They also compare it with the oracle's
analytic gradients directly, with grouped K/V heads, and at exactly the
scratch's size.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests.parity import TOL_GRAD
from workloads import Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 8 << 20


@pytest.fixture(scope="module")
def lib():
    import block_sparse_softmax_gb300 as bss
    return bss.library()


def _call_noalloc(lib, x, o, lse, causal, scale):
    B, H, L, d = x["q"].shape
    Hkv = x["k"].shape[1]
    dq = torch.empty_like(x["q"])
    dk, dv = torch.empty_like(x["k"]), torch.empty_like(x["v"])
    delta = torch.empty((B, H, L), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.attn_bwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                              o.data_ptr(), lse.data_ptr(), x["do"].data_ptr(), dq.data_ptr(),
                              dk.data_ptr(), dv.data_ptr(), delta.data_ptr(), B, H, Hkv, L, d,
                              scale, int(causal), stream)
    assert st == 0, lib.attn_last_error_message()
    return dq, dk, dv, delta


def _against_oracle(cpu, w, got, heads):
    """Every element of dQ, dK, dV of the listed (b, h) query heads against the
    oracle's analytic gradients (per query head; with grouped heads dK and dV
    are compared as the sum over the group)."""
    q, k, v, do = (to_f64(cpu[n]) for n in ("q", "k", "v", "do"))
    H, Hkv = q.shape[1], k.shape[1]
    G = H // Hkv
    gq, gk, gv, _ = oracle.attention_backward(q, k, v, do, w.scale, causal=w.causal)
    dq, dk, dv, _ = got
    for b, h in heads:
        for name, a, r in (("dq", dq[b, h], gq[b, h]), ("dk", dk[b, h // G], gk[b, h // G]),
                           ("dv", dv[b, h // G], gv[b, h // G])):
            err = np.abs(a.double().cpu().numpy() - r).max()
            assert err <= TOL_GRAD, f"head {(b, h)}: max|d{name}| = {err:.3e}"


@pytest.mark.parametrize("order", ["first", "second"])
def test_noalloc_matches_attn_bwd_on_two_calls_in_a_row(lib, order):
    import block_sparse_softmax_gb300 as bss
    problems = [Workload("na1", 1, 4, 1000, 128, True, seed=61, backward=True),
                Workload("na2", 2, 3, 700, 64, False, seed=62, backward=True)]
    if order == "second":
        problems.reverse()
    for w in problems:
        x = {n: t.cuda() for n, t in make_inputs(w).items()}
        o, lse = bss.attn_fwd(x["q"], x["k"], x["v"], causal=w.causal, scale=w.scale)
        ref = bss.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=w.causal,
                           scale=w.scale)
        got = _call_noalloc(lib, x, o, lse, w.causal, w.scale)
        torch.cuda.synchronize()
        assert bss.attn_poll_status() == 0
        dq, dk, dv, delta = got
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
        assert torch.equal(delta, ref[3])
        assert (dq.float() - ref[0].float()).abs().max().item() <= TOL_GRAD
        assert torch.isfinite(dq).all()


@pytest.mark.parametrize("H,Hkv", [(3, 3), (4, 2)])
def test_noalloc_matches_the_oracle(lib, H, Hkv):
    """Small causal problems, plain and with grouped K/V heads, against the
    oracle's gradients on two calls in a row."""
    import block_sparse_softmax_gb300 as bss
    w = Workload("na_or", 1, H, 300, 64, True, seed=63 + H, backward=True, Hkv=Hkv)
    cpu = make_inputs(w)
    x = {n: t.cuda() for n, t in cpu.items()}
    o, lse = bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale)
    for _ in range(2):
        got = _call_noalloc(lib, x, o, lse, True, w.scale)
        torch.cuda.synchronize()
        assert bss.attn_poll_status() == 0
        _against_oracle(cpu, w, got, [(0, h) for h in range(H)])


def test_noalloc_at_the_scratch_limit(lib):
    """B*H*L*d exactly 8388608 (1 x 16 x 4096 x 128, causal): the whole scratch
    in use.  dK, dV and D equal attn_bwd's; dQ is within the gradient
    tolerance of attn_bwd's everywhere and of the oracle on two heads."""
    import block_sparse_softmax_gb300 as bss
    w = Workload("na_full", 1, 16, 4096, 128, True, seed=65, backward=True)
    assert w.B * w.H * w.L * w.d == SCRATCH_FLOATS
    cpu = make_inputs(w)
    x = {n: t.cuda() for n, t in cpu.items()}
    o, lse = bss.attn_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale)
    ref = bss.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=True, scale=w.scale)
    got = _call_noalloc(lib, x, o, lse, True, w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    assert torch.equal(got[3], ref[3])
    assert (got[0].float() - ref[0].float()).abs().max().item() <= TOL_GRAD
    q, k, v, do = (to_f64(cpu[n]) for n in ("q", "k", "v", "do"))
    heads = [(0, 0), (0, 15)]
    gq, gk, gv, _ = oracle.attention_backward(q, k, v, do, w.scale, causal=True, heads=heads)
    for n_, (b, h) in enumerate(heads):
        for name, a, r in (("dq", got[0][b, h], gq[n_]), ("dk", got[1][b, h], gk[n_]),
                           ("dv", got[2][b, h], gv[n_])):
            err = np.abs(a.double().cpu().numpy() - r).max()
            assert err <= TOL_GRAD, f"head {(b, h)}: max|d{name}| = {err:.3e}"


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # 1 x 16 x 4097 x 128 > 8388608 floats: rejected before any device work
    p = ctypes.c_void_p(16 * 4096)
    st = lib.attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, p, 1, 16, 16, 4097, 128, 0.125, 1, None)
    assert st == 6
    assert b"exceeds the static scratch" in lib.attn_last_error_message()
    # exactly at the limit is accepted by the size check (fails later only on the
    # null pointer test here, which is ATTN_ERR_INVALID_ARG, not the size error)
    st = lib.attn_bwd_noalloc(None, p, p, p, p, p, p, p, p, p, 1, 16, 16, 4096, 128, 0.125, 1, None)
    assert st == 1
