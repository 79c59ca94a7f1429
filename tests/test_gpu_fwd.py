"""Forward parity on the GPU through the C ABI: dense and causal attention,
ragged tails, offsets, the pages' worked example, closed forms and the watchdog."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.parity import (TOL_LSE, TOL_O, compare_forward, oracle_forward, tile_edge_rows,
                          to_cuda)
from workloads import CAUSAL_4K, DENSE_SMALL, CAUSAL_16K, Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


def test_dense_small_matches_oracle(bss):
    w = DENSE_SMALL
    inp = to_cuda(make_inputs(w))
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=False, scale=w.scale)
    torch.cuda.synchronize()
    O_ref, l_ref = oracle_forward(make_inputs(w), w.scale)
    compare_forward(o, lse, O_ref, l_ref, "dense L=256 d=64")
    assert bss.attn_poll_status() == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 63, 128, 129, 300, 513])
def test_shapes_with_ragged_tails(bss, d, causal, L):
    w = Workload("t", 2, 2, L, d, causal, seed=1000 + L + d)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o = torch.full_like(inp["q"], float("nan"))          # poisoned: every valid element
    lse = torch.full((2, 2, L), float("nan"), device="cuda")  # must be written
    bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=causal, scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=causal)
    compare_forward(o, lse, O_ref, l_ref, f"L={L} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Lq,Lk,q0,k0", [(200, 333, 150, 0), (300, 260, 0, 100), (130, 500, 400, 0),
                                         (257, 129, 5, 300)])
def test_causal_offsets_nonsquare(bss, d, Lq, Lk, q0, k0):
    g = torch.Generator().manual_seed(Lq * 7 + Lk)
    q = torch.randn(1, 3, Lq, d, generator=g).bfloat16()
    k = torch.randn(1, 3, Lk, d, generator=g).bfloat16()
    v = torch.randn(1, 3, Lk, d, generator=g).bfloat16()
    scale = d ** -0.5
    o, lse = bss.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale, q_offset=q0,
                          k_offset=k0)
    O_ref, l_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), scale, causal=True,
                                            q_offset=q0, k_offset=k0)
    compare_forward(o, lse, O_ref, l_ref, f"Lq={Lq} Lk={Lk} q0={q0} k0={k0}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Lq,Lk,q0,causal", [
    (100, 300, 100, True),    # rows 100-127 see block 0 only: the odd-block state is empty
    (128, 640, 0, False),     # five key blocks: the even slot takes one more
    (64, 512, 448, True),     # four key blocks, every row sees all of them
    (40, 256, 0, False),      # exactly two key blocks
    (1, 1000, 999, True),     # one query row
    (300, 700, 400, True),    # a full pair, then a single-tile pair
])
def test_single_tile_pairs(bss, d, Lq, Lk, q0, causal):
    """A pair whose second query tile lies past the last row takes its key blocks
    in turn in both tile slots and merges the two states per row; the result is
    the same attention."""
    g = torch.Generator().manual_seed(Lq * 11 + Lk + d)
    q = torch.randn(2, 2, Lq, d, generator=g).bfloat16()
    k = torch.randn(2, 2, Lk, d, generator=g).bfloat16()
    v = torch.randn(2, 2, Lk, d, generator=g).bfloat16()
    scale = d ** -0.5
    o = torch.full((2, 2, Lq, d), float("nan"), device="cuda").bfloat16()
    lse = torch.full((2, 2, Lq), float("nan"), device="cuda")
    bss.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, q_offset=q0, out=o,
                 lse=lse)
    torch.cuda.synchronize()
    O_ref, l_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), scale,
                                            causal=causal, q_offset=q0)
    compare_forward(o, lse, O_ref, l_ref, f"Lq={Lq} Lk={Lk} q0={q0} causal={causal}")
    assert bss.attn_poll_status() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_single_tile_pair_partial_state(bss, d):
    """The partial state (m, l, acc) of a single-tile pair, where some rows'
    keys all fall in the even blocks, against the oracle's state."""
    Lq, Lk, q0 = 100, 300, 100
    g = torch.Generator().manual_seed(d)
    q = torch.randn(1, 2, Lq, d, generator=g).bfloat16()
    k = torch.randn(1, 2, Lk, d, generator=g).bfloat16()
    v = torch.randn(1, 2, Lk, d, generator=g).bfloat16()
    scale = d ** -0.5
    m, l, acc = bss.attn_fwd_partial(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale,
                                     q_offset=q0)
    torch.cuda.synchronize()
    for h in range(2):
        M = oracle.allowed_rows(np.arange(Lq) + q0, Lk, causal=True)
        mr, lr, Ar = oracle.partial_state(to_f64(q)[0, h], to_f64(k)[0, h], to_f64(v)[0, h],
                                          scale, M)
        mg = m[0, h].double().cpu().numpy()
        lg = l[0, h].double().cpu().numpy()
        Ag = acc[0, h].double().cpu().numpy()
        assert not np.any(np.isneginf(mr)) and not np.any(np.isneginf(mg))
        assert np.abs(mg - mr).max() <= TOL_LSE
        assert np.abs((Ag / lg[:, None]) - (Ar / lr[:, None])).max() <= TOL_O
        assert np.abs((mg + np.log(lg)) - (mr + np.log(lr))).max() <= TOL_LSE
        assert lg.min() >= 1.0 - 1e-3      # the max element contributes e^0 = 1
    assert bss.attn_poll_status() == 0


def test_empty_key_set_gives_empty_rows(bss):
    q = torch.randn(1, 1, 100, 64).bfloat16().cuda()
    k = torch.randn(1, 1, 64, 64).bfloat16().cuda()
    o, lse = bss.attn_fwd(q, k, k, causal=True, q_offset=0, k_offset=1000)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_causal_4k_full_size_sampled_rows(bss):
    """The B=4 H=16 L=4096 d=128 causal workload, in the launch configuration of
    the benchmark, checked on sampled heads and rows."""
    w = CAUSAL_4K
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale)
    torch.cuda.synchronize()
    rows = tile_edge_rows(w.L, seed=1)
    heads = [(0, 0), (1, 7), (3, 15)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=heads, causal=True)
    for n, (b, h) in enumerate(heads):
        compare_forward(o[b, h, rows], lse[b, h, rows], O_ref[n], l_ref[n], f"head {(b, h)}")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_causal_16k_sampled_rows(bss):
    w = CAUSAL_16K
    cpu = make_inputs(w, B=1, H=2)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale)
    torch.cuda.synchronize()
    rows = tile_edge_rows(w.L, n_random=32, seed=5)[::3]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=[(0, 1)], causal=True)
    compare_forward(o[0, 1, rows], lse[0, 1, rows], O_ref[0], l_ref[0], "L=16384")


# ---------------------------------------------------------------------------
# Pins on the GPU: values fixed by the pages and by closed forms
# ---------------------------------------------------------------------------

def _overflow_keys(d):
    """Keys whose dot product with q = (1,...,1,0,...) is exactly 1000, 999, 1001:
    sums of powers of two spread over 8 dimensions (each exact in bf16)."""
    parts = {1000: [512, 256, 128, 64, 32, 8], 999: [512, 256, 128, 64, 32, 4, 2, 1],
             1001: [512, 256, 128, 64, 32, 8, 1]}
    k = torch.zeros(3, d)
    for j, logit in enumerate((1000, 999, 1001)):
        for t, x in enumerate(parts[logit]):
            k[j, t] = float(x)
    return k


@pytest.mark.parametrize("d", [64, 128])
def test_three_logit_overflow_example(bss, d):
    """'A three-logit numerical check' (Exact Blocks, Rings, and Sparsity, section 2):
    logits 1000, 999, 1001 with values 2, 4, 10 give 7.50199 without overflow,
    both in one tile and as two partial states merged."""
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "three_logit.json")))
    q = torch.zeros(1, 1, 128, d)
    q[..., :8] = 1.0
    k = _overflow_keys(d)[None, None]
    v = torch.zeros(1, 1, 3, d)
    v[0, 0, :, 0] = torch.tensor([2.0, 4.0, 10.0])
    q, k, v = (t.bfloat16().cuda() for t in (q, k, v))
    o, lse = bss.attn_fwd(q, k, v, scale=1.0)
    torch.cuda.synchronize()
    assert abs(o[0, 0, :, 0].float() - g["output"]).max().item() <= TOL_O
    assert abs(lse[0, 0].double() - g["lse"]).max().item() <= TOL_LSE
    # tile 1 = keys {1000, 999}, tile 2 = key {1001}: partial states, then the merge
    s1 = bss.attn_fwd_partial(q, k[:, :, :2].contiguous(), v[:, :, :2].contiguous(), scale=1.0)
    s2 = bss.attn_fwd_partial(q, k[:, :, 2:].contiguous(), v[:, :, 2:].contiguous(), scale=1.0)
    torch.cuda.synchronize()
    assert torch.allclose(s1[0], torch.full_like(s1[0], g["after_tile1"]["m"]))
    assert abs(s1[1] - g["after_tile1"]["l"]).max().item() < 1e-3
    assert abs(s1[2][..., 0] - g["after_tile1"]["A"]).max().item() < 2e-2
    m = torch.stack([s1[0], s2[0]])
    l = torch.stack([s1[1], s2[1]])
    acc = torch.stack([s1[2], s2[2]])
    om, lm = bss.attn_merge_states(m, l, acc)
    torch.cuda.synchronize()
    assert abs(om[0, 0, :, 0].float() - g["output"]).max().item() <= TOL_O
    assert abs(lm[0, 0].double() - g["lse"]).max().item() <= TOL_LSE


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_keys_closed_form(bss, causal):
    """All keys equal: O_i = mean of the visible V rows, LSE_i = s_i + ln(count)."""
    L, d = 300, 128
    g = torch.Generator().manual_seed(7)
    q = torch.randn(1, 2, L, d, generator=g).bfloat16()
    k = torch.randn(1, 2, 1, d, generator=g).bfloat16().expand(1, 2, L, d).contiguous()
    v = torch.randn(1, 2, L, d, generator=g).bfloat16()
    scale = d ** -0.5
    o, lse = bss.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    vf = v.double()
    if causal:
        mean = torch.cumsum(vf, dim=2) / torch.arange(1, L + 1, dtype=torch.float64)[:, None]
        count = torch.arange(1, L + 1, dtype=torch.float64)
    else:
        mean = vf.mean(dim=2, keepdim=True).expand_as(vf)
        count = torch.full((L,), float(L), dtype=torch.float64)
    s = scale * (q.double() @ k.double()[:, :, :1].transpose(-1, -2))[..., 0]
    assert (o.double().cpu() - mean).abs().max().item() <= TOL_O
    assert (lse.double().cpu() - (s + torch.log(count))).abs().max().item() <= TOL_LSE


def test_dominant_key_closed_form(bss):
    """One key aligned with every query at large magnitude: O_i -> V_{j*}."""
    L, d, jstar = 256, 64, 77
    u = torch.zeros(d)
    u[:4] = torch.tensor([2.0, -1.0, 0.5, 1.0])
    k = torch.zeros(1, 1, L, d)
    k[0, 0, jstar] = u
    q = (8.0 * u).expand(1, 1, L, d).contiguous()
    v = torch.randn(1, 1, L, d, generator=torch.Generator().manual_seed(3))
    q, k, v = (t.bfloat16() for t in (q, k, v))
    scale = 1.0
    o, lse = bss.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale)
    torch.cuda.synchronize()
    t_logit = float((q[0, 0, 0].double() @ k[0, 0, jstar].double()))
    w = math.exp(t_logit * scale)
    vd = v.double()[0, 0]
    expect = (w * vd[jstar] + vd.sum(0) - vd[jstar]) / (w + L - 1)
    assert (o[0, 0].double().cpu() - expect).abs().max().item() <= TOL_O
    assert abs(lse[0, 0].double().cpu() - math.log(w + L - 1)).max().item() <= TOL_LSE


def test_shift_invariance_on_device(bss):
    """Appending a dimension with K = 1 and Q = c_i/scale adds c_i to every logit
    of row i: O is unchanged and LSE moves by exactly c_i."""
    L, d = 384, 64
    g = torch.Generator().manual_seed(11)
    q = torch.randn(1, 1, L, d, generator=g)
    k = torch.randn(1, 1, L, d, generator=g)
    v = torch.randn(1, 1, L, d, generator=g)
    q[..., -1] = 0
    k[..., -1] = 0
    scale = 0.125
    c = torch.randint(-40, 40, (L,), generator=g).double()
    q2, k2 = q.clone(), k.clone()
    q2[0, 0, :, -1] = (c / scale).float()
    k2[..., -1] = 1.0
    args = lambda a, b: (a.bfloat16().cuda(), b.bfloat16().cuda(), v.bfloat16().cuda())
    for causal in (False, True):
        o1, l1 = bss.attn_fwd(*args(q, k), causal=causal, scale=scale)
        o2, l2 = bss.attn_fwd(*args(q2, k2), causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert (o1.float() - o2.float()).abs().max().item() <= TOL_O
        assert ((l2.double() - l1.double()).cpu()[0, 0] - c).abs().max().item() <= TOL_LSE


def test_watchdog_gives_up_and_reports(bss):
    """A wait that nobody completes returns after its limit with ATTN_ERR_TIMEOUT;
    the context stays usable."""
    assert bss.attn_poll_status() == 0
    bss.attn_watchdog_selftest(1 << 20)
    assert bss.attn_poll_status() == bss.ERR_TIMEOUT
    assert bss.attn_poll_status() == 0
    x = torch.ones(4, device="cuda")
    assert x.sum().item() == 4.0


def test_ex2_rate_probe(bss):
    """The exponential-rate kernel runs clean, rejects bad arguments, and its
    rate lies between 1 and 64 exponentials per clock per SM at 1-2.2 GHz."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.zeros(1, device="cuda")
    with pytest.raises(bss.AttnError):
        bss.attn_probe_ex2_rate(0, 16, sink=sink)
    n = bss.attn_probe_ex2_rate(sms * 8, 64, sink=sink)       # warm-up
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(1_000_000)
    a.record()
    n = bss.attn_probe_ex2_rate(sms * 8, 1024, sink=sink)
    b.record()
    torch.cuda.synchronize()
    rate = n / (a.elapsed_time(b) * 1e-3)
    assert sms * 1.0 * 1e9 <= rate <= sms * 64 * 2.2e9
    assert sink.item() == 0.0
    assert bss.attn_poll_status() == 0
