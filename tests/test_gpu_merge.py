"""Partial states over KV chunks and their merge on the GPU (the Ring-Attention
combine on one device): the state itself against the oracle, chunked == unchunked
in any order, empty states, and the long B=1 H=8 L=131072 workload."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import (TOL_LSE, TOL_O, compare_forward, oracle_forward, tile_edge_rows,
                          to_cuda)
from workloads import SPLITKV_128K, Workload, chunk_bounds, make_inputs, sample_rows, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("s,e", [(0, 300), (250, 700), (640, 1000)])
def test_partial_state_matches_oracle(bss, d, s, e):
    L = 1000
    w = Workload("p", 1, 2, L, d, True, seed=s + e)
    cpu = make_inputs(w)
    q = cpu["q"].cuda()
    kc = cpu["k"][:, :, s:e].contiguous().cuda()
    vc = cpu["v"][:, :, s:e].contiguous().cuda()
    m, l, acc = bss.attn_fwd_partial(q, kc, vc, causal=True, scale=w.scale, k_offset=s)
    torch.cuda.synchronize()
    qn, kn, vn = (to_f64(cpu[n]) for n in ("q", "k", "v"))
    for h in range(2):
        M = oracle.allowed_rows(np.arange(L), e - s, causal=True, k_offset=s)
        mr, lr, Ar = oracle.partial_state(qn[0, h], kn[0, h, s:e], vn[0, h, s:e], w.scale, M)
        mg = m[0, h].double().cpu().numpy()
        lg = l[0, h].double().cpu().numpy()
        Ag = acc[0, h].double().cpu().numpy()
        empty = np.isneginf(mr)
        assert np.array_equal(np.isneginf(mg), empty)
        assert np.all(lg[empty] == 0)          # acc of an empty state is not written
        f = ~empty
        # m is the exact maximum; l and A share it, so A/l and m + ln l are the
        # chunk's O and LSE
        assert np.abs(mg[f] - mr[f]).max() <= TOL_LSE
        assert np.abs((Ag[f] / lg[f, None]) - (Ar[f] / lr[f, None])).max() <= TOL_O
        assert np.abs((mg[f] + np.log(lg[f])) - (mr[f] + np.log(lr[f]))).max() <= TOL_LSE
        assert lg[f].min() >= 1.0 - 1e-3          # the max element contributes e^0 = 1


@pytest.mark.parametrize("chunks", [2, 3, 8])
@pytest.mark.parametrize("causal", [True, False])
def test_split_kv_merge_equals_oracle_and_unsplit(bss, chunks, causal):
    L, d = 1100, 128
    w = Workload("m", 1, 3, L, d, causal, seed=chunks)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], chunks, causal=causal,
                                  scale=w.scale)
    o1, l1 = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=causal)
    compare_forward(o, lse, O_ref, l_ref, f"{chunks} chunks")
    assert (o.float() - o1.float()).abs().max().item() <= TOL_O
    assert (lse - l1).abs().max().item() <= TOL_LSE


def test_merge_order_does_not_matter(bss):
    """Chunk states merged in three orders: each result matches the oracle's
    unchunked attention, and the orders agree with each other."""
    L, d, C = 700, 64, 5
    w = Workload("o", 2, 2, L, d, True, seed=31)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    bounds = chunk_bounds(L, C)
    states = [bss.attn_fwd_partial(inp["q"], inp["k"][:, :, s:e].contiguous(),
                                   inp["v"][:, :, s:e].contiguous(), causal=True, k_offset=s)
              for s, e in bounds]
    outs = []
    for perm in ([0, 1, 2, 3, 4], [4, 2, 0, 3, 1], [3, 4, 1, 0, 2]):
        m = torch.stack([states[i][0] for i in perm])
        l = torch.stack([states[i][1] for i in perm])
        a = torch.stack([states[i][2] for i in perm])
        outs.append(bss.attn_merge_states(m, l, a))
    torch.cuda.synchronize()
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=True)
    for n_, (o, lse) in enumerate(outs):
        compare_forward(o, lse, O_ref, l_ref, f"merge order {n_}")
    for o, lse in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 1e-2
        assert (lse - outs[0][1]).abs().max().item() <= 1e-5


def _per_chunk(bss, inp, bounds, scale, q_offset=0):
    """attn_fwd_partial once per key chunk (chunks copied out, as a Ring step
    receives them), then attn_merge_states over the stacked states."""
    q = inp["q"]
    B, H, Lq, d = q.shape
    C = len(bounds)
    m = torch.empty(C, B, H, Lq, device="cuda")
    l = torch.empty_like(m)
    acc = torch.empty(C, B, H, Lq, d, device="cuda")
    for c, (s, e) in enumerate(bounds):
        bss.attn_fwd_partial(q, inp["k"][:, :, s:e].contiguous(), inp["v"][:, :, s:e].contiguous(),
                             causal=True, scale=scale, q_offset=q_offset, k_offset=s, m=m[c],
                             l=l[c], acc=acc[c])
    o, lse = bss.attn_merge_states(m, l, acc)
    return o, lse, m


def test_per_chunk_partials_and_merge_against_the_oracle(bss):
    """The Ring combine as separate launches: 8 chunk states of a causal
    L = 4096 head set, merged, against the oracle on tile-edge and chunk-edge
    rows.  Rows 0..511 see only the first chunk, so 7 of their 8 states are
    empty."""
    L, d = 4096, 128
    w = Workload("pc", 1, 4, L, d, True, seed=33)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    bounds = chunk_bounds(L, 8)
    o, lse, m = _per_chunk(bss, inp, bounds, w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.isneginf(m[1:, :, :, :512]).all()          # empty chunk states
    rows = tile_edge_rows(L, seed=5)
    heads = [(0, 0), (0, 3)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=heads, causal=True)
    for n_, (b, h) in enumerate(heads):
        compare_forward(o[b, h, rows], lse[b, h, rows], O_ref[n_], l_ref[n_], f"head {(b, h)}")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_per_chunk_merge_with_a_chunk_wholly_in_the_future(bss):
    """Keys extend 512 positions past the last query: the ninth chunk is empty
    for every row, the merge skips it, and the result is the oracle's."""
    Lq, Lk, d = 1536, 2048, 64
    w = Workload("pf", 1, 2, Lk, d, True, seed=34)
    cpu = make_inputs(w)
    cpu["q"] = cpu["q"][:, :, :Lq].contiguous()
    inp = to_cuda(cpu)
    bounds = chunk_bounds(Lk, 4)
    o, lse, m = _per_chunk(bss, inp, bounds, w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.isneginf(m[3]).all()
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=True)
    compare_forward(o, lse, O_ref, l_ref, "future chunk")


def test_merge_of_empty_states(bss):
    C, B, H, L, d = 3, 1, 2, 130, 64
    m = torch.full((C, B, H, L), float("-inf"), device="cuda")
    l = torch.zeros_like(m)
    acc = torch.full((C, B, H, L, d), float("nan"), device="cuda")   # never read
    m[1, 0, 1, 5] = 2.0
    l[1, 0, 1, 5] = 4.0
    acc[1, 0, 1, 5] = 8.0
    o, lse = bss.attn_merge_states(m, l, acc)
    torch.cuda.synchronize()
    assert torch.isneginf(lse).sum().item() == B * H * L - 1
    assert torch.all(o[0, 0] == 0)
    assert torch.allclose(o[0, 1, 5].float(), torch.full((d,), 2.0, device="cuda"))
    assert abs(lse[0, 1, 5].item() - (2.0 + np.log(4.0))) < 1e-5


def test_long_context_split_kv_full_size(bss):
    """B=1 H=8 L=131072 d=128 causal, values x0.5, 8 contiguous KV chunks each
    attended separately then merged; compared with the unsplit kernel on every
    row and with the oracle on sampled rows."""
    w = SPLITKV_128K
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], w.chunks, causal=True,
                                  scale=w.scale)
    o1, l1 = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert (o.float() - o1.float()).abs().max().item() <= TOL_O
    assert (lse - l1).abs().max().item() <= TOL_LSE
    rows = sample_rows(w.L, w.chunks, 96, seed=w.seed)
    heads = [(0, 0), (0, 5)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=heads, causal=True)
    for n_, (b, h) in enumerate(heads):
        compare_forward(o[b, h, rows], lse[b, h, rows], O_ref[n_], l_ref[n_], f"head {(b, h)}")


def test_long_context_per_chunk_launches_full_size(bss):
    """B=1 H=8 L=131072 d=128, the long workload as its description has it:
    each of the 8 contiguous KV chunks attended separately (one
    attn_fwd_partial launch each) and the states merged; against the oracle on
    sampled rows of two heads."""
    w = SPLITKV_128K
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse, m = _per_chunk(bss, inp, chunk_bounds(w.L, w.chunks), w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    del m
    rows = sample_rows(w.L, w.chunks, 96, seed=w.seed)
    heads = [(0, 2), (0, 7)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=heads, causal=True)
    for n_, (b, h) in enumerate(heads):
        compare_forward(o[b, h, rows], lse[b, h, rows], O_ref[n_], l_ref[n_], f"head {(b, h)}")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True])
def test_long_chunk_partial_state_matches_oracle(bss, causal):
    """One chunk of 4296 keys (34 blocks, the last one 72 keys) at d=128: the
    kernel with 256-key score tiles takes chunks of 4096 keys or more.  The
    state against the oracle, dense and causal (the chunk starts at key 700,
    so the first 700 query rows see none of it under the causal mask)."""
    L, s, e = 5000, 700, 4996
    w = Workload("pl", 1, 2, L, 128, causal, seed=71)
    cpu = make_inputs(w)
    q = cpu["q"][:, :, :300 + 128 * 9].contiguous()
    Lq = q.shape[2]
    kc = cpu["k"][:, :, s:e].contiguous().cuda()
    vc = cpu["v"][:, :, s:e].contiguous().cuda()
    m, l, acc = bss.attn_fwd_partial(q.cuda(), kc, vc, causal=causal, scale=w.scale, k_offset=s)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    qn, kn, vn = (to_f64(t) for t in (q, cpu["k"], cpu["v"]))
    for h in range(2):
        M = oracle.allowed_rows(np.arange(Lq), e - s, causal=causal, k_offset=s)
        mr, lr, Ar = oracle.partial_state(qn[0, h], kn[0, h, s:e], vn[0, h, s:e], w.scale, M)
        mg = m[0, h].double().cpu().numpy()
        lg = l[0, h].double().cpu().numpy()
        Ag = acc[0, h].double().cpu().numpy()
        empty = np.isneginf(mr)
        assert np.array_equal(np.isneginf(mg), empty)
        assert causal == bool(empty.any())
        assert np.all(lg[empty] == 0)
        f = ~empty
        assert np.abs(mg[f] - mr[f]).max() <= TOL_LSE
        assert np.abs((Ag[f] / lg[f, None]) - (Ar[f] / lr[f, None])).max() <= TOL_O
        assert np.abs((mg[f] + np.log(lg[f])) - (mr[f] + np.log(lr[f]))).max() <= TOL_LSE
        assert lg[f].min() >= 1.0 - 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_split_kv_long_chunks_match_oracle(bss, causal):
    """L=9000 in 2 chunks (4608 keys, then 4392 with a partial last block) at
    d=128, B=1 H=3: both chunks run the kernel with 256-key score tiles.  The
    merged O and LSE against the oracle on every tile edge and random rows,
    and against the unsplit forward."""
    L = 9000
    w = Workload("sl", 1, 3, L, 128, causal, seed=73)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], 2, causal=causal, scale=w.scale)
    o1, l1 = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    rows = tile_edge_rows(L, n_random=32, seed=5)[::3]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, causal=causal)
    compare_forward(o[:, :, rows], lse[:, :, rows], O_ref, l_ref, f"2 long chunks causal={causal}")
    assert (o.float() - o1.float()).abs().max().item() <= TOL_O
    assert (lse - l1).abs().max().item() <= TOL_LSE
