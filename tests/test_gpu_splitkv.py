"""Split-KV / decode-shaped forward on the GPU (attn_fwd_splitkv through the C
ABI): the keys cut into chunks whose partial states are computed in one launch
and merged, checked against the oracle for decode shapes (few queries at the
end of a long causal cache), prefill shapes, chunk counts above the number of
key blocks, and the B=4 H=16 Lq=16 Lk=16384 decode workload."""
import numpy as np
import pytest
import torch

from tests.parity import TOL_LSE, TOL_O, compare_forward, oracle_forward, to_cuda
from workloads import DECODE_16K, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


def _decode_inputs(B, H, Lq, Lk, d, seed):
    """Queries are the last Lq positions of a [B, H, Lk, d] draw."""
    w = Workload("dec", B, H, Lk, d, True, seed, Lq=Lq)
    cpu = make_inputs(w)
    return w, cpu


@pytest.mark.parametrize("B,H,Lq,Lk,d,chunks", [
    (2, 4, 1, 3000, 128, 8),        # single query token
    (1, 8, 16, 5000, 64, 16),
    (2, 2, 200, 2048, 128, 4),      # more queries than a tile
    (1, 2, 7, 300, 128, 16),        # more chunks asked than key blocks: 3 chunks
    (1, 1, 5, 100, 64, 4),          # fewer keys than one block
    (2, 4, 16, 1100, 128, 8),       # chunks of 256 keys and a last one of 76:
    (1, 4, 100, 1100, 64, 8),       # two-block items beside a one-block item
])
def test_decode_shapes_match_oracle(bss, B, H, Lq, Lk, d, chunks):
    w, cpu = _decode_inputs(B, H, Lq, Lk, d, seed=Lq + Lk)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], chunks, causal=True,
                                  scale=w.scale, q_offset=Lk - Lq)
    o1, l1 = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale,
                          q_offset=Lk - Lq)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=True, q_offset=Lk - Lq)
    compare_forward(o, lse, O_ref, l_ref, f"decode Lq={Lq} Lk={Lk} chunks={chunks}")
    assert (o.float() - o1.float()).abs().max().item() <= TOL_O
    assert (lse - l1).abs().max().item() <= TOL_LSE


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("chunks", [1, 2, 5, 64])
def test_prefill_shapes_match_oracle(bss, causal, chunks):
    """Lq = Lk: chunks in the causal future of a query tile are skipped for it."""
    L, d = 1300, 128
    w = Workload("pf", 1, 2, L, d, causal, seed=chunks)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], chunks, causal=causal,
                                  scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=causal)
    compare_forward(o, lse, O_ref, l_ref, f"prefill chunks={chunks} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_queries_before_every_key_are_empty(bss, d):
    """Causal with k_offset beyond the first queries: those rows see no key in
    any chunk, so their merged state is empty (O = 0, LSE = -inf)."""
    Lq, Lk = 300, 1000
    w = Workload("ko", 1, 2, Lk, d, True, seed=7, Lq=Lq)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], 4, causal=True, scale=w.scale,
                                  q_offset=0, k_offset=100)
    torch.cuda.synchronize()
    assert torch.all(torch.isneginf(lse[:, :, :100])) and torch.all(o[:, :, :100] == 0)
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=True, q_offset=0, k_offset=100)
    compare_forward(o, lse, O_ref, l_ref, "k_offset")


def test_decode_workload_full_size(bss):
    """B=4 H=16, 16 queries at the end of a 16384-key causal cache, in the
    benchmark's launch configuration (2 chunks) and in 16 chunks: every row
    against the oracle for two heads, and all heads against the unsplit kernel."""
    w = DECODE_16K
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    qo = w.L - w.Lq
    o1, l1 = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=True, scale=w.scale, q_offset=qo)
    heads = [(0, 0), (3, 15)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, heads=heads, causal=True, q_offset=qo)
    for chunks in (w.chunks, 16):
        o, lse = bss.attn_fwd_splitkv(inp["q"], inp["k"], inp["v"], chunks, causal=True,
                                      scale=w.scale, q_offset=qo)
        torch.cuda.synchronize()
        assert bss.attn_poll_status() == 0
        assert (o.float() - o1.float()).abs().max().item() <= TOL_O
        assert (lse - l1).abs().max().item() <= TOL_LSE
        for n_, (b, h) in enumerate(heads):
            compare_forward(o[b, h], lse[b, h], O_ref[n_], l_ref[n_],
                            f"head {(b, h)}, {chunks} chunks")
    for n_, (b, h) in enumerate(heads):
        compare_forward(o1[b, h], l1[b, h], O_ref[n_], l_ref[n_], f"unsplit head {(b, h)}")
