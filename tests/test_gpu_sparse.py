"""Block-sparse forward parity on the GPU: the local + global + random pattern
with duplicates, an empty row and a partial last block; unstructured lists;
set semantics (order and duplicates never matter); equivalence with the dense
kernels when every block is listed; bad entries reported."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import (TOL_LSE, TOL_O, compare_forward, oracle_forward, tile_edge_rows,
                          to_cuda)
from workloads import (SPARSE_16K, Workload, local_global_random_blocklist, make_inputs,
                       random_blocklist)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_local_global_random_pattern_reduced(bss, d, causal):
    L = 2048 - 64                                   # 16 blocks, the last one half full
    n = (L + 127) // 128
    rp, ci = local_global_random_blocklist(n, seed=2)
    w = Workload("s", 1, 2, L, d, causal, seed=2)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o = torch.full_like(inp["q"], float("nan"))
    lse = torch.full((1, 2, L), float("nan"), device="cuda")
    bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal, scale=w.scale,
                             out=o, lse=lse)
    torch.cuda.synchronize()
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=causal, block=128, row_ptr=rp, col_idx=ci)
    compare_forward(o, lse, O_ref, l_ref, f"pattern d={d} causal={causal}")
    assert torch.all(torch.isneginf(lse[:, :, (n // 2) * 128:(n // 2 + 1) * 128]))
    assert bss.attn_poll_status() == 0


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("d", [64, 128])
def test_unstructured_lists(bss, seed, d):
    L = 1000
    n = (L + 127) // 128
    rp, ci = random_blocklist(n, n, seed=seed, max_per_row=5)
    causal = seed % 2 == 1
    w = Workload("u", 2, 1, L, d, causal, seed=40 + seed)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal,
                                      scale=w.scale)
    torch.cuda.synchronize()
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=causal, block=128, row_ptr=rp, col_idx=ci)
    compare_forward(o, lse, O_ref, l_ref, f"random list seed={seed}")


def _repeat_rows(rp, ci, times, rng=None):
    """Each row's entries `times` times over, in a random order when `rng`."""
    rows = [np.repeat(ci[rp[a]:rp[a + 1]], times) for a in range(len(rp) - 1)]
    if rng is not None:
        rows = [rng.permutation(r) for r in rows]
    return (rp * times).astype(np.int32), np.concatenate(rows).astype(np.int32)


@pytest.mark.parametrize("d", [64, 128])
def test_order_and_duplicates_are_bit_identical(bss, d):
    """A block list is a set: the raw list, a permutation of every row, the
    normalised list, and the normalised rows listed 2, 3 and 4 times over
    (permuted) give the same bits.  The kernel a launch runs depends on d and
    L only, never on the lists."""
    L = 1500
    n = (L + 127) // 128
    rp, ci = random_blocklist(n, n, seed=9, max_per_row=7, p_empty=0.1)
    cp, cc = bss.attn_blocklist_normalize(rp, ci, n)
    rng = np.random.default_rng(0)
    lists = {"raw": (rp, ci), "raw permuted": _repeat_rows(rp, ci, 1, rng),
             "normalised": (cp, cc), "twice": _repeat_rows(cp, cc, 2),
             "3x": _repeat_rows(cp, cc, 3, rng), "4x": _repeat_rows(cp, cc, 4, rng)}
    w = Workload("p", 1, 2, L, d, True, seed=5)
    inp = to_cuda(make_inputs(w))
    out = {k: bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], r, c, causal=True)
           for k, (r, c) in lists.items()}
    torch.cuda.synchronize()
    for k, x in out.items():
        assert torch.equal(out["raw"][0], x[0]) and torch.equal(out["raw"][1], x[1]), k


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,L", [(64, 700), (64, 777), (128, 1900), (128, 2047)])
def test_all_blocks_listed_equals_dense_kernel(bss, causal, L, d):
    """Where a pair of query tiles is full, both kernels visit the same blocks in
    the same order and agree bit for bit.  At d=64 a last pair with a single
    tile (rows 768-776 at L=777) is split over both tile slots by the dense
    kernel, which sums its blocks in another order: those rows agree within the
    tolerance.  At d=128 (15 and 16 blocks) both launches run the kernel with
    256-key score tiles: one query tile an item and key blocks two at a time
    in ascending order; where the count is odd the block-sparse item scores
    its last block alone and the dense one beside a masked block, whose P is
    exactly zero: every row agrees bit for bit."""
    n = (L + 127) // 128
    if causal:
        rows = [list(range(a + 1)) for a in range(n)]
    else:
        rows = [list(range(n))[::-1] for _ in range(n)]
    rp = np.cumsum([0] + [len(r) for r in rows]).astype(np.int32)
    ci = np.array([c for r in rows for c in r], np.int32)
    inp = to_cuda(make_inputs(Workload("a", 2, 2, L, d, causal, seed=77)))
    o_s, l_s = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal)
    o_d, l_d = bss.attn_fwd(inp["q"], inp["k"], inp["v"], causal=causal)
    torch.cuda.synchronize()
    full = (L // 256) * 256 if d == 64 and 0 < L % 256 <= 128 else L    # rows in full pairs
    assert torch.equal(o_s[:, :, :full], o_d[:, :, :full])
    assert torch.equal(l_s[:, :, :full], l_d[:, :, :full])
    if full < L:
        assert (o_s[:, :, full:].float() - o_d[:, :, full:].float()).abs().max().item() <= TOL_O
        assert (l_s[:, :, full:] - l_d[:, :, full:]).abs().max().item() <= TOL_LSE


def test_future_blocks_contribute_nothing(bss):
    L, d = 1024, 64
    n = L // 128
    base = [[a, 0] for a in range(n)]
    extra = [[a, 0, min(n - 1, a + 2), n - 1] for a in range(n)]     # future blocks added
    mk = lambda rows: (np.cumsum([0] + [len(r) for r in rows]).astype(np.int32),
                       np.array([c for r in rows for c in r], np.int32))
    inp = to_cuda(make_inputs(Workload("f", 1, 1, L, d, True, seed=3)))
    a = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], *mk(base), causal=True)
    b = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], *mk(extra), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_bad_entries_are_ignored_and_reported(bss):
    L, d = 512, 64
    rp = np.array([0, 2, 4, 6, 9], np.int32)
    good = np.array([0, 0, 1, 0, 2, 1, 3, 0, 1], np.int32)
    bad = good.copy()
    bad[3] = 57          # out of range: ignored
    bad[8] = -2          # negative: ignored
    inp = to_cuda(make_inputs(Workload("b", 1, 1, L, d, True, seed=8)))
    assert bss.attn_poll_status() == 0
    out = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, bad, causal=True)
    assert bss.attn_poll_status() == bss.ERR_BAD_BLOCKLIST
    rows_wo = [[0, 0], [1], [2, 1], [3, 0]]
    rp2 = np.cumsum([0] + [len(r) for r in rows_wo]).astype(np.int32)
    ci2 = np.array([c for r in rows_wo for c in r], np.int32)
    exp = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp2, ci2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out[0], exp[0]) and torch.equal(out[1], exp[1])


def test_blocksparse_16k_full_size_sampled(bss):
    """B=2 H=16 L'=16320 d=128 with the generated list (empty row 64, partial
    last block), the benchmark's launch configuration; sampled heads and rows."""
    w = SPARSE_16K
    rp, ci = local_global_random_blocklist(w.n_blocks, seed=w.seed)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.all(torch.isneginf(lse[:, :, 64 * 128:65 * 128]))
    assert torch.all(o[:, :, 64 * 128:65 * 128] == 0)
    rows = tile_edge_rows(w.L, n_random=48, seed=2)[::2]
    rows = np.unique(np.concatenate([rows, np.arange(64 * 128 - 2, 65 * 128 + 2)]))
    heads = [(0, 3), (1, 12)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=heads, causal=True, block=128,
                                  row_ptr=rp, col_idx=ci)
    for n_, (b, h) in enumerate(heads):
        compare_forward(o[b, h, rows], lse[b, h, rows], O_ref[n_], l_ref[n_], f"head {(b, h)}")
    assert torch.isfinite(o).all()


@pytest.mark.parametrize("d,causal,repeat", [(128, True, 1), (128, False, 1), (64, True, 1),
                                             (128, True, 4), (128, False, 4)])
def test_persistent_items_odd_tile_count_per_head_lists(bss, d, causal, repeat):
    """More items than SMs (2 x 24 heads x 13 query pairs = 624), so that each
    CTA runs several in turn and prepares the next item's bitmaps while the
    current one runs; 25 query tiles, so that under the causal mask the first
    items (the last pairs) hold a single tile and the CTA hands back the Q
    buffer its empty slot never read; one random list per head, with empty
    rows, duplicates and future blocks.  Whole heads against the oracle, each
    head's items spread over the whole launch; with every entry listed once
    and 4 times over (the same sets)."""
    n = 25
    L = n * 128 - 50
    B, H = 2, 24
    w = Workload("persist", B, H, L, d, causal, seed=31 + d)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    lists = [random_blocklist(n, n, seed=100 + x) for x in range(B * H)]
    lists = [(r * repeat, np.repeat(c, repeat)) for r, c in lists]
    rp = np.zeros((B * H, n + 1), np.int32)
    cis, off = [], 0
    for x, (r, c) in enumerate(lists):
        rp[x] = r + off
        cis.append(c)
        off += len(c)
    ci = np.concatenate(cis).astype(np.int32)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.isfinite(o).all()
    for b, h in ((0, 0), (0, 17), (1, 6), (1, 23)):
        r, c = lists[b * H + h]
        O_ref, l_ref = oracle_forward(cpu, w.scale, heads=[(b, h)], causal=causal, block=128,
                                      row_ptr=r, col_idx=c)
        compare_forward(o[b, h], lse[b, h], O_ref[0], l_ref[0], f"head {(b, h)}")


@pytest.mark.parametrize("repeat", [1, 8])
@pytest.mark.parametrize("causal", [True, False])
def test_odd_and_even_block_counts(bss, causal, repeat):
    """Rows listing 0 to 7 blocks (a lone last block, a lone first block, the
    diagonal alone, the partial last block alone), d=128, whole heads against
    the oracle, with every entry listed once and 8 times over (the same
    sets).  At d=128 a lone last block is scored by itself (an N=128 MMA and
    one V tile)."""
    L, d = 1100, 128                                 # 9 blocks, the last one 76 keys
    n = (L + 127) // 128
    rows = [[], [1], [0, 1], [2, 0, 1], [3], [4, 2, 0, 3, 1], [8], [1, 3, 5, 6, 0, 2, 4],
            [8, 0, 2]]
    if causal:
        rows[6] = [6]
        rows[8] = [8, 7, 6, 5, 4, 3, 2]
    rows = [r * repeat for r in rows]
    rp = np.cumsum([0] + [len(r) for r in rows]).astype(np.int32)
    ci = np.array([c for r in rows for c in r], np.int32)
    w = Workload("odd", 2, 3, L, d, causal, seed=61)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=causal,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=causal, block=128, row_ptr=rp, col_idx=ci)
    compare_forward(o, lse, O_ref, l_ref, f"odd counts causal={causal}")


@pytest.mark.parametrize("n_blocks", [2048, 2049])
def test_longest_key_ranges_at_d128(bss, n_blocks):
    """One head at d=128 with 2048 key blocks (the most one item's bitmap
    covers in the kernel with 256-key score tiles) and 2049 (handed to the
    two-tile kernel, whose bitmaps cover up to 4096 blocks), the last block
    partial; every entry listed twice.  Sampled rows against the oracle, the
    emptied middle block exactly empty."""
    L = n_blocks * 128 - 40
    w = Workload("sparse_long", 1, 1, L, 128, True, seed=n_blocks)
    cpu = make_inputs(w)
    rp, ci = local_global_random_blocklist(n_blocks, seed=n_blocks)
    rp, ci = 2 * rp, np.repeat(ci, 2)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    e = n_blocks // 2
    assert torch.all(torch.isneginf(lse[0, 0, e * 128:(e + 1) * 128]))
    assert torch.all(o[0, 0, e * 128:(e + 1) * 128] == 0)
    rng = np.random.default_rng(n_blocks)
    rows = np.unique(np.concatenate([np.arange(0, 3), np.arange(e * 128 - 2, e * 128 + 2),
                                     np.arange(L - 130, L, 5), rng.integers(0, L, size=24)]))
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, causal=True, block=128, row_ptr=rp,
                                  col_idx=ci)
    compare_forward(o[0, 0, rows], lse[0, 0, rows], O_ref[0, 0], l_ref[0, 0], f"{n_blocks} blocks")
    assert torch.isfinite(o).all()


def test_long_lists_16k_full_size_sampled(bss):
    """B=2 H=16 L'=16320 d=128 with 16 local and 8 random blocks a row (about
    24 entries), causal; sampled heads and rows against the oracle, the
    emptied middle row exactly empty."""
    w = SPARSE_16K
    rp, ci = local_global_random_blocklist(w.n_blocks, seed=w.seed, n_local=16, n_random=8)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert torch.all(torch.isneginf(lse[:, :, 64 * 128:65 * 128]))
    rows = tile_edge_rows(w.L, n_random=48, seed=4)[::2]
    heads = [(0, 5), (1, 9)]
    O_ref, l_ref = oracle_forward(cpu, w.scale, rows=rows, heads=heads, causal=True, block=128,
                                  row_ptr=rp, col_idx=ci)
    for n_, (b, h) in enumerate(heads):
        compare_forward(o[b, h, rows], lse[b, h, rows], O_ref[n_], l_ref[n_], f"head {(b, h)}")
    assert torch.isfinite(o).all()
