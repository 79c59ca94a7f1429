"""attn_blocklist_stats on the GPU against the oracle's pinned block-list
accounting: listed blocks (duplicates once), executed tiles, listed blocks
wholly in the causal future (flagged, not rejected) and logical allowed pairs
(block-sparse attention patterns page, 'Count active blocks and acknowledge the
changed operator').  Integer work: the counts must match exactly."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import compare_forward, oracle_forward, to_cuda
from workloads import (SPARSE_16K, Workload, local_global_random_blocklist, make_inputs,
                       random_blocklist)

pytestmark = pytest.mark.gpu

FIELDS = ("listed", "executed", "future", "pairs")


@pytest.fixture(scope="module")
def bss():
    import block_sparse_softmax_gb300 as m
    m.library()
    return m


def _expect(rp, ci, L, causal):
    s = oracle.blocklist_stats(rp, ci, L, causal=causal)
    return [s[f] for f in FIELDS]


@pytest.mark.parametrize("L,causal,seed", [(1000, True, 0), (1000, False, 1), (129, True, 2),
                                           (4096, True, 3), (300, True, 4), (1, True, 5)])
def test_random_lists_match_the_oracle(bss, L, causal, seed):
    n = (L + 127) // 128
    rp, ci = random_blocklist(n, n, seed=seed)          # future blocks, duplicates, empty rows
    got = bss.attn_blocklist_stats(rp, ci, L, causal=causal)
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert got.cpu().tolist() == [_expect(rp, ci, L, causal)]


def test_block_sparse_workload_list_with_added_future_blocks(bss):
    """The L' = 16320 local + global + random list, then the same list with two
    future blocks appended to every non-empty row (duplicated once more): the
    future count grows, the executed tiles and the pairs do not."""
    L = SPARSE_16K.L
    n = SPARSE_16K.n_blocks
    rp, ci = local_global_random_blocklist(n, seed=2)
    rows = [list(ci[rp[a]:rp[a + 1]]) for a in range(n)]
    rows2 = [r + ([a + 1, min(n - 1, a + 5), a + 1] if r and a + 1 < n else []) for a, r in
             enumerate(rows)]
    rp2 = np.zeros(n + 1, np.int32)
    for a, r in enumerate(rows2):
        rp2[a + 1] = rp2[a] + len(r)
    ci2 = np.array([c for r in rows2 for c in r], np.int32)
    got = bss.attn_blocklist_stats(rp, ci, L, causal=True).cpu().tolist()[0]
    got2 = bss.attn_blocklist_stats(rp2, ci2, L, causal=True).cpu().tolist()[0]
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert got == _expect(rp, ci, L, True)
    assert got2 == _expect(rp2, ci2, L, True)
    assert got[2] == 0 and got2[2] > 0
    assert got2[1] == got[1] and got2[3] == got[3]


def test_one_list_per_head(bss):
    L, lists = 700, 6
    n = (L + 127) // 128
    per = [random_blocklist(n, n, seed=20 + i) for i in range(lists)]
    rp = np.zeros((lists, n + 1), np.int32)
    cis = []
    off = 0
    for i, (r, c) in enumerate(per):
        rp[i] = r + off
        cis.append(c)
        off += len(c)
    ci = np.concatenate(cis).astype(np.int32)
    got = bss.attn_blocklist_stats(rp, ci, L, causal=True).cpu().tolist()
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    assert got == [_expect(r, c, L, True) for r, c in per]


def test_future_blocks_contribute_nothing_to_the_forward(bss):
    """A list whose rows also name future blocks gives the forward of the list
    without them (the oracle's mask drops them by the token rule)."""
    L, d = 900, 64
    n = (L + 127) // 128
    w = Workload("fut", 1, 2, L, d, True, seed=41)
    cpu = make_inputs(w)
    inp = to_cuda(cpu)
    rows = [[a, 0, min(n - 1, a + 2), a // 2] for a in range(n)]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    ci = np.array([c for r in rows for c in r], np.int32)
    o, lse = bss.attn_fwd_blocksparse(inp["q"], inp["k"], inp["v"], rp, ci, causal=True,
                                      scale=w.scale)
    st = bss.attn_blocklist_stats(rp, ci, L, causal=True).cpu().tolist()[0]
    torch.cuda.synchronize()
    assert bss.attn_poll_status() == 0
    O_ref, l_ref = oracle_forward(cpu, w.scale, causal=True, block=128, row_ptr=rp, col_idx=ci)
    compare_forward(o, lse, O_ref, l_ref, "list with future blocks")
    assert st == _expect(rp, ci, L, True) and st[2] == n - 1


def test_malformed_entries_are_reported_and_skipped(bss):
    L = 512
    rp = np.array([0, 2, 4, 6, 8], np.int32)
    ci = np.array([0, 9, 1, -1, 2, 1, 3, 3], np.int32)      # 9 and -1 are out of range
    got = bss.attn_blocklist_stats(rp, ci, L, causal=True).cpu().tolist()[0]
    assert bss.attn_poll_status() == 3                     # ATTN_ERR_BAD_BLOCKLIST
    good_rp = np.array([0, 1, 2, 4, 5], np.int32)
    good_ci = np.array([0, 1, 2, 1, 3], np.int32)
    assert got == _expect(good_rp, good_ci, L, True)


def test_empty_sequence_gives_zero_counts(bss):
    out = bss.attn_blocklist_stats(np.zeros(1, np.int32), np.zeros(0, np.int32), 0, causal=True)
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [[0, 0, 0, 0]]
