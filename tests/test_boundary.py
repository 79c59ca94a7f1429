"""The C ABI without a GPU: the library loads, exports every function the header
declares, normalises block lists exactly as the oracle's set semantics say,
and rejects bad arguments with status codes before touching the device."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from workloads import local_global_random_blocklist, random_blocklist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    from block_sparse_softmax_gb300 import build
    build.build()
    from block_sparse_softmax_gb300 import _lib
    return _lib.load()


def _declared_functions():
    names = []
    for f in os.listdir(HEADER_DIR):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \t\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("attn_fwd", "attn_fwd_partial", "attn_merge_states", "attn_fwd_blocksparse",
                     "attn_blocklist_normalize", "attn_bwd", "attn_bwd_workspace_bytes",
                     "attn_poll_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from block_sparse_softmax_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for name in _declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None
    # the binding wraps exactly the declared set
    from block_sparse_softmax_gb300 import _lib
    assert sorted(_lib.exported_names()) == _declared_functions()


def test_status_strings_and_version(lib):
    assert lib.attn_status_string(0) == b"ATTN_OK"
    assert lib.attn_status_string(3) == b"ATTN_ERR_BAD_BLOCKLIST"
    assert lib.attn_status_string(99) == b"ATTN_ERR_UNKNOWN"
    assert lib.attn_version() >= 100


def _normalize(lib, rp, ci, n_kblk):
    rp = np.ascontiguousarray(rp, dtype=np.int32)
    ci = np.ascontiguousarray(ci, dtype=np.int32)
    out_rp = np.zeros_like(rp)
    out_ci = np.zeros(max(1, len(ci)), dtype=np.int32)
    nnz = np.zeros(1, dtype=np.int32)
    st = lib.attn_blocklist_normalize(rp.ctypes.data, ci.ctypes.data if len(ci) else None,
                                      len(rp) - 1, n_kblk, out_rp.ctypes.data, out_ci.ctypes.data,
                                      nnz.ctypes.data)
    return st, out_rp, out_ci[:nnz[0]]


@pytest.mark.parametrize("seed", range(6))
def test_blocklist_normalize_matches_oracle_exactly(lib, seed):
    if seed == 0:
        rp, ci = local_global_random_blocklist(128, seed=2)
        nk = 128
    else:
        nk = 3 + 7 * seed
        rp, ci = random_blocklist(nk + seed, nk, seed=seed, max_per_row=9)
    st, out_rp, out_ci = _normalize(lib, rp, ci, nk)
    assert st == 0
    ref_rp, ref_ci = oracle.blocklist_normalize(rp, ci, nk)
    assert np.array_equal(out_rp, ref_rp)
    assert np.array_equal(out_ci, ref_ci)
    # the realised block mask equals the oracle's set, row by row
    sets = oracle.blocklist_sets(rp, ci, nk)
    for a, s in enumerate(sets):
        assert set(out_ci[out_rp[a]:out_rp[a + 1]].tolist()) == s


@pytest.mark.parametrize("rp,ci", [
    ([0, 2, 1], [0, 1]),
    ([0, 1], [4]),
    ([0, 1], [-1]),
    ([1, 2], [0, 1]),
])
def test_blocklist_normalize_rejects_malformed(lib, rp, ci):
    st, _, _ = _normalize(lib, np.array(rp), np.array(ci), 4)
    assert st == 3


def test_argument_errors_return_codes_before_any_device_work(lib):
    P = ctypes.c_void_p(16 * 1000)       # aligned dummy addresses, never dereferenced
    bad = ctypes.c_void_p(16 * 1000 + 2)
    args = lambda q=P, d=64, scale=0.125, B=1, H=1, Hkv=1: (q, P, P, P, P, B, H, Hkv, 256, 256, d, scale,
                                                            0, 0, 0, None)
    assert lib.attn_fwd(*args(d=96)) == 2                 # unsupported head dim
    assert lib.attn_fwd(*args(q=None)) == 1               # null pointer
    assert lib.attn_fwd(*args(q=bad)) == 1                # misaligned pointer
    assert lib.attn_fwd(*args(scale=float("nan"))) == 1   # non-finite scale
    assert lib.attn_fwd(*args(scale=-1.0)) == 1           # non-positive scale
    assert lib.attn_fwd(*args(B=0)) == 1                  # empty batch
    assert lib.attn_fwd(*args(H=6, Hkv=4)) == 1           # K/V heads must divide the query heads
    assert lib.attn_fwd(*args(H=6, Hkv=0)) == 1
    assert lib.attn_fwd(*args(H=2, Hkv=3)) == 1
    # block size other than 128, CSR row count mismatch, too many key blocks
    assert lib.attn_fwd_blocksparse(P, P, P, P, P, 1, 1, 1, 256, 64, 0.125, 1, 64, P, P, 1, 2, 4,
                                    None) == 2
    assert lib.attn_fwd_blocksparse(P, P, P, P, P, 1, 1, 1, 256, 64, 0.125, 1, 128, P, P, 1, 3, 4,
                                    None) == 3
    assert lib.attn_fwd_blocksparse(P, P, P, P, P, 1, 1, 1, 4097 * 128, 64, 0.125, 1, 128, P, P, 1,
                                    4097, 4, None) == 2
    # lists must divide the B*H heads into equal groups
    assert lib.attn_fwd_blocksparse(P, P, P, P, P, 2, 3, 3, 256, 64, 0.125, 1, 128, P, P, 4, 2, 4,
                                    None) == 3
    # merge: chunk count out of range
    assert lib.attn_merge_states(0, P, P, P, P, P, 1, 1, 16, 64, None) == 1
    assert lib.attn_merge_states(65, P, P, P, P, P, 1, 1, 16, 64, None) == 1
    # backward: workspace too small
    ws = lib.attn_bwd_workspace_bytes(2, 3, 100, 64)
    assert ws == 2 * 3 * 100 * 64 * 4
    assert lib.attn_bwd(P, P, P, P, P, P, P, P, P, P, P, ws - 4, 2, 3, 3, 100, 64, 0.125, 1, None) == 6
    # split-KV forward: chunks of ceil(Lk / n) keys rounded up to 128; workspace =
    # acc | m | l of every chunk, each part at a 256-byte boundary
    wsk = lib.attn_fwd_splitkv_workspace_bytes(2, 3, 100, 1000, 64, 4)
    assert wsk == 4 * 600 * 64 * 4 + 2 * 9728
    assert lib.attn_fwd_splitkv_workspace_bytes(2, 3, 100, 1000, 64, 65) == 0
    kv = lambda n=4, ws_=wsk: (P, P, P, P, P, P, ws_, 2, 3, 1, 100, 1000, 64, 0.125, 1, 900, 0, n,
                                  None)
    assert lib.attn_fwd_splitkv(*kv(n=0)) == 1                   # chunk count out of range
    assert lib.attn_fwd_splitkv(*kv(n=65)) == 1
    assert lib.attn_fwd_splitkv(*kv(ws_=wsk - 4)) == 6           # workspace too small
    # block-sparse backward: workspace = accumulator (256-byte aligned) + bitmap
    # of ceil(L/128) columns of ceil(ceil(L/128)/32) words per list (256-byte
    # aligned) + the key tiles' launch order (B*H*ceil(L/128) int32)
    up = lambda x: ((x + 255) // 256) * 256
    wss = lib.attn_bwd_blocksparse_workspace_bytes(2, 3, 1000, 64, 1)
    acc = 2 * 3 * 1000 * 64 * 4
    assert wss == up(acc) + up(8 * 1 * 4) + 2 * 3 * 8 * 4
    assert lib.attn_bwd_blocksparse_workspace_bytes(2, 3, 1000, 64, 6) == (
        up(acc) + up(6 * 8 * 1 * 4) + 2 * 3 * 8 * 4)
    assert lib.attn_bwd_blocksparse_workspace_bytes(1, 2, 9000, 64, 2) == (
        up(2 * 9000 * 64 * 4) + up(2 * 71 * 3 * 4) + 2 * 71 * 4)
    assert lib.attn_bwd_blocksparse_workspace_bytes(2, 3, 1000, 64, 4) == 0   # 4 does not divide 6
    sp = lambda block=128, nq=8, ws_=wss, rp=P: (P, P, P, P, P, P, P, P, P, P, P, ws_, 2, 3, 3,
                                                 1000, 64, 0.125, 1, block, rp, P, 1, nq, 4, None)
    assert lib.attn_bwd_blocksparse(*sp(block=64)) == 2          # block size other than 128
    assert lib.attn_bwd_blocksparse(*sp(nq=7)) == 3              # CSR row count mismatch
    assert lib.attn_bwd_blocksparse(*sp(rp=None)) == 1           # missing row_ptr
    assert lib.attn_bwd_blocksparse(*sp(ws_=wss - 4)) == 6       # workspace too small
    # main-kernel timing hook: both events or neither (no device work)
    assert lib.attn_bwd_time_main(P, None) == 1
    assert lib.attn_bwd_time_main(None, P) == 1
    assert lib.attn_bwd_time_main(None, None) == 0
    # exponential-rate probe: sink and sizes
    assert lib.attn_probe_ex2_rate(None, 8, 16, None) == 1
    assert lib.attn_probe_ex2_rate(bad, 8, 16, None) == 1        # misaligned sink
    assert lib.attn_probe_ex2_rate(P, 0, 16, None) == 1
    assert lib.attn_probe_ex2_rate(P, 8, 0, None) == 1


def test_binding_fails_loudly_on_cpu_tensors():
    import torch
    import block_sparse_softmax_gb300 as bss
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        bss.attn_fwd(q, q, q)


@pytest.mark.parametrize("L,top_r,local,causal,n_lists", [
    (1000, 2, 3, True, 1), (1000, 2, 3, False, 2), (129, 4, 1, True, 1), (600, 0, 2, True, 3),
    (900, 9, 0, False, 1), (2560, 4, 4, True, 2), (128, 3, 4, True, 1)])
def test_select_entry_count_matches_the_oracle(lib, L, top_r, local, causal, n_lists):
    """The selector's list sizes do not depend on the scores: the library's
    closed-form count equals the entries of the oracle's lists."""
    import numpy as np
    from oracle.select import select_blocks
    rng = np.random.default_rng(L + top_r)
    q = rng.standard_normal((1, 6, L, 8)).astype(np.float32)
    k = rng.standard_normal((1, 3, L, 8)).astype(np.float32)
    _, col_idx, _ = select_blocks(q, k, 0.35, top_r=top_r, local=local, causal=causal,
                                  n_lists=n_lists)
    assert lib.attn_select_blocks_nnz(L, top_r, local, int(causal), n_lists) == len(col_idx)
    assert lib.attn_select_blocks_nnz(L, top_r, local, int(causal), 0) == -1
