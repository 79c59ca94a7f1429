"""GB300-native exact, causal, block-sparse and chunk-merged softmax attention.

Thin PyTorch-facing binding over the C ABI of ``libbss_attn.so`` (declared in
``include/bss_attn.h``).  PyTorch only provides device memory and the current
CUDA stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: calls fail loudly when the library is not built or
the tensors are not on a CUDA device.

Functions carry the C names: ``attn_fwd``, ``attn_fwd_partial``,
``attn_merge_states``, ``attn_fwd_splitkv``, ``attn_blocklist_normalize``,
``attn_blocklist_stats``, ``attn_fwd_blocksparse``, ``attn_select_blocks``,
``attn_bwd``, ``attn_bwd_blocksparse``, ``attn_bwd_noalloc``, ``attn_poll_status``,
``attn_bwd_time_main``, ``attn_watchdog_selftest``, ``attn_probe_ex2_rate``.  Each
call runs on the
device of its tensors and on that device's current stream.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

from . import _lib

__all__ = [
    "AttnError", "attn_fwd", "attn_fwd_partial", "attn_merge_states", "attn_fwd_splitkv",
    "attn_fwd_splitkv_workspace_bytes", "attn_blocklist_normalize", "attn_blocklist_stats",
    "attn_fwd_blocksparse", "attn_select_blocks", "attn_select_blocks_workspace_bytes",
    "attn_select_blocks_nnz", "attn_bwd", "attn_bwd_workspace_bytes", "attn_bwd_blocksparse",
    "attn_bwd_blocksparse_workspace_bytes", "attn_bwd_noalloc", "attn_poll_status",
    "attn_bwd_time_main", "attn_watchdog_selftest", "attn_probe_ex2_rate", "library",
]

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_BAD_BLOCKLIST = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_WORKSPACE = 6


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _lib.load()
        name = lib.attn_status_string(status).decode()
        detail = lib.attn_last_error_message().decode()
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))
        self.status = status
        self.name = name


def library():
    """The loaded ctypes library (raises if it has not been built)."""
    return _lib.load()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise AttnError(status, where)


def _stream_of(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: Sequence[int]) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _scale(scale: Optional[float], d: int) -> float:
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = False,
             scale: Optional[float] = None, q_offset: int = 0, k_offset: int = 0,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None
             ) -> Tuple[torch.Tensor, torch.Tensor]:
    """O [B,H,Lq,d] bf16 and LSE [B,H,Lq] fp32 of exact (optionally causal) attention.
    k and v may have fewer heads than q (grouped query heads)."""
    B, H, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    _need(q, "q", torch.bfloat16, (B, H, Lq, d))
    _need(k, "k", torch.bfloat16, (B, Hkv, Lk, d))
    _need(v, "v", torch.bfloat16, (B, Hkv, Lk, d))
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Lq), device=q.device, dtype=torch.float32) if lse is None else lse
    _need(out, "out", torch.bfloat16, (B, H, Lq, d))
    _need(lse, "lse", torch.float32, (B, H, Lq))
    with torch.cuda.device(q.device):
        st = _lib.load().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, H, Hkv, Lq, Lk, d, _scale(scale, d), int(causal),
                                  int(q_offset), int(k_offset), _stream_of(q))
    _check(st, "attn_fwd")
    return out, lse


def attn_fwd_partial(q, k, v, *, causal: bool = False, scale: Optional[float] = None,
                     q_offset: int = 0, k_offset: int = 0, m=None, l=None, acc=None):
    """Unnormalised state (m, l, acc) of the query rows over one KV chunk."""
    B, H, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    _need(q, "q", torch.bfloat16, (B, H, Lq, d))
    _need(k, "k", torch.bfloat16, (B, Hkv, Lk, d))
    _need(v, "v", torch.bfloat16, (B, Hkv, Lk, d))
    dev = q.device
    m = torch.empty((B, H, Lq), device=dev, dtype=torch.float32) if m is None else m
    l = torch.empty((B, H, Lq), device=dev, dtype=torch.float32) if l is None else l
    acc = torch.empty((B, H, Lq, d), device=dev, dtype=torch.float32) if acc is None else acc
    _need(m, "m", torch.float32, (B, H, Lq))
    _need(l, "l", torch.float32, (B, H, Lq))
    _need(acc, "acc", torch.float32, (B, H, Lq, d))
    with torch.cuda.device(q.device):
        st = _lib.load().attn_fwd_partial(q.data_ptr(), k.data_ptr(), v.data_ptr(), m.data_ptr(),
                                          l.data_ptr(), acc.data_ptr(), B, H, Hkv, Lq, Lk, d,
                                          _scale(scale, d), int(causal), int(q_offset), int(k_offset),
                                          _stream_of(q))
    _check(st, "attn_fwd_partial")
    return m, l, acc


def attn_merge_states(m: torch.Tensor, l: torch.Tensor, acc: torch.Tensor, *, out=None, lse=None):
    """Merge C chunk states (m, l [C,B,H,L]; acc [C,B,H,L,d]) into O (bf16) and LSE."""
    C, B, H, L, d = acc.shape
    _need(m, "m", torch.float32, (C, B, H, L))
    _need(l, "l", torch.float32, (C, B, H, L))
    _need(acc, "acc", torch.float32, (C, B, H, L, d))
    out = torch.empty((B, H, L, d), device=acc.device, dtype=torch.bfloat16) if out is None else out
    lse = torch.empty((B, H, L), device=acc.device, dtype=torch.float32) if lse is None else lse
    _need(out, "out", torch.bfloat16, (B, H, L, d))
    _need(lse, "lse", torch.float32, (B, H, L))
    with torch.cuda.device(acc.device):
        st = _lib.load().attn_merge_states(C, m.data_ptr(), l.data_ptr(), acc.data_ptr(),
                                           out.data_ptr(), lse.data_ptr(), B, H, L, d,
                                           _stream_of(acc))
    _check(st, "attn_merge_states")
    return out, lse


def attn_fwd_splitkv_workspace_bytes(B: int, H: int, Lq: int, Lk: int, d: int, chunks: int) -> int:
    return int(_lib.load().attn_fwd_splitkv_workspace_bytes(B, H, Lq, Lk, d, chunks))


def attn_fwd_splitkv(q, k, v, chunks: int, *, causal: bool = False, scale: Optional[float] = None,
                     q_offset: int = 0, k_offset: int = 0, workspace: Optional[torch.Tensor] = None,
                     out=None, lse=None):
    """Exact attention with the keys cut into ``chunks`` chunks (each a multiple of
    128 keys) whose partial states are computed in one launch and merged: the
    split-KV / decode-shaped forward (the Ring-Attention combine on one GPU)."""
    B, H, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    _need(q, "q", torch.bfloat16, (B, H, Lq, d))
    _need(k, "k", torch.bfloat16, (B, Hkv, Lk, d))
    _need(v, "v", torch.bfloat16, (B, Hkv, Lk, d))
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Lq), device=q.device, dtype=torch.float32) if lse is None else lse
    _need(out, "out", torch.bfloat16, (B, H, Lq, d))
    _need(lse, "lse", torch.float32, (B, H, Lq))
    nbytes = attn_fwd_splitkv_workspace_bytes(B, H, Lq, Lk, d, chunks)
    if workspace is None:
        workspace = torch.empty(max(16, nbytes), device=q.device, dtype=torch.uint8)
    with torch.cuda.device(q.device):
        st = _lib.load().attn_fwd_splitkv(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            workspace.data_ptr(), workspace.numel() * workspace.element_size(), B, H, Hkv, Lq, Lk,
            d, _scale(scale, d), int(causal), int(q_offset), int(k_offset), int(chunks), _stream_of(q))
    _check(st, "attn_fwd_splitkv")
    return out, lse


def attn_select_blocks_workspace_bytes(B: int, H: int, L: int, d: int) -> int:
    return int(_lib.load().attn_select_blocks_workspace_bytes(B, H, L, d))


def attn_select_blocks_nnz(L: int, top_r: int, local_blocks: int, causal: bool,
                           n_lists: int = 1) -> int:
    """Entries of the lists attn_select_blocks writes (all lists together)."""
    return int(_lib.load().attn_select_blocks_nnz(L, top_r, local_blocks, int(causal), n_lists))


def attn_select_blocks(q, k, top_r: int, *, local_blocks: int = 1, causal: bool = True,
                       n_lists: int = 1, scale: Optional[float] = None, block: int = 128,
                       workspace: Optional[torch.Tensor] = None):
    """Block lists from mean-pooled scores: (row_ptr [n_lists, n+1], col_idx) int32 on
    q's device, the input of attn_fwd_blocksparse / attn_bwd_blocksparse."""
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    _need(q, "q", torch.bfloat16, (B, H, L, d))
    _need(k, "k", torch.bfloat16, (B, Hkv, L, d))
    lib = _lib.load()
    n = (L + block - 1) // block
    nnz = attn_select_blocks_nnz(L, top_r, local_blocks, causal, n_lists)
    if nnz < 0:
        raise AttnError(ERR_INVALID_ARG, "attn_select_blocks: invalid arguments")
    row_ptr = torch.empty((n_lists, n + 1), device=q.device, dtype=torch.int32)
    col_idx = torch.empty(max(1, nnz), device=q.device, dtype=torch.int32)
    nbytes = attn_select_blocks_workspace_bytes(B, H, L, d)
    if workspace is None:
        workspace = torch.empty(max(16, nbytes), device=q.device, dtype=torch.uint8)
    with torch.cuda.device(q.device):
        st = lib.attn_select_blocks(q.data_ptr(), k.data_ptr(), B, H, Hkv, L, d, _scale(scale, d),
                                    int(causal), int(block), int(top_r), int(local_blocks),
                                    int(n_lists), row_ptr.data_ptr(), col_idx.data_ptr(),
                                    workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                    _stream_of(q))
    _check(st, "attn_select_blocks")
    return row_ptr, col_idx[:nnz]


def attn_blocklist_normalize(row_ptr, col_idx, n_kblk: int) -> Tuple[np.ndarray, np.ndarray]:
    """Canonical CSR (ascending, duplicates removed), computed by the library on the host."""
    rp = np.ascontiguousarray(np.asarray(row_ptr, dtype=np.int32))
    ci = np.ascontiguousarray(np.asarray(col_idx, dtype=np.int32))
    n_qblk = len(rp) - 1
    out_rp = np.zeros(n_qblk + 1, dtype=np.int32)
    out_ci = np.zeros(max(1, len(ci)), dtype=np.int32)
    nnz = np.zeros(1, dtype=np.int32)
    st = _lib.load().attn_blocklist_normalize(
        rp.ctypes.data, ci.ctypes.data if len(ci) else None, n_qblk, n_kblk, out_rp.ctypes.data,
        out_ci.ctypes.data, nnz.ctypes.data)
    _check(st, "attn_blocklist_normalize")
    return out_rp, out_ci[:int(nnz[0])].copy()


def _csr_on_device(row_ptr, col_idx, device):
    """int32 CSR on the tensors' device as (row_ptr, col_idx, nnz, n_lists,
    n_qblk).  A 1-D row_ptr is one list shared by every head; a 2-D
    [n_lists, n_qblk + 1] row_ptr holds one list per group of heads, each
    with offsets into the one col_idx.  An empty col_idx gets a one-element
    placeholder (never read) so that its pointer is valid."""
    rp = torch.as_tensor(np.asarray(row_ptr, dtype=np.int32) if not torch.is_tensor(row_ptr)
                         else row_ptr).to(device=device, dtype=torch.int32).contiguous()
    ci = torch.as_tensor(np.asarray(col_idx, dtype=np.int32) if not torch.is_tensor(col_idx)
                         else col_idx).to(device=device, dtype=torch.int32).contiguous()
    n_lists = 1 if rp.dim() == 1 else rp.shape[0]
    n_qblk = rp.shape[-1] - 1
    if ci.numel() == 0:
        return rp, torch.zeros(1, device=device, dtype=torch.int32), 0, n_lists, n_qblk
    return rp, ci, ci.numel(), n_lists, n_qblk


def attn_fwd_blocksparse(q, k, v, row_ptr, col_idx, *, causal: bool = False,
                         scale: Optional[float] = None, block: int = 128, out=None, lse=None):
    """Attention over per-query-block CSR lists of key blocks (raw form accepted)."""
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    _need(q, "q", torch.bfloat16, (B, H, L, d))
    _need(k, "k", torch.bfloat16, (B, Hkv, L, d))
    _need(v, "v", torch.bfloat16, (B, Hkv, L, d))
    rp, ci, nnz, n_lists, n_qblk = _csr_on_device(row_ptr, col_idx, q.device)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, L), device=q.device, dtype=torch.float32) if lse is None else lse
    _need(out, "out", torch.bfloat16, (B, H, L, d))
    _need(lse, "lse", torch.float32, (B, H, L))
    with torch.cuda.device(q.device):
        st = _lib.load().attn_fwd_blocksparse(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Hkv, L,
            d, _scale(scale, d), int(causal), int(block), rp.data_ptr(), ci.data_ptr(), n_lists, n_qblk,
            nnz, _stream_of(q))
    _check(st, "attn_fwd_blocksparse")
    return out, lse


STATS_FIELDS = ("listed", "executed", "future", "pairs")


def attn_blocklist_stats(row_ptr, col_idx, L: int, *, causal: bool = False, block: int = 128,
                         device=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """What each block list asks for, counted on the GPU: int64 [n_lists, 4] on the
    device with, per list, the listed (query block, key block) pairs (duplicates
    once), the executed tiles, the listed blocks wholly in the causal future
    (skipped by the kernels) and the logical allowed pairs (``STATS_FIELDS``)."""
    dev = (row_ptr.device if torch.is_tensor(row_ptr) and row_ptr.is_cuda else
           torch.device("cuda", torch.cuda.current_device()) if device is None else device)
    rp, ci, nnz, n_lists, n_qblk = _csr_on_device(row_ptr, col_idx, dev)
    out = torch.empty((n_lists, 4), device=dev, dtype=torch.int64) if out is None else out
    _need(out, "out", torch.int64, (n_lists, 4))
    with torch.cuda.device(dev):
        st = _lib.load().attn_blocklist_stats(rp.data_ptr(), ci.data_ptr(), n_lists, n_qblk, nnz,
                                              int(L), int(causal), int(block), out.data_ptr(),
                                              torch.cuda.current_stream(dev).cuda_stream)
    _check(st, "attn_blocklist_stats")
    return out


def attn_bwd_workspace_bytes(B: int, H: int, L: int, d: int) -> int:
    return int(_lib.load().attn_bwd_workspace_bytes(B, H, L, d))


def attn_bwd(q, k, v, o, lse, dout, *, causal: bool = False, scale: Optional[float] = None,
             workspace: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None, delta=None):
    """Gradients (dq, dk, dv) bf16 and delta = rowsum(dO * O) fp32, by recomputation."""
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    for name, t in (("q", q), ("o", o), ("dout", dout)):
        _need(t, name, torch.bfloat16, (B, H, L, d))
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, (B, Hkv, L, d))
    _need(lse, "lse", torch.float32, (B, H, L))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    delta = torch.empty((B, H, L), device=q.device, dtype=torch.float32) if delta is None else delta
    nbytes = attn_bwd_workspace_bytes(B, H, L, d)
    if workspace is None:
        workspace = torch.empty(max(16, nbytes), device=q.device, dtype=torch.uint8)
    with torch.cuda.device(q.device):
        st = _lib.load().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), delta.data_ptr(), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), B, H, Hkv, L,
                                  d, _scale(scale, d), int(causal), _stream_of(q))
    _check(st, "attn_bwd")
    return dq, dk, dv, delta


def attn_bwd_blocksparse_workspace_bytes(B: int, H: int, L: int, d: int, n_lists: int = 1) -> int:
    return int(_lib.load().attn_bwd_blocksparse_workspace_bytes(B, H, L, d, n_lists))


def attn_bwd_blocksparse(q, k, v, o, lse, dout, row_ptr, col_idx, *, causal: bool = False,
                         scale: Optional[float] = None, block: int = 128,
                         workspace: Optional[torch.Tensor] = None, dq=None, dk=None, dv=None,
                         delta=None):
    """Gradients of attn_fwd_blocksparse with the same block list (raw CSR accepted)."""
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    for name, t in (("q", q), ("o", o), ("dout", dout)):
        _need(t, name, torch.bfloat16, (B, H, L, d))
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, (B, Hkv, L, d))
    _need(lse, "lse", torch.float32, (B, H, L))
    rp, ci, nnz, n_lists, n_qblk = _csr_on_device(row_ptr, col_idx, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    delta = torch.empty((B, H, L), device=q.device, dtype=torch.float32) if delta is None else delta
    nbytes = attn_bwd_blocksparse_workspace_bytes(B, H, L, d, n_lists)
    if workspace is None:
        workspace = torch.empty(max(16, nbytes), device=q.device, dtype=torch.uint8)
    with torch.cuda.device(q.device):
        st = _lib.load().attn_bwd_blocksparse(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), delta.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), B, H, Hkv, L, d, _scale(scale, d),
            int(causal), int(block), rp.data_ptr(), ci.data_ptr(), n_lists, n_qblk, nnz, _stream_of(q))
    _check(st, "attn_bwd_blocksparse")
    return dq, dk, dv, delta


NOALLOC_SCRATCH_FLOATS = 8 << 20


def attn_bwd_noalloc(q, k, v, o, lse, dout, *, causal: bool = False,
                     scale: Optional[float] = None, dq=None, dk=None, dv=None, delta=None):
    """attn_bwd without a workspace, for callers that cannot allocate device memory:
    the library keeps the fp32 dQ accumulator in a static 32 MiB device array
    (B*H*L*d <= 8388608).  Calls share that array, so calls that overlap on the GPU
    race; the first call on a device should come before any stream capture.
    Outputs not given are allocated here by PyTorch, as for every other binding."""
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    for name, t in (("q", q), ("o", o), ("dout", dout)):
        _need(t, name, torch.bfloat16, (B, H, L, d))
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, (B, Hkv, L, d))
    _need(lse, "lse", torch.float32, (B, H, L))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    delta = torch.empty((B, H, L), device=q.device, dtype=torch.float32) if delta is None else delta
    with torch.cuda.device(q.device):
        st = _lib.load().attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                          lse.data_ptr(), dout.data_ptr(), dq.data_ptr(),
                                          dk.data_ptr(), dv.data_ptr(), delta.data_ptr(), B, H, Hkv,
                                          L, d, _scale(scale, d), int(causal), _stream_of(q))
    _check(st, "attn_bwd_noalloc")
    return dq, dk, dv, delta


def attn_poll_status(device=None) -> int:
    """Synchronise the device's current stream and return (and clear) the
    kernels' error word of that device (default: the current device)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        return int(_lib.load().attn_poll_status(stream))


def attn_bwd_time_main(begin: Optional[torch.cuda.Event] = None,
                       end: Optional[torch.cuda.Event] = None) -> None:
    """Record ``begin`` and ``end`` (torch.cuda.Event, enable_timing=True, on
    the device of the calls) just before and after the main kernel of every
    following backward call, so that ``begin.elapsed_time(end)`` is that
    kernel's own duration; ``attn_bwd_time_main()`` stops it.  Stop it before
    the events are dropped."""
    def handle(e):
        if e is None:
            return None
        if not e.cuda_event:       # the CUDA event is created at its first record
            e.record()
        return e.cuda_event
    _check(_lib.load().attn_bwd_time_main(handle(begin), handle(end)), "attn_bwd_time_main")


def attn_probe_ex2_rate(blocks: int, iters: int, sink: Optional[torch.Tensor] = None,
                        device=None) -> int:
    """Launch the exponential-rate kernel on the current stream; returns the
    number of exponentials it evaluates (the caller times the launch)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    sink = torch.zeros(1, device=dev, dtype=torch.float32) if sink is None else sink
    stream = torch.cuda.current_stream(dev).cuda_stream
    _check(_lib.load().attn_probe_ex2_rate(sink.data_ptr(), int(blocks), int(iters), stream),
           "attn_probe_ex2_rate")
    return int(blocks) * 256 * 8 * int(iters)


def attn_watchdog_selftest(timeout_cycles: int = 1 << 20, device=None) -> None:
    stream = torch.cuda.current_stream(device).cuda_stream
    _check(_lib.load().attn_watchdog_selftest(int(timeout_cycles), stream), "attn_watchdog_selftest")
