"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and builds block lists.  It holds none of
the attention arithmetic: neither the CUDA library nor the CPU oracle is
imported here, and both sides receive exactly the tensors produced below.

Input recipe (every workload):
  * ``torch.Generator('cpu').manual_seed(seed)``; ``torch.randn`` in fp32, drawn
    in the order Q, K, V (then dO for backward workloads), each of shape
    [B, H, L, d]; optionally multiplied by a value scale; rounded to bf16.
  * the oracle receives the bf16 values upcast to fp64, so a comparison measures
    kernel error, not input rounding.

Block lists (the local + global + random pattern named on the block-sparse
attention patterns page, section "Count active blocks and acknowledge the
changed operator"): for query block a, the local blocks a, a-1, a-2, a-3 (those
>= 0), then the global block 0, then two blocks drawn uniformly with
replacement from the earlier blocks 0..a-1 (row 0 draws none) by
``numpy.random.default_rng(seed).integers(0, a)``, in row order.  Raw order and
duplicates are kept; one row (the middle one) is emptied after generation.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

BLOCK = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int
    causal: bool
    seed: int
    value_scale: float = 1.0
    sparse: bool = False
    chunks: int = 1          # split-KV chunks merged afterwards
    backward: bool = False
    description: str = ""
    Lq: Optional[int] = None  # decode-shaped: only the last Lq rows of the draw are queries
    Hkv: Optional[int] = None  # grouped key/value heads (None: Hkv = H)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def n_blocks(self) -> int:
        return (self.L + BLOCK - 1) // BLOCK


# The five workloads of the study, plus the long dense-causal target shape.
DENSE_SMALL = Workload("dense_L256_d64", 1, 1, 256, 64, False, 0,
                       description="dense exact attention, B=1 H=1 L=256 d=64, no mask")
CAUSAL_4K = Workload("causal_B4_H16_L4096_d128", 4, 16, 4096, 128, True, 1,
                     description="causal dense forward, B=4 H=16 L=4096 d=128")
SPARSE_16K = Workload("blocksparse_B2_H16_L16320_d128", 2, 16, 16320, 128, True, 2,
                      sparse=True,
                      description="block-sparse causal forward, local+global+random "
                                  "blocks of 128, L'=16320 (partial last block), one empty row")
SPLITKV_128K = Workload("splitkv_B1_H8_L131072_d128", 1, 8, 131072, 128, True, 3,
                        value_scale=0.5, chunks=8,
                        description="long causal forward, 8 KV chunks merged by the "
                                    "online-softmax combine")
BWD_8K = Workload("fwdbwd_B8_H16_L8192_d64", 8, 16, 8192, 64, True, 4, backward=True,
                  description="causal forward + recompute backward, B=8 H=16 L=8192 d=64")
CAUSAL_16K = Workload("causal_B2_H16_L16384_d128", 2, 16, 16384, 128, True, 1,
                      description="dense causal forward at L=16384, d=128 (B=2 H=16)")

# Decode-shaped split-KV forward (the Ring combine's other use): the queries
# are the last 16 positions of the draw (q_offset = L - 16, causal) against a
# 16384-key cache cut into 2 chunks, so that the 64 heads give 128 work items:
# one wave on the 148 SMs, one item boundary per SM.
DECODE_16K = Workload("decode_B4_H16_Lq16_Lk16384_d128", 4, 16, 16384, 128, True, 5, chunks=2,
                      Lq=16,
                      description="decode-shaped forward: 16 queries at the end of a 16384-key "
                                  "causal cache, 2 KV chunks merged")

# Grouped key/value heads: the L=16384 causal shape with 4 key/value heads, each
# shared by 4 query heads; forward and backward.
GQA_16K = Workload("gqa_B2_H16_Hkv4_L16384_d128", 2, 16, 16384, 128, True, 6, backward=True,
                   Hkv=4,
                   description="causal forward + backward, 16 query heads over 4 shared "
                               "key/value heads, L=16384 d=128")

ALL = [DENSE_SMALL, CAUSAL_4K, SPARSE_16K, SPLITKV_128K, BWD_8K, CAUSAL_16K, DECODE_16K, GQA_16K]
BY_NAME = {w.name: w for w in ALL}


def randn_bf16(shape, seed: int, count: int, value_scale: float = 1.0,
               shapes=None) -> List[torch.Tensor]:
    """``count`` tensors of ``shape`` (or of the listed ``shapes``) drawn in order
    from one seeded CPU generator."""
    g = torch.Generator("cpu").manual_seed(seed)
    out = []
    for shape in (shapes if shapes is not None else [shape] * count):
        t = torch.randn(shape, generator=g, dtype=torch.float32)
        if value_scale != 1.0:
            t = t * value_scale
        out.append(t.to(torch.bfloat16))
    return out


def make_inputs(w: Workload, L: Optional[int] = None, B: Optional[int] = None,
                H: Optional[int] = None, Hkv: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """bf16 CPU tensors q, k, v (and do for backward workloads): q and do
    [B,H,L,d], k and v [B,Hkv,L,d] (Hkv = H unless the workload groups heads).

    ``L``, ``B``, ``H``, ``Hkv`` override the workload's sizes for reduced test
    cases; the distribution and draw order stay the same.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    L = w.L if L is None else L
    Hkv = (w.Hkv if w.Hkv is not None else H) if Hkv is None else Hkv
    n = 4 if w.backward else 3
    qs, kvs = (B, H, L, w.d), (B, Hkv, L, w.d)
    ts = randn_bf16(None, w.seed, n, w.value_scale, shapes=[qs, kvs, kvs, qs][:n])
    names = ["q", "k", "v", "do"][:n]
    out = dict(zip(names, ts))
    if w.Lq is not None:                 # decode-shaped: queries are the last Lq positions
        out["q"] = out["q"][:, :, L - w.Lq:].contiguous()
    return out


def to_f64(t: torch.Tensor) -> np.ndarray:
    """The exact bf16 values as a float64 numpy array."""
    return t.to(torch.float64).numpy()


def local_global_random_blocklist(n_blocks: int, seed: int, n_local: int = 4,
                                  n_random: int = 2, empty_row: Optional[int] = -1
                                  ) -> Tuple[np.ndarray, np.ndarray]:
    """Raw CSR (row_ptr, col_idx) int32 for the local + global + random pattern.

    Entries are kept in generation order, duplicates included.  ``empty_row``
    (-1 = the middle row n//2, None = no empty row) has its list cleared after
    all rows were drawn, so the random stream does not depend on it.
    """
    rng = np.random.default_rng(seed)
    rows: List[List[int]] = []
    for a in range(n_blocks):
        row = [a - t for t in range(n_local) if a - t >= 0]
        row.append(0)
        if a >= 1:
            for _ in range(n_random):
                row.append(int(rng.integers(0, a)))
        rows.append(row)
    if empty_row is not None:
        r = n_blocks // 2 if empty_row == -1 else empty_row
        rows[r] = []
    row_ptr = np.zeros(n_blocks + 1, dtype=np.int32)
    for a, row in enumerate(rows):
        row_ptr[a + 1] = row_ptr[a] + len(row)
    col_idx = np.array([c for row in rows for c in row], dtype=np.int32)
    return row_ptr, col_idx


def random_blocklist(n_qblk: int, n_kblk: int, seed: int, max_per_row: int = 6,
                     p_empty: float = 0.15) -> Tuple[np.ndarray, np.ndarray]:
    """Unstructured raw CSR for tests: random length rows, random order, duplicates."""
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(n_qblk):
        if rng.random() < p_empty:
            rows.append([])
            continue
        k = int(rng.integers(1, max_per_row + 1))
        rows.append([int(x) for x in rng.integers(0, n_kblk, size=k)])
    row_ptr = np.zeros(n_qblk + 1, dtype=np.int32)
    for a, row in enumerate(rows):
        row_ptr[a + 1] = row_ptr[a] + len(row)
    col_idx = np.array([c for row in rows for c in row], dtype=np.int32)
    return row_ptr, col_idx


def chunk_bounds(L: int, chunks: int) -> List[Tuple[int, int]]:
    """Contiguous [start, end) key ranges of (nearly) equal size."""
    step = (L + chunks - 1) // chunks
    return [(s, min(L, s + step)) for s in range(0, L, step)]


def sample_rows(L: int, chunks: int, n: int, seed: int) -> np.ndarray:
    """Rows checked for the long split-KV workload: the edges of every 128-row
    tile around the start, every chunk boundary +-1, the last row, and random
    rows from the workload's numpy stream; sorted and unique."""
    fixed = {0, 1, 127, 128, L - 1}
    for s, _ in chunk_bounds(L, chunks):
        for r in (s - 1, s, s + 1):
            if 0 <= r < L:
                fixed.add(r)
    rng = np.random.default_rng(seed)
    rest = rng.integers(0, L, size=max(0, n - len(fixed)))
    rows = np.unique(np.concatenate([np.array(sorted(fixed)), rest]))
    return rows.astype(np.int64)
