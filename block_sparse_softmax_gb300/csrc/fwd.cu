// Fused attention forward for sm_103a: dense, causal, block-sparse, and the
// partial-state (split-KV) variant, in one warp-specialised kernel.
//
// What it computes ("Exact Blocks, Rings, and Sparsity", section 2, 'What the
// forward kernel keeps on chip'; "FlashAttention: Fast and Memory Efficient
// Exact Attention with IO Awareness", section 5.2): a query tile stays on chip
// while K/V tiles stream past; each 128x128 score tile is folded into the
// running state (m, l, A) and discarded, so S and P never reach HBM.
//
// How it is laid out on the SM (a GB300 design, not the pages' Triton one):
//   * a work item is TWO consecutive 128-row query tiles of one (b, h) that
//     share a single K/V stream: each K/V tile is loaded once for 256 rows;
//   * the kernel is persistent: one CTA per SM takes item after item, handed
//     out greedily by the hardware's cluster launch control (the CTA cancels a
//     not-yet-started CTA of the grid and does its item), so set-up is paid
//     once and one item's epilogue overlaps the next item's loads and MMAs;
//   * warp 0 issues TMA loads (128-byte swizzled boxes of 128 rows x 64 d) into
//     a ring of K and V stages and schedules items; warp 1 (one thread) issues
//     every tcgen05.mma; in a block-sparse launch warp 3 claims the next item
//     and builds its bitmaps; warpgroups 1 and 2 (warps 4-7, 8-11) run the online
//     softmax and the epilogue of tile 0 and tile 1, one thread per query row
//     (TMEM lane = row), with a larger register budget handed over from
//     warpgroup 0 (setmaxnreg);
//   * TMEM (512 columns): S0 | S1 | O0 | O1.  S = Q K^T is written by an SS
//     MMA; the softmax warpgroup reads its row, writes P (bf16) back into the
//     upper half of the same S columns, and P V accumulates into O by a TS MMA
//     with P as the tensor-memory A operand;
//   * the two tiles alternate on the tensor core (P V of tile 0, S of tile 0's
//     next block, P V of tile 1, S of tile 1's next block), so one warpgroup's
//     exponentials overlap the other tile's MMAs;
//   * a pair with a single query tile (short query blocks: decoding, a ragged
//     last pair) puts the same rows in both slots and deals the key blocks to
//     them in turn, then merges the two states per row in the epilogue, so the
//     overlap above is kept; when every query block is one tile (decoding) a
//     single Q buffer serves both slots and the other becomes a third K stage;
//   * exponentials are base 2 with scale*log2(e) folded in; the running max is
//     only moved (and O rescaled in TMEM) when it grows by more than 2^8, which
//     keeps the result exact because l and A always share the same reference m;
//   * causal: blocks wholly in the future are never visited, the element mask
//     is applied only where a block crosses the diagonal or the sequence end;
//   * block-sparse: an item's two CSR rows become bitmaps in shared memory
//     (duplicates collapse, order is irrelevant); every role visits the union
//     in ascending order, each tile computing only the blocks of its own list.
//     Two bitmap buffers let the next item's be built while the current item
//     runs.
#include "common.cuh"

namespace bss {
namespace {

// DEC: every query block is a single tile (Lq <= 128, decoding).  Both tile
// slots then compute on the same query rows, so one Q buffer serves both and
// the second becomes one more K stage (deeper key prefetch for a stream that
// is bound by memory latency rather than by the tensor core).
template <int D, bool DEC = false, bool SPARSE = false>
struct FwdCfg {
  static constexpr int kChunks = D / 64;                   // 128-byte swizzle atoms across d
  static constexpr int kChunkBytes = kTileM * 128;         // 128 rows x 128 bytes
  static constexpr int kTileBytes = kTileM * D * 2;
  static constexpr int kQSlots = DEC ? 1 : 2;
  static constexpr int kStagesK = ((D == 128) ? 2 : 4) + (DEC ? 1 : 0);
  static constexpr int kStagesV = (D == 128) ? 3 : 4;   // V is consumed last: deeper prefetch
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQSlots * kTileBytes;
  static constexpr int kVOff = kKOff + kStagesK * kTileBytes;
  static constexpr int kBarOff = kVOff + kStagesV * kTileBytes;
  // q_full[2] q_empty[2] k_full[SK] k_empty[SK] v_full[SV] v_empty[SV] s_full[2]
  // p_full[2] o_full[2] o_empty[2] item_full[2] item_empty[2] clc mma_done
  static constexpr int kBarQFull = 0;
  static constexpr int kBarQEmpty = 2;
  static constexpr int kBarKFull = 4;
  static constexpr int kBarKEmpty = kBarKFull + kStagesK;
  static constexpr int kBarVFull = kBarKEmpty + kStagesK;
  static constexpr int kBarVEmpty = kBarVFull + kStagesV;
  static constexpr int kBarSFull = kBarVEmpty + kStagesV;
  static constexpr int kBarPFull = kBarSFull + 2;
  static constexpr int kBarOFull = kBarPFull + 2;
  static constexpr int kBarOEmpty = kBarOFull + 2;
  static constexpr int kBarItemFull = kBarOEmpty + 2;
  static constexpr int kBarItemEmpty = kBarItemFull + 2;
  static constexpr int kBarClc = kBarItemEmpty + 2;
  static constexpr int kBarMmaDone = kBarClc + 1;
  static constexpr int kBarXFull = kBarMmaDone + 1;    // tile 1's row state handed over
  static constexpr int kBarXEmpty = kBarXFull + 1;     // ... and read by tile 0
  static constexpr int kBarBmEmpty = kBarXEmpty + 1;   // [2] an item's bitmaps walked by every role
  static constexpr int kNumBars = kBarBmEmpty + (SPARSE ? 2 : 0);
  // 16-byte aligned: cancel answer (16) | TMEM base | abort flag | next item [2]
  static constexpr int kMiscOff = (kBarOff + kNumBars * 8 + 15) & ~15;
  static constexpr int kClcOff = kMiscOff;
  static constexpr int kTmemSlotOff = kMiscOff + 16;
  static constexpr int kAbortOff = kMiscOff + 20;
  static constexpr int kNextItemOff = kMiscOff + 24;
  static constexpr int kBitmapWords = kMaxKBlocks / 32;
  static constexpr int kBitmapOff = kMiscOff + 32;
  // A dense launch has no bitmaps; the same bytes carry the (m, mt, l) rows
  // one softmax warpgroup hands to the other (three arrays of 128 floats).
  // A block-sparse launch keeps the bitmaps of two items there (two per item,
  // one word per 32 key blocks of the launch) and, in the region's last 16
  // bytes, the first item's CSR row bounds.  Its region takes what the 227 KB
  // leave, up to four bitmaps of the largest key range.  (The dense kernels
  // keep their own smaller layout: the block-sparse barriers and region in
  // them measured 0.9 % slower at L=16384, for no use.)
  static constexpr int kXchOff = kBitmapOff;
  static constexpr int kXchBytes = 3 * kTileM * 4;
  static constexpr int kRegionFree = 232448 - 1024 - kBitmapOff;
  static constexpr int kRegionWanted = 4 * kBitmapWords * 4 + 16;
  static constexpr int kBitmapRegion =
      !SPARSE ? kXchBytes : (kRegionFree < kRegionWanted ? kRegionFree : kRegionWanted);
  static_assert(kBitmapRegion >= kXchBytes &&
                    (!SPARSE || kBitmapRegion >= 2 * kBitmapWords * 4 + 16),
                "one item's bitmaps and the row bounds (or the exchanged rows) must fit");
  static constexpr int kSmemBytes = kBitmapOff + kBitmapRegion + 1024;
  static_assert(kSmemBytes <= 232448, "forward shared memory exceeds the 227 KB a CTA may use");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;                      // S_t at t*128
  static constexpr uint32_t kColP = 64;                     // P_t at S_t + 64 (bf16 pairs)
  static constexpr uint32_t kColO = 256;                    // O_t at 256 + t*D
  static constexpr int kThreads = 384;
  // Readers of each next-item slot: the MMA thread and one lane of each of the
  // eight softmax warps (and the producer in a block-sparse launch, where
  // warp 3 writes the slots).
  static constexpr int kItemReaders = 1 + 8;
};

// Register split per warpgroup (setmaxnreg): warpgroup 0 (TMA and scheduler,
// MMA, an idle warp, and warp 3: idle, or preparing block-sparse items) gets
// kLow registers a thread, the two softmax warpgroups
// kHigh.  Each SM sub-partition holds one warp of every warpgroup, so
// kLow + 2 kHigh must stay within its 512 registers a lane, and the whole
// split within the 384 * 168 registers the launch holds (launch_one refuses
// to launch if ptxas gave the kernel fewer than 168 a thread, which would
// leave setmaxnreg.inc waiting for registers that never come).  The
// block-sparse instantiations take the same split: with 152/176 their
// softmax warpgroups spilled, and 136/184 measured 3.5 % faster.  Their
// producer's Q loads for later items spill a few bytes (8 at d=128).
template <bool SPARSE>
struct FwdRegs {
  static constexpr uint32_t kLow = 136;
  static constexpr uint32_t kHigh = 184;
  static constexpr uint32_t kLaunchRegs = 168;
  static_assert(kLow + 2 * kHigh <= 512, "register split exceeds an SM sub-partition");
  static_assert(128 * kLow + 256 * kHigh <= 384 * kLaunchRegs, "register split exceeds the launch");
};

// One work item: two consecutive 128-row query tiles of one (b, h), which
// share a single K/V stream.  Items are numbered by fwd_item below: in groups
// of heads, row-pair-major inside a group with every head of a pair side by
// side; under a causal mask the last pair (whose rows see the most keys) comes
// first, so that the longest items start first.
struct FwdItem {
  int b, h, bh;
  int hkv;         // K/V head read by query head h
  int c;           // key chunk (0 without a split)
  int kbase;       // row of the chunk's first key in K and V
  int Lkc;         // keys in the chunk
  long long koff;  // absolute position of the chunk's first key (causal mask)
  int r0[2];       // first query row of each tile
  int kbmax[2];    // last key block (of the chunk) each tile can see (-1: none)
  // Alternating item: the pair has a single query tile (its second tile lies
  // past the last row) and a dense key range of at least two blocks.  Both
  // tile slots then hold the SAME query rows and take the key blocks in turn
  // (slot 0 the even blocks, slot 1 the odd ones), so that one slot's softmax
  // overlaps the other slot's MMAs as in a full pair; the two partial states
  // of each row are merged in the epilogue.  Short query blocks (decoding)
  // are all of this kind.
  bool alt;
};

// Items come in groups of p.head_group query heads (every group but the last
// full).  Inside a group they are numbered row-pair-major, then key chunk,
// then head: under a causal mask the last pair (whose rows see the most keys)
// comes first, and the heads of one pair and chunk sit side by side.  The
// items running at any moment then read the K and V of one group's heads,
// which the host sizes to stay in L2, instead of streaming every head's K and
// V through it.
template <bool CAUSAL, bool ALT>
__device__ __forceinline__ FwdItem fwd_item(int item, const FwdParams& p) {
  FwdItem it;
  const int BH = p.B * p.H;
  const int gh = p.head_group;
  const int per_group = gh * p.n_chunks * p.n_pairs;
  const int grp = item / per_group;
  const int gsz = min(gh, BH - grp * gh);
  const int within = item - grp * per_group;
  const int per_rank = gsz * p.n_chunks;
  const int rank = within / per_rank;
  const int rem = within - rank * per_rank;
  it.c = rem / gsz;
  it.bh = grp * gh + (rem - it.c * gsz);
  it.b = it.bh / p.H;
  it.h = it.bh - it.b * p.H;
  it.hkv = it.h / (p.H / p.Hkv);
  it.kbase = it.c * p.chunk_len;
  it.Lkc = min(p.chunk_len, p.Lk - it.kbase);
  it.koff = p.k_offset + it.kbase;
  const int pair = CAUSAL ? (p.n_pairs - 1 - rank) : rank;
  it.r0[0] = pair * 2 * kTileM;
  it.r0[1] = it.r0[0] + kTileM;
  const int nk = it.Lkc > 0 ? (it.Lkc + kTileN - 1) / kTileN : 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    if (it.r0[t] >= p.Lq || nk == 0) {
      it.kbmax[t] = -1;
    } else if (CAUSAL) {
      const long long r_last = min(it.r0[t] + kTileM - 1, p.Lq - 1);
      const long long lim = r_last + p.q_offset - it.koff;
      it.kbmax[t] = lim < 0 ? -1 : static_cast<int>(lim / kTileN < nk - 1 ? lim / kTileN : nk - 1);
    } else {
      it.kbmax[t] = nk - 1;
    }
  }
  it.alt = ALT && it.r0[1] >= p.Lq && it.kbmax[0] >= 1;
  if (it.alt) {
    it.r0[1] = it.r0[0];
    it.kbmax[1] = it.kbmax[0];
  }
  return it;
}

// The ordered list of key blocks an item visits and which of its two tiles
// takes part in each.  Every role walks it identically.
struct Schedule {
  int kbmax0, kbmax1;          // last block a tile can see (-1: none)
  const uint32_t* bm0;         // block-sparse bitmaps (nullptr: dense prefix)
  const uint32_t* bm1;
  bool alt;                    // alternating item: block kb belongs to slot kb & 1

  __device__ __forceinline__ Schedule(const FwdItem& it, const uint32_t* bitmap, int words)
      : kbmax0(it.kbmax[0]), kbmax1(it.kbmax[1]), bm0(bitmap),
        bm1(bitmap ? bitmap + words : nullptr), alt(it.alt) {}

  __device__ __forceinline__ int member(int kb) const {
    if (alt) return kb <= kbmax0 ? 1 << (kb & 1) : 0;
    int m = 0;
    if (kb <= kbmax0 && (bm0 == nullptr || ((bm0[kb >> 5] >> (kb & 31)) & 1u))) m |= 1;
    if (kb <= kbmax1 && (bm1 == nullptr || ((bm1[kb >> 5] >> (kb & 31)) & 1u))) m |= 2;
    return m;
  }
  __device__ __forceinline__ int next(int kb) const {
    const int lim = max(kbmax0, kbmax1);
    if (bm0 == nullptr) return (kb + 1 <= lim) ? kb + 1 : -1;
    int c = kb + 1;
    while (c <= lim) {
      const int w = c >> 5;
      const uint32_t bits = (bm0[w] | bm1[w]) & (0xFFFFFFFFu << (c & 31));
      if (bits == 0) {
        c = (w + 1) << 5;
        continue;
      }
      const int cand = (w << 5) + __ffs(bits) - 1;
      if (cand > lim) return -1;
      if (member(cand)) return cand;
      c = cand + 1;
    }
    return -1;
  }
  // The last block tile t computes (-1: none).
  __device__ __forceinline__ int last(int t) const {
    if (alt) return ((kbmax0 & 1) == t) ? kbmax0 : kbmax0 - 1;
    const int lim = t ? kbmax1 : kbmax0;
    const uint32_t* bm = t ? bm1 : bm0;
    if (bm == nullptr || lim < 0) return lim;
    for (int w = lim >> 5; w >= 0; --w) {
      uint32_t bits = bm[w];
      if (w == (lim >> 5)) bits &= (2u << (lim & 31)) - 1u;
      if (bits) return (w << 5) + 31 - __clz(bits);
    }
    return -1;
  }
};

// Persistent over work items.  The grid holds one CTA per item, but a running
// CTA does not exit after its own item: when its producer has issued the loads
// of an item's last key block it asks the hardware (cluster launch control) to
// cancel a CTA that has not started yet and takes over that CTA's item.  So
// one CTA per SM streams item after item, with set-up paid once, the next
// item's Q and K loads and S = Q K^T overlapping the previous item's epilogue,
// and the items handed out greedily in order (longest first under a causal
// mask).  The producer passes each next item index to the other roles through
// a two-slot ring in shared memory.  In a block-sparse launch warp 3 takes the
// producer's part in this: it claims the next item as soon as a bitmap buffer
// is free (about one item ahead), builds the item's bitmaps there and writes
// the ring, so that the producer finds the next item ready when it reaches
// the end of the current one.
template <int D, bool CAUSAL, bool SPARSE, bool PARTIAL, bool ALT, bool DEC>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  constexpr bool kAlt = ALT && !SPARSE;   // single-tile pairs may alternate
  constexpr bool kDec = DEC && kAlt;      // one Q buffer for both slots
  using C = FwdCfg<D, kDec, SPARSE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + C::kBarOff;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::kTmemSlotOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);
  volatile int* next_item = reinterpret_cast<volatile int*>(smem + C::kNextItemOff);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + C::kBitmapOff);

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int tid = static_cast<int>(threadIdx.x);
  const bool tr = BSS_TRACE_ON(p, blockIdx.x);
  (void)tr;
  // A launch whose earlier CTAs already timed out stops at once instead of
  // timing out CTA by CTA.
  if (*reinterpret_cast<volatile int*>(p.err) == ATTN_ERR_TIMEOUT) return;

  // ---- set-up: barriers, tensor memory, block-sparse bitmaps -------------
  // A block-sparse CTA builds its first item's bitmaps here.  The item's two
  // CSR row bounds are read first (into the last 16 bytes of the bitmap
  // region) and its two Q tiles are loaded as soon as the barriers exist, so
  // that both latencies overlap the rest of the set-up instead of preceding
  // the first key block.  Later items' bitmaps come from warp 3, in the other
  // of two buffers (bw words a bitmap); a key range too long for two buffers
  // runs one item per CTA.
  const int bw = SPARSE ? ((p.Lk + kTileN - 1) / kTileN + 31) >> 5 : 0;
  const bool persist_sparse = SPARSE && 16 * bw + 16 <= C::kBitmapRegion;
  int* rp_s = reinterpret_cast<int*>(smem + C::kBitmapOff + C::kBitmapRegion - 16);
  // the bitmaps of the n-th item a CTA runs (nullptr: a dense key range)
  auto item_bm = [&](int n) -> const uint32_t* {
    return SPARSE ? bitmap + (n & 1) * 2 * bw : nullptr;
  };
  if (SPARSE && tid < 4) {
    const FwdItem it0 = fwd_item<CAUSAL, kAlt>(blockIdx.x, p);
    const int t = tid >> 1;
    const int qb = it0.r0[t] / kTileM;
    int v = INT_MIN;                             // no such query block
    if (it0.r0[t] < p.Lq && qb < p.n_qblk)
      v = __ldg(p.row_ptr + static_cast<size_t>(it0.bh / p.heads_per_list) * (p.n_qblk + 1) + qb +
                (tid & 1));
    rp_s[tid] = v;
  }
  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kBarQFull + t), 1);
      mbar_init(bar(C::kBarQEmpty + t), 1);
      mbar_init(bar(C::kBarSFull + t), 1);
      mbar_init(bar(C::kBarPFull + t), 4 * 32);
      mbar_init(bar(C::kBarOFull + t), 1);
      mbar_init(bar(C::kBarOEmpty + t), 4 * 32);
      mbar_init(bar(C::kBarItemFull + t), 1);
      mbar_init(bar(C::kBarItemEmpty + t), C::kItemReaders + (SPARSE ? 1 : 0));
      // producer, MMA thread, one lane of each softmax warp
      if (SPARSE) mbar_init(bar(C::kBarBmEmpty + t), 1 + 1 + 8);
    }
    for (int s = 0; s < C::kStagesK; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
    }
    for (int s = 0; s < C::kStagesV; ++s) {
      mbar_init(bar(C::kBarVFull + s), 1);
      mbar_init(bar(C::kBarVEmpty + s), 1);
    }
    mbar_init(bar(C::kBarClc), 1);
    mbar_init(bar(C::kBarMmaDone), 1);
    mbar_init(bar(C::kBarXFull), 4 * 32);
    mbar_init(bar(C::kBarXEmpty), 4 * 32);
    *abort_flag = 0;
    fence_barrier_init();
    if (SPARSE) {
      // both Q tiles of the item (a tile past Lq reads the zero fill)
      const FwdItem it0 = fwd_item<CAUSAL, kAlt>(blockIdx.x, p);
      for (int t = 0; t < 2; ++t) {
        const uint32_t qs = sbase + C::kQOff + t * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kBarQFull + t), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(qs + c * C::kChunkBytes, &tmQ, bar(C::kBarQFull + t), c * 64, it0.r0[t], it0.h,
                      it0.b);
      }
    }
  }
  if (warp == 0) {
    tmem_alloc(sbase + C::kTmemSlotOff, C::kTmemCols);
    tmem_relinquish();
  }
  BSS_TRACE_EV(p, tr && tid == 0, 6, 0);
  if (SPARSE) {
    const int nk = (p.Lk + kTileN - 1) / kTileN;
    for (int i = tid; i < 2 * bw; i += C::kThreads) bitmap[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int beg = rp_s[2 * t];
      const int end = rp_s[2 * t + 1];
      if (beg == INT_MIN) continue;              // no such query block
      if (beg < 0 || end < beg || end > p.nnz) {
        if (tid == 0) record_error(p.err, ATTN_ERR_BAD_BLOCKLIST);
        continue;
      }
      for (int e = beg + tid; e < end; e += C::kThreads) {
        const int c = __ldg(p.col_idx + e);
        if (c < 0 || c >= nk) {
          record_error(p.err, ATTN_ERR_BAD_BLOCKLIST);
          continue;
        }
        atomicOr(bitmap + t * bw + (c >> 5), 1u << (c & 31));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
  regs_set<FwdRegs<SPARSE>::kLow, FwdRegs<SPARSE>::kLaunchRegs>();
  if (warp == 0) {
    // =================== TMA producer and item scheduler ===================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int item = static_cast<int>(blockIdx.x);
      int n = 0;              // items finished
      int ik = 0, iv = 0;     // K and V tiles loaded (over all items)
      int qn[2] = {SPARSE ? 1 : 0, SPARSE ? 1 : 0};   // Q tiles loaded into each tile slot
                              // (a block-sparse CTA's two were loaded at set-up)
      int clc_k = 0;          // cancel requests answered
      bool clc_live = !SPARSE;
      bool clc_out = false;   // a cancel request is in flight
      bool ok = true;
      auto request_item = [&]() {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar(C::kBarClc), 16);
        clc_try_cancel(sbase + C::kClcOff, bar(C::kBarClc));
        clc_out = true;
      };
      while (ok) {
        const FwdItem it = fwd_item<CAUSAL, kAlt>(item, p);
        const Schedule sch(it, item_bm(n), bw);
        bool qloaded[2] = {SPARSE && n == 0, SPARSE && n == 0};
        for (int kb = sch.next(-1); kb >= 0;) {
          const int nkb = sch.next(kb);
          // The next item is asked for as this item's last block is loaded.
          if (nkb < 0 && clc_live) request_item();
          const int mask = sch.member(kb);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int q = kDec ? 0 : t;   // the Q buffer tile slot t reads
            if (((mask >> t) & 1) && !qloaded[q] && ok) {
              if (qn[q] > 0 &&
                  !wait_bar(bar(C::kBarQEmpty + q), (qn[q] - 1) & 1, abort_flag, p.err)) {
                ok = false;
                break;
              }
              const uint32_t qs = sbase + C::kQOff + q * C::kTileBytes;
              mbar_arrive_expect_tx(bar(C::kBarQFull + q), C::kTileBytes);
#pragma unroll
              for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(qs + c * C::kChunkBytes, &tmQ, bar(C::kBarQFull + q), c * 64, it.r0[t],
                            it.h, it.b);
              ++qn[q];
              qloaded[q] = true;
            }
          }
          if (!ok) break;
          const int sk = ik % C::kStagesK;
          if (ik >= C::kStagesK &&
              !wait_bar(bar(C::kBarKEmpty + sk), ((ik / C::kStagesK) & 1) ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          BSS_TRACE_EV(p, tr, 0, 2 * ik);
          const uint32_t ks = sbase + C::kKOff + sk * C::kTileBytes;
          mbar_arrive_expect_tx(bar(C::kBarKFull + sk), C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(ks + c * C::kChunkBytes, &tmK, bar(C::kBarKFull + sk), c * 64, it.kbase + kb * kTileN,
                        it.hkv, it.b);
          ++ik;
          const int sv = iv % C::kStagesV;
          if (iv >= C::kStagesV &&
              !wait_bar(bar(C::kBarVEmpty + sv), ((iv / C::kStagesV) & 1) ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          BSS_TRACE_EV(p, tr, 0, 2 * iv + 1);
          const uint32_t vs = sbase + C::kVOff + sv * C::kTileBytes;
          mbar_arrive_expect_tx(bar(C::kBarVFull + sv), C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(vs + c * C::kChunkBytes, &tmV, bar(C::kBarVFull + sv), c * 64, it.kbase + kb * kTileN,
                        it.hkv, it.b);
          ++iv;
          kb = nkb;
        }
        if (!ok) break;
        if (SPARSE) {
          // block-sparse: this item's bitmaps are walked; warp 3 has claimed
          // and prepared the next item, which the ring holds
          mbar_arrive(bar(C::kBarBmEmpty + (n & 1)));
          const int s = n & 1;
          if (!wait_bar(bar(C::kBarItemFull + s), (n >> 1) & 1, abort_flag, p.err)) break;
          const int next = next_item[s];
          mbar_arrive(bar(C::kBarItemEmpty + s));
          ++n;
          if (next < 0) break;
          item = next;
          continue;
        }
        if (clc_live && !clc_out) request_item();   // an item without blocks
        int next = -1;
        if (clc_out) {
          if (!wait_bar(bar(C::kBarClc), clc_k & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          clc_out = false;
          ++clc_k;
          int x = -1;
          if (clc_query(sbase + C::kClcOff, x)) {
            if (x >= 0 && x < p.n_items) {
              next = x;
            } else {
              record_error(p.err, ATTN_ERR_CUDA);   // not an index of this grid
              clc_live = false;
            }
          } else {
            clc_live = false;                        // nothing left to take
          }
        }
        const int s = n & 1;
        if (n >= 2 &&
            !wait_bar(bar(C::kBarItemEmpty + s), ((n >> 1) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        next_item[s] = next;
        mbar_arrive(bar(C::kBarItemFull + s));
        ++n;
        if (next < 0) break;
        item = next;
      }
      // Drain: every copy issued has landed before the CTA may exit (on the
      // normal path these waits return at once).
      for (int j = max(0, ik - C::kStagesK); j < ik; ++j)
        drain_bar(bar(C::kBarKFull + j % C::kStagesK), (j / C::kStagesK) & 1);
      for (int j = max(0, iv - C::kStagesV); j < iv; ++j)
        drain_bar(bar(C::kBarVFull + j % C::kStagesV), (j / C::kStagesV) & 1);
      for (int t = 0; t < 2; ++t)
        if (qn[t] > 0) drain_bar(bar(C::kBarQFull + t), (qn[t] - 1) & 1);
      if (clc_out) drain_bar(bar(C::kBarClc), clc_k & 1);
    }
  } else if (warp == 1) {
    // =================== MMA issuer (one thread) ===================
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(kTileM, kTileN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileM, D, false, true);
      int item = static_cast<int>(blockIdx.x);
      int n = 0;                // items finished
      int i = 0;                // key blocks consumed (over all items)
      int qn[2] = {0, 0};       // Q tiles consumed per tile slot
      int pcount[2] = {0, 0};   // P tiles consumed per tile
      int on[2] = {0, 0};       // O accumulations handed to the epilogue per tile
      bool ok = true;
      while (ok) {
        const FwdItem it = fwd_item<CAUSAL, kAlt>(item, p);
        const Schedule sch(it, item_bm(n), bw);
        const int lastkb[2] = {sch.last(0), sch.last(1)};
        bool qready[2] = {false, false};
        bool ostarted[2] = {false, false};

        // the item's last S of any tile frees a Q buffer shared by both slots
        const int qlast = lastkb[0] > lastkb[1] ? lastkb[0] : lastkb[1];
        auto issue_qk = [&](int t, int sk, int kb) -> bool {
          const int q = kDec ? 0 : t;
          if (!qready[q]) {
            if (!wait_bar(bar(C::kBarQFull + q), qn[q] & 1, abort_flag, p.err)) return false;
            qready[q] = true;
          }
          const uint64_t dq = sdesc_sw128(sbase + C::kQOff + q * C::kTileBytes, 16, 1024);
          const uint64_t dk = sdesc_sw128(sbase + C::kKOff + sk * C::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
            mma_ss(tmem + C::kColS + t * 128, sdesc_add(dq, off), sdesc_add(dk, off), kIdescQK,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kBarSFull + t));
          // Q of this tile is free for the next item once its last S lands.
          if (kb == (kDec ? qlast : lastkb[t])) mma_commit(bar(C::kBarQEmpty + q));
          return true;
        };
        auto issue_pv = [&](int t, int sv) -> bool {
          if (!ostarted[t] && on[t] > 0) {
            // O_t still holds the previous item's result until its epilogue read it
            if (!wait_bar(bar(C::kBarOEmpty + t), (on[t] - 1) & 1, abort_flag, p.err)) return false;
            tc_fence_after();
          }
          const uint64_t dv = sdesc_sw128(sbase + C::kVOff + sv * C::kTileBytes, C::kChunkBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk) {
            mma_ts(tmem + C::kColO + t * D, tmem + C::kColS + t * 128 + C::kColP + kk * 8,
                   sdesc_add(dv, kk * 16 * 128), kIdescPV,
                   (ostarted[t] || kk > 0) ? 1u : 0u);
          }
          ostarted[t] = true;
          return true;
        };

        if (kAlt && it.alt) {
          // Each key block serves one slot (kb & 1): S0(0) S1(1), then for
          // every block its slot's P V followed by that slot's S two blocks on.
          const int nb = it.kbmax[0] + 1;
          auto alt_qk = [&](const int t, int kb) -> bool {
            const int j = i + kb;
            const int sk = j % C::kStagesK;
            if (!wait_bar(bar(C::kBarKFull + sk), (j / C::kStagesK) & 1, abort_flag, p.err)) return false;
            tc_fence_after();
            if (!issue_qk(t, sk, kb)) return false;
            mma_commit(bar(C::kBarKEmpty + sk));
            return true;
          };
          auto alt_step = [&](const int t, int kb) -> bool {
            const int j = i + kb;
            const int sv = j % C::kStagesV;
            if (!wait_bar(bar(C::kBarVFull + sv), (j / C::kStagesV) & 1, abort_flag, p.err)) return false;
            if (!wait_bar(bar(C::kBarPFull + t), pcount[t] & 1, abort_flag, p.err)) return false;
            ++pcount[t];
            tc_fence_after();
            if (!issue_pv(t, sv)) return false;
            mma_commit(bar(C::kBarVEmpty + sv));
            return kb + 2 < nb ? alt_qk(t, kb + 2) : true;
          };
          ok = alt_qk(0, 0) && alt_qk(1, 1);
          for (int kb = 0; kb < nb && ok; kb += 2) {
            ok = alt_step(0, kb);
            if (ok && kb + 1 < nb) ok = alt_step(1, kb + 1);
          }
          i += nb;
        } else {
        int kb = sch.next(-1);
        int mask = kb >= 0 ? sch.member(kb) : 0;
        if (kb >= 0) {
          const int sk = i % C::kStagesK;
          ok = wait_bar(bar(C::kBarKFull + sk), (i / C::kStagesK) & 1, abort_flag, p.err);
          if (ok) {
            tc_fence_after();
            if (ok && (mask & 1)) ok = issue_qk(0, sk, kb);
            if (ok && (mask & 2)) ok = issue_qk(1, sk, kb);
            if (ok) mma_commit(bar(C::kBarKEmpty + sk));
          }
        }
        while (kb >= 0 && ok) {
          const int nkb = sch.next(kb);
          const int nmask = nkb >= 0 ? sch.member(nkb) : 0;
          const int sv = i % C::kStagesV;
          const int skn = (i + 1) % C::kStagesK;
          if (!wait_bar(bar(C::kBarVFull + sv), (i / C::kStagesV) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          BSS_TRACE_EV(p, tr, 1, 4 * i);
          tc_fence_after();
          bool kready = false;
          // tile t's P V of this block, then its S of the next block; called
          // with constant t so that the per-tile counters stay in registers
          auto tile_step = [&](const int t) -> bool {
            if ((mask >> t) & 1) {
              if (!wait_bar(bar(C::kBarPFull + t), pcount[t] & 1, abort_flag, p.err)) return false;
              ++pcount[t];
              BSS_TRACE_EV(p, tr, 1, 4 * i + 1 + t);
              tc_fence_after();
              if (!issue_pv(t, sv)) return false;
            }
            if ((nmask >> t) & 1) {
              if (!kready) {
                if (!wait_bar(bar(C::kBarKFull + skn), ((i + 1) / C::kStagesK) & 1, abort_flag, p.err))
                  return false;
                tc_fence_after();
                kready = true;
              }
              return issue_qk(t, skn, nkb);
            }
            return true;
          };
          ok = tile_step(0) && tile_step(1);
          if (!ok) break;
          BSS_TRACE_EV(p, tr, 1, 4 * i + 3);
          mma_commit(bar(C::kBarVEmpty + sv));
          if (nkb >= 0) mma_commit(bar(C::kBarKEmpty + skn));
          kb = nkb;
          mask = nmask;
          ++i;
        }
        }
        if (!ok) break;
        if (SPARSE) {
          mbar_arrive(bar(C::kBarBmEmpty + (n & 1)));   // this item's bitmaps walked
          // The first item's two Q tiles were loaded at set-up: a tile with no
          // block in it hands its buffer back once the load has landed (so
          // that the next item's Q load into it waits on the right phase).
          bool qok = true;
          if (n == 0) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (lastkb[t] < 0 && qok) {
                qok = wait_bar(bar(C::kBarQFull + t), qn[t] & 1, abort_flag, p.err);
                if (qok) {
                  mbar_arrive(bar(C::kBarQEmpty + t));
                  qready[t] = true;
                }
              }
            }
          }
          if (!qok) break;
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (ostarted[t]) {
            mma_commit(bar(C::kBarOFull + t));
            ++on[t];
          }
          if (qready[t]) ++qn[t];
        }
        const int s = n & 1;
        if (!wait_bar(bar(C::kBarItemFull + s), (n >> 1) & 1, abort_flag, p.err)) break;
        const int next = next_item[s];
        mbar_arrive(bar(C::kBarItemEmpty + s));
        ++n;
        if (next < 0) break;
        item = next;
      }
      // every MMA issued has completed before tensor memory is released
      mma_commit(bar(C::kBarMmaDone));
      drain_bar(bar(C::kBarMmaDone), 0);
    }
  } else if (SPARSE && warp == 3) {
    // =================== block-sparse item preparation (warp 3) ===================
    // Item k (k >= 1) of this CTA: claimed by cluster launch control (the CTA
    // cancels a not-yet-started CTA of the grid and takes its item), its two
    // bitmaps built in buffer k & 1 from its CSR rows, and its index written
    // to ring slot (k - 1) & 1, which every role reads at the end of item
    // k - 1.  The buffer was last used by item k - 2, so the claim comes as
    // soon as every role has walked that item: about one item ahead.  (A
    // claim made only once the producer had issued item k - 1's loads left
    // the producer waiting for the bitmaps and measured 4 % slower.)
    const int nk = (p.Lk + kTileN - 1) / kTileN;
    bool live = persist_sparse;   // false: every item claimed, or one item per CTA
    int clc_k = 0;                // cancel requests answered
    bool clc_out = false;         // a cancel request is in flight
    for (int k = 1;; ++k) {
      const int s = (k - 1) & 1;  // ring slot carrying item k
      const int b = k & 1;        // bitmap buffer of item k
      // the slot's previous entry (item k - 2) has been read by every role
      if (k >= 3 && !__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarItemEmpty + s),
                                                      (((k - 1) >> 1) & 1) ^ 1, abort_flag, p.err)))
        break;
      int next = -1;
      if (live) {
        // the buffer's previous item (k - 2) has been walked by every role
        if (k >= 2 && !__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarBmEmpty + b),
                                                        ((k - 2) >> 1) & 1, abort_flag, p.err)))
          break;
        int x = -1, got = 0, fail = 0;
        if (lane == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bar(C::kBarClc), 16);
          clc_try_cancel(sbase + C::kClcOff, bar(C::kBarClc));
          clc_out = true;
          if (!wait_bar(bar(C::kBarClc), clc_k & 1, abort_flag, p.err)) {
            fail = 1;
          } else {
            clc_out = false;
            ++clc_k;
            if (clc_query(sbase + C::kClcOff, x)) {
              if (x >= 0 && x < p.n_items)
                got = 1;
              else
                record_error(p.err, ATTN_ERR_CUDA);   // not an index of this grid
            }
          }
        }
        if (__shfl_sync(0xFFFFFFFFu, fail, 0)) break;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        x = __shfl_sync(0xFFFFFFFFu, x, 0);
        if (got)
          next = x;
        else
          live = false;   // nothing left to take (no request follows a failed one)
      }
      if (next >= 0) {
        // the item's bitmaps: clear the buffer, then one bit per listed block
        const FwdItem it = fwd_item<CAUSAL, kAlt>(next, p);
        uint32_t* bm = bitmap + b * 2 * bw;
        for (int i = lane; i < 2 * bw; i += 32) bm[i] = 0u;
        int v = INT_MIN;                           // no such query block
        if (lane < 4) {
          const int t = lane >> 1;
          const int qb = it.r0[t] / kTileM;
          if (it.r0[t] < p.Lq && qb < p.n_qblk)
            v = __ldg(p.row_ptr + static_cast<size_t>(it.bh / p.heads_per_list) * (p.n_qblk + 1) +
                      qb + (lane & 1));
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int beg = __shfl_sync(0xFFFFFFFFu, v, 2 * t);
          const int end = __shfl_sync(0xFFFFFFFFu, v, 2 * t + 1);
          if (beg == INT_MIN) continue;
          if (beg < 0 || end < beg || end > p.nnz) {
            if (lane == 0) record_error(p.err, ATTN_ERR_BAD_BLOCKLIST);
            continue;
          }
          for (int e = beg + lane; e < end; e += 32) {
            const int c = __ldg(p.col_idx + e);
            if (c < 0 || c >= nk) {
              record_error(p.err, ATTN_ERR_BAD_BLOCKLIST);
              continue;
            }
            atomicOr(bm + t * bw + (c >> 5), 1u << (c & 31));
          }
        }
        __threadfence_block();
        __syncwarp();
      }
      if (lane == 0) {
        next_item[s] = next;
        mbar_arrive(bar(C::kBarItemFull + s));   // releases the bitmaps built above
      }
      if (next < 0) break;
    }
    if (lane == 0 && clc_out) drain_bar(bar(C::kBarClc), clc_k & 1);
  }
  } else {
    regs_set<FwdRegs<SPARSE>::kHigh, FwdRegs<SPARSE>::kLaunchRegs>();
    // =================== softmax warpgroups (warps 4-7: tile 0, 8-11: tile 1) ===================
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;                      // TMEM lane quarter of this warp
    const int row_in_tile = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kColS + t * 128;
    const uint32_t tP = tS + C::kColP;
    const uint32_t tO = tmem + lane_base + C::kColO + t * D;
    const float sl2 = p.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const bool trw = tr && lane == 0 && wq == 0;
    (void)trw;

    float* xch = reinterpret_cast<float*>(smem + C::kXchOff);

    int item = static_cast<int>(blockIdx.x);
    int n = 0;          // items finished
    int cnt = 0;        // S tiles consumed (over all items)
    int on0 = 0, on1 = 0;  // O accumulations completed per slot (both warpgroups count both)
    int nx = 0;         // row states handed over (alternating items)
    bool ok = true;
    while (ok) {
      const FwdItem it = fwd_item<CAUSAL, kAlt>(item, p);
      const Schedule sch(it, item_bm(n), bw);
      // block-sparse: whether slot 0 (1) accumulates into O_0 (O_1) in this
      // item, read before the item's bitmaps are released
      const bool has0 = SPARSE && sch.last(0) >= 0;
      const bool has1 = SPARSE && sch.last(1) >= 0;
      const int r0 = t ? it.r0[1] : it.r0[0];
      const int row = r0 + row_in_tile;

      float m2 = NEG_INF;     // reference max (log2 units), moved only by > 8
      float mt = NEG_INF;     // exact running max (log2 units)
      float l = 0.f;
      int ci = 0;             // blocks of this item
      for (int kb = sch.next(-1); kb >= 0; kb = sch.next(kb)) {
        if (!((sch.member(kb) >> t) & 1)) continue;
        // warp-uniform outcome: the loads below are warp-collective
        if (!__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarSFull + t), cnt & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        BSS_TRACE_EV(p, trw, 2 + t, 4 * cnt);
        tc_fence_after();
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);

        // element mask: only where the block crosses the diagonal or the end
        const int kstart = kb * kTileN;
        const bool edge = (kstart + kTileN > it.Lkc) ||
                          (CAUSAL && (static_cast<long long>(kstart) + kTileN - 1 + it.koff >
                                      static_cast<long long>(r0) + p.q_offset));
        if (edge) {
          long long lim = static_cast<long long>(it.Lkc) - 1 - kstart;
          if (CAUSAL) lim = min(lim, static_cast<long long>(row) + p.q_offset - it.koff - kstart);
          const int jl = static_cast<int>(max(-1ll, min(127ll, lim)));
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j > jl) s[c][j] = __float_as_uint(NEG_INF);
        }
        // row max over 8 independent chains of three-input max (short chains)
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(s[0][u]);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = (c == 0 ? 8 : 0); j < 32; j += 16)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              mx[u] = fmax3(mx[u], __uint_as_float(s[c][j + u]), __uint_as_float(s[c][j + 8 + u]));
        const float mblk = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
        BSS_TRACE_EV(p, trw, 2 + t, 4 * cnt + 1);
        mt = fmaxf(mt, mblk);
        float alpha = 1.f;
        bool moved = false;
        if (mblk > m2 + 8.f) {
          alpha = ex2(m2 - mblk);
          m2 = mblk;
          moved = true;
        }
        const float mu = (m2 == NEG_INF) ? 0.f : m2;
        // pairs of columns: one packed FMA for the two exponents' arguments,
        // one packed add into four pairs of running sums
        float rs[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) rs[u] = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int c = half * 2 + c2;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(s[c][j]), __uint_as_float(s[c][j + 1]), sl2, sl2, -mu,
                    -mu);
              const float p0 = ex2(x0);
              const float p1 = ex2(x1);
              const int u = (j >> 1) & 3;
              fadd2(rs[2 * u], rs[2 * u + 1], rs[2 * u], rs[2 * u + 1], p0, p1);
              pk[c2 * 16 + j / 2] = pack_bf16(p0, p1);
            }
          }
          tmem_st32(tP + half * 32, pk);
        }
        l = l * alpha + (((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7])));
        BSS_TRACE_EV(p, trw, 2 + t, 4 * cnt + 2);
        // rescale O when this row's reference max moved and O already holds data
        const bool fix = moved && ci > 0;
        if (__any_sync(0xFFFFFFFFu, fix)) {
          const float a = fix ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * a);
            tmem_st32(tO + c * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kBarPFull + t));
        BSS_TRACE_EV(p, trw, 2 + t, 4 * cnt + 3);
        ++cnt;
        ++ci;
      }
      if (!ok) break;
      if (SPARSE) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kBarBmEmpty + (n & 1)));   // bitmaps walked
      }

      if (kAlt && it.alt && t == 1) {
        // Alternating item: this row's state over the odd key blocks goes to
        // tile 0's warpgroup, which merges it with the even blocks' state (and
        // reads O_1 from tensor memory) and writes the row.
        if (nx > 0 &&
            !__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarXEmpty), (nx - 1) & 1, abort_flag, p.err)))
          break;
        xch[row_in_tile] = m2;
        xch[kTileM + row_in_tile] = mt;
        xch[2 * kTileM + row_in_tile] = l;
        mbar_arrive(bar(C::kBarXFull));
        ++nx;
      } else {
      // ---- epilogue: O_t is read out of TMEM at once and released to the
      // next item's P V before the global stores ----
      uint32_t o[D / 32][32];
      if (kAlt && it.alt) {
        // merge the two slots' states of this row: both are (m, l, A) over
        // disjoint key blocks, rescaled to the larger reference max; the
        // merged A goes back into O_0, which the epilogue below reads
        if (!__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarXFull), nx & 1, abort_flag, p.err))) break;
        const float m2b = xch[row_in_tile];
        const float mtb = xch[kTileM + row_in_tile];
        const float lb = xch[2 * kTileM + row_in_tile];
        mbar_arrive(bar(C::kBarXEmpty));
        ++nx;
        const float mm = fmaxf(m2, m2b);
        const float a0 = (m2 == NEG_INF) ? 0.f : ex2(m2 - mm);
        const float a1 = (m2b == NEG_INF) ? 0.f : ex2(m2b - mm);
        m2 = mm;
        mt = fmaxf(mt, mtb);
        l = l * a0 + lb * a1;
        if (!__all_sync(0xFFFFFFFFu,
                        wait_bar(bar(C::kBarOFull + 0), on0 & 1, abort_flag, p.err) &&
                            wait_bar(bar(C::kBarOFull + 1), on1 & 1, abort_flag, p.err)))
          break;
        tc_fence_after();
        const uint32_t tO1 = tmem + lane_base + C::kColO + D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x[32], y[32];
          tmem_ld32(tO + c * 32, x);
          tmem_ld32(tO1 + c * 32, y);
          tmem_ld_wait(x);
          tmem_ld_wait(y);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float x0, x1;
            fmul2(x0, x1, __uint_as_float(x[j]), __uint_as_float(x[j + 1]), a0, a0);
            ffma2(x0, x1, __uint_as_float(y[j]), __uint_as_float(y[j + 1]), a1, a1, x0, x1);
            x[j] = __float_as_uint(x0);
            x[j + 1] = __float_as_uint(x1);
          }
          tmem_st32(tO + c * 32, x);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kBarOEmpty + 1));
      }
      if (ci > 0) {
        if (!__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarOFull + t), (t ? on1 : on0) & 1, abort_flag, p.err)))
          break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + c * 32, o[c]);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld_wait(o[c]);
        tc_fence_before();
        mbar_arrive(bar(C::kBarOEmpty + t));
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) o[c][j] = 0u;
      }
      BSS_TRACE_EV(p, trw, 4 + t, 2 * n);
      const bool inb = row < p.Lq;
      // partial states of chunk c follow those of chunks 0 .. c-1
      const size_t rows0 = static_cast<size_t>(it.c) * p.B * p.H * p.Lq + static_cast<size_t>(it.bh) * p.Lq;
      const size_t row_g = rows0 + (inb ? row : 0);
      // first row of this warp (rows past Lq are masked out of `valid`)
      const size_t wrow0 = rows0 + (r0 + wq * 32);
      if (PARTIAL) {
        // An empty state (m = -inf) is fully described by m and l; its acc
        // row is not written (a merge never reads it).
        const float factor = (mt == NEG_INF || ci == 0) ? 0.f : ex2(m2 - mt);
        const uint32_t valid = __ballot_sync(0xFFFFFFFFu, inb && ci > 0 && mt != NEG_INF);
        if (valid) {
          uint8_t* base = reinterpret_cast<uint8_t*>(p.acc_out + wrow0 * D);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[c][j] = __float_as_uint(__uint_as_float(o[c][j]) * factor);
            transpose_octets(o[c], lane);
            store_octet_lines(o[c], base + c * 128, D * 4, valid, lane);
          }
        }
        if (inb) {
          p.m_out[row_g] = (mt == NEG_INF) ? NEG_INF : mt * kLn2;
          p.l_out[row_g] = l * factor;
        }
      } else {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const uint32_t valid = __ballot_sync(0xFFFFFFFFu, inb);
        uint8_t* base = reinterpret_cast<uint8_t*>(p.o + wrow0 * D);
#pragma unroll
        for (int g2 = 0; g2 < D / 64; ++g2) {
          // line g2 of a row: columns 64 g2 .. 64 g2 + 63 as 32 bf16 pairs
          uint32_t w[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int c = 2 * g2 + k / 16;
            const int j = (2 * k) % 32;
            w[k] = pack_bf16(__uint_as_float(o[c][j]) * inv, __uint_as_float(o[c][j + 1]) * inv);
          }
          transpose_octets(w, lane);
          store_octet_lines(w, base + g2 * 128, D * 2, valid, lane);
        }
        if (inb) p.lse[row_g] = l > 0.f ? (m2 + __log2f(l)) * kLn2 : NEG_INF;
      }
      }
      on0 += (SPARSE ? has0 : sch.last(0) >= 0) ? 1 : 0;
      on1 += (SPARSE ? has1 : sch.last(1) >= 0) ? 1 : 0;
      BSS_TRACE_EV(p, trw, 4 + t, 2 * n + 1);
      // ---- next item ----
      const int s = n & 1;
      if (!__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarItemFull + s), (n >> 1) & 1, abort_flag, p.err)))
        break;
      const int next = next_item[s];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kBarItemEmpty + s));
      ++n;
      if (next < 0) break;
      item = next;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool SPARSE, bool PARTIAL, bool ALT, bool DEC>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t st) {
  using C = FwdCfg<D, DEC && ALT && !SPARSE, SPARSE>;
  auto kern = attn_fwd_kernel<D, CAUSAL, SPARSE, PARTIAL, ALT, DEC>;
  constexpr int kMaxDev = 64;
  static bool configured[kMaxDev] = {};  // the attribute is per device and function
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    if (fa.numRegs < static_cast<int>(FwdRegs<SPARSE>::kLaunchRegs)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  kern<<<p.n_items, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, bool causal, bool sparse, bool partial, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                       cudaStream_t st) {
  // The alternating schedule of single-tile pairs is compiled into every dense
  // kernel; a launch whose pairs are all full runs an instantiation without
  // it (partial states, and the bf16 output at d=128, where that copy
  // compiles without register spills and measured 1.7 % faster; at d=64 the
  // copy with the path measured faster and serves every launch).  A launch
  // whose query rows fit one tile (decoding) runs the instantiation with a
  // single Q buffer and one more K stage.
  // d = 128 without block lists: the kernel with 256-key score tiles
  // (fwd_wide.cu), for partial states only where the chunks hold at least
  // 4096 keys.  Its items are one query tile against one chunk, and each
  // item's first S waits for its Q tile to arrive from DRAM; with short
  // chunks those waits dominate, and this kernel's two-tile items (half as
  // many) run faster: 8 chunks of 512 keys at B=4 H=16 L=4096 took 0.576 ms
  // there against 0.507 ms here, chunks of 2048 keys ran alike, and chunks of
  // 16384 keys 8 % faster there.
  // Block-sparse launches at d = 128 run it too, up to the key range its
  // bitmaps cover: at B=2 H=16 L'=16320 (causal) it ran lists of 6.5, 12.6,
  // 23.8 and 44.6 entries a row 4 %, 12 %, 17 % and 16 % faster than this
  // kernel.
  if (d == 128 && !sparse && (!partial || p.chunk_len >= 4096))
    return launch_fwd_wide(causal, partial, false, tq, tk, tv, p, st);
  if (d == 128 && sparse && !partial && fwd_wide_takes_sparse(p.Lk))
    return launch_fwd_wide(causal, false, true, tq, tk, tv, p, st);
  const bool single_tile_pair = (p.Lq % (2 * kTileM)) != 0 && (p.Lq % (2 * kTileM)) <= kTileM;
  const bool alt = !sparse && (single_tile_pair || (!partial && d == 64));
  const bool dec = alt && p.Lq >= 1 && p.Lq <= kTileM;
#define BSS_FWD_CASE(DD, CA, SP, PA, AL, DE)                                              \
  if (d == DD && causal == CA && sparse == SP && partial == PA && alt == AL && dec == DE) \
    return launch_one<DD, CA, SP, PA, AL, DE>(tq, tk, tv, p, st);
#define BSS_FWD_CASE_D(DD, CA, SP, PA, AL) \
  BSS_FWD_CASE(DD, CA, SP, PA, AL, false)  \
  BSS_FWD_CASE(DD, CA, SP, PA, AL, true)
  BSS_FWD_CASE(128, false, false, false, false, false)
  BSS_FWD_CASE(128, true, false, false, false, false)
  BSS_FWD_CASE_D(64, false, false, false, true)
  BSS_FWD_CASE_D(64, true, false, false, true)
  BSS_FWD_CASE_D(128, false, false, false, true)
  BSS_FWD_CASE_D(128, true, false, false, true)
  BSS_FWD_CASE_D(64, false, false, true, true)
  BSS_FWD_CASE_D(64, true, false, true, true)
  BSS_FWD_CASE_D(128, false, false, true, true)
  BSS_FWD_CASE_D(128, true, false, true, true)
  BSS_FWD_CASE(64, false, false, true, false, false)
  BSS_FWD_CASE(64, true, false, true, false, false)
  BSS_FWD_CASE(128, false, false, true, false, false)
  BSS_FWD_CASE(128, true, false, true, false, false)
  BSS_FWD_CASE(64, false, true, false, false, false)
  BSS_FWD_CASE(64, true, true, false, false, false)
  BSS_FWD_CASE(128, false, true, false, false, false)
  BSS_FWD_CASE(128, true, true, false, false, false)
#undef BSS_FWD_CASE_D
#undef BSS_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace bss
