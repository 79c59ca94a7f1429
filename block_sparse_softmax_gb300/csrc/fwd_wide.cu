// Fused attention forward for sm_103a at head dimension 128, dense, causal or
// block-sparse: the kernel attn_fwd and attn_fwd_blocksparse run for those
// launches (bf16 output), and attn_fwd_partial and attn_fwd_splitkv for their
// long key chunks (fp32 partial states).
//
// What it computes is what attn_fwd_kernel computes ("Exact Blocks, Rings,
// and Sparsity", section 2, 'What the forward kernel keeps on chip';
// "FlashAttention: Fast and Memory Efficient Exact Attention with IO
// Awareness", section 5.2): a query tile stays on chip while key/value tiles
// stream past, each block of scores is folded into the running state
// (m, l, A), and S and P never reach HBM.
//
// How it is laid out differently:
//   * a work item is ONE 128-row query tile; each step scores a PAIR of
//     128-key blocks with M128 N256 MMAs.  On GB300 an N=256 tcgen05.mma with
//     both operands in shared memory costs the tensor pipe about 170 cycles
//     against about 105 for an N=128 one, so a pair's scores take a fifth
//     less pipe time than two single blocks' (P V is N=128 either way);
//   * TMEM (512 columns): S (256 fp32) | P (256 keys as bf16 pairs, 128) |
//     O (128 fp32).  P has columns of its own, so the next pair's S is issued
//     as soon as the softmax holds the current S in registers, and its MMAs
//     run while the softmax computes the exponentials;
//   * both softmax warpgroups work on the one tile: warpgroup X takes key
//     block X of every pair (S columns 128X ..), and the two exchange their
//     rows' block maxima through shared memory (mbarriers with bounded
//     waits) so that both use one reference max.  Each keeps its own row sum,
//     writes its half of P, and rescales and stores its half of O's columns.
//     P V runs block by block: block X's 8 MMAs wait for warpgroup X's P
//     only, and their completion frees only block X's P columns, so
//     warpgroup 0 writes the next P while block 1's MMAs still run (an O
//     rescale still waits for both);
//   * shared memory: Q (32 KB) | two stages of key-block pairs (64 KB each;
//     the two blocks' 64-column chunks interleaved, so that one descriptor of
//     256 rows covers the pair) | two V tile stages (32 KB each).  The
//     producer keeps K one step ahead of V;
//   * persistent: one CTA per SM takes item after item by cluster launch
//     control, as attn_fwd_kernel does; under a causal mask the tiles that
//     see the most keys come first;
//   * block-sparse ("Exact Blocks, Rings, and Sparsity", section 5; the
//     block-sparse attention patterns page, 'Block-sparse attention'): the
//     listed blocks of the tile's query block, as a set (duplicates and order
//     do not matter), in ascending order, taken two at a time; an odd last
//     block is scored alone (N=128) and its P V takes one V tile.  Warp 3
//     claims each next item and builds its bitmap (one bit per key block) in
//     the other of two buffers while the current item runs.
#include "common.cuh"

namespace bss {
namespace {

template <bool SPARSE>
struct WideCfg {
  static constexpr int D = 128;
  static constexpr int kChunks = D / 64;                   // 128-byte swizzle atoms across d
  static constexpr int kChunkBytes = kTileM * 128;         // 128 rows x 64 d
  static constexpr int kTileBytes = kTileM * D * 2;        // one 128-row tile
  static constexpr int kPairBytes = 2 * kTileBytes;        // two key blocks
  static constexpr int kStagesK = 2;                       // key-block pairs
  static constexpr int kStagesV = 2;                       // V tiles
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTileBytes;
  static constexpr int kVOff = kKOff + kStagesK * kPairBytes;
  static constexpr int kBarOff = kVOff + kStagesV * kTileBytes;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarQEmpty = 1;
  static constexpr int kBarKFull = 2;       // [2]
  static constexpr int kBarKEmpty = 4;      // [2]
  static constexpr int kBarVFull = 6;       // [2]
  static constexpr int kBarVEmpty = 8;      // [2]
  static constexpr int kBarSFull = 10;      // a pair's S in TMEM
  static constexpr int kBarSFree = 11;      // ... read into registers by both warpgroups
  // [2] P of key block X written by warpgroup X; block 0's also waits for
  // warpgroup 1's rescale of its half of O (the P V of block 0 writes all of O)
  static constexpr int kBarPFull = 12;
  static constexpr int kBarPvDone = 14;     // [2] a pair's P V of block X completed (P block X free)
  static constexpr int kBarXch = 16;        // [2] row values exchanged, by parity
  static constexpr int kBarOFull = 18;
  static constexpr int kBarOEmpty = 19;
  static constexpr int kBarItemFull = 20;   // [2]
  static constexpr int kBarItemEmpty = 22;  // [2]
  static constexpr int kBarClc = 24;
  static constexpr int kBarMmaDone = 25;
  static constexpr int kBarBmEmpty = 26;    // [2] block-sparse: an item's bitmap walked by every role
  static constexpr int kNumBars = 26 + (SPARSE ? 2 : 0);
  // cancel answer (16) | TMEM base | abort flag | next item [2]
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kClcOff = kMiscOff;
  static constexpr int kTmemSlotOff = kMiscOff + 16;
  static constexpr int kAbortOff = kMiscOff + 20;
  static constexpr int kNextItemOff = kMiscOff + 24;
  // exchanged row values: [parity][warpgroup][128 rows] fp32
  static constexpr int kXchOff = kMiscOff + 32;
  static constexpr int kXchBytes = 2 * 2 * kTileM * 4;
  // block-sparse: the bitmaps of two items follow (one word per 32 key
  // blocks of the launch each)
  static constexpr int kPayload = kXchOff + kXchBytes;
  static constexpr int kBitmapOff = kPayload;
  static_assert(kMiscOff % 16 == 0, "the cancel answer needs 16-byte alignment");
  static_assert(kPayload <= 232448, "forward shared memory exceeds the 227 KB a CTA may use");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;      // S: 256 fp32 columns (key block X at 128 X)
  static constexpr uint32_t kColP = 256;    // P: 256 keys, bf16 pairs (block X at 256 + 64 X)
  static constexpr uint32_t kColO = 384;    // O: 128 fp32 columns (half X at 384 + 64 X)
  static constexpr int kThreads = 384;
  // readers of each next-item slot: the MMA thread and one lane of each
  // softmax warp (and the producer in a block-sparse launch, where warp 3
  // writes the slots); the walkers of a block-sparse item's bitmap: the
  // producer, the MMA thread and one lane of each softmax warp
  static constexpr int kItemReaders = 1 + 8 + (SPARSE ? 1 : 0);
  static constexpr int kBmWalkers = 1 + 1 + 8;
};

// Shared memory a launch takes: the layout's bytes plus alignment slack.  The
// layout may leave less than 1024 bytes of slack; the kernel relies on the
// dynamic shared memory base being 1024-aligned and checks, before touching
// anything, that its offset from that boundary fits the slack.
__host__ __device__ constexpr int wide_slack(int used) {
  return used + 1024 <= 232448 ? 1024 : 232448 - used;
}
template <bool SPARSE>
__host__ __device__ constexpr int wide_used(int bitmap_words) {
  return WideCfg<SPARSE>::kPayload + (SPARSE ? 2 * 4 * bitmap_words : 0);
}
// key blocks a block-sparse launch of this kernel addresses (longer key
// ranges run attn_fwd_kernel)
constexpr int kWideMaxSparseBlocks = 2048;
static_assert(wide_slack(wide_used<true>(kWideMaxSparseBlocks / 32)) >= 256,
              "the bitmaps leave too little alignment slack");
static_assert(wide_slack(wide_used<false>(0)) >= 256, "too little alignment slack");

// Block-sparse bitmaps.  The first listed block after `after` (-1: none).
__device__ __forceinline__ int bm_next(const uint32_t* bm, int words, int after) {
  const int c = after + 1;
  int w = c >> 5;
  if (w >= words) return -1;
  uint32_t bits = bm[w] & (0xFFFFFFFFu << (c & 31));
  while (bits == 0u) {
    if (++w >= words) return -1;
    bits = bm[w];
  }
  return (w << 5) + __ffs(bits) - 1;
}
__device__ __forceinline__ int bm_count(const uint32_t* bm, int words) {
  int n = 0;
  for (int w = 0; w < words; ++w) n += __popc(bm[w]);
  return n;
}

// Register split per warpgroup (as in attn_fwd_kernel): warpgroup 0 (TMA and
// scheduler, MMA, two idle warps) 136 registers a thread, the two softmax
// warpgroups 184; the launch holds 168 a thread.
constexpr uint32_t kWideLow = 136;
constexpr uint32_t kWideHigh = 184;
constexpr uint32_t kWideLaunchRegs = 168;
static_assert(kWideLow + 2 * kWideHigh <= 512, "register split exceeds an SM sub-partition");
static_assert(128 * kWideLow + 256 * kWideHigh <= 384 * kWideLaunchRegs,
              "register split exceeds the launch");

// One work item: a 128-row query tile of one (b, h) against one key chunk
// (every key when the launch has one chunk).  Items come in groups of
// p.head_group query heads; inside a group tile-major, then chunk, with the
// heads side by side, and under a causal mask the last tile (whose rows see
// the most keys) first.
struct WideItem {
  int b, h, bh, hkv;
  int c;           // key chunk
  int kbase;       // row of the chunk's first key in K and V
  int Lkc;         // keys in the chunk
  long long koff;  // absolute position of the chunk's first key (causal mask)
  int r0;          // first query row
  int kbmax;       // last key block (of the chunk) the tile can see (-1: none)
  int ns;          // steps: pairs of key blocks (2k, 2k + 1) of the chunk
};

// A launch with a bf16 output (CHUNKED false) has one chunk holding every key.
template <bool CAUSAL, bool CHUNKED>
__device__ __forceinline__ WideItem wide_item(int item, const FwdParams& p, int n_tiles) {
  WideItem it;
  const int BH = p.B * p.H;
  const int gh = p.head_group;
  const int chunks = CHUNKED ? p.n_chunks : 1;
  const int per_group = gh * chunks * n_tiles;
  const int grp = item / per_group;
  const int gsz = min(gh, BH - grp * gh);
  const int within = item - grp * per_group;
  const int per_rank = gsz * chunks;
  const int rank = within / per_rank;
  const int rem = within - rank * per_rank;
  it.c = CHUNKED ? rem / gsz : 0;
  it.bh = grp * gh + (rem - it.c * gsz);
  it.b = it.bh / p.H;
  it.h = it.bh - it.b * p.H;
  it.hkv = it.h / (p.H / p.Hkv);
  it.kbase = CHUNKED ? it.c * p.chunk_len : 0;
  it.Lkc = CHUNKED ? min(p.chunk_len, p.Lk - it.kbase) : p.Lk;
  it.koff = CHUNKED ? p.k_offset + it.kbase : p.k_offset;
  const int tile = CAUSAL ? (n_tiles - 1 - rank) : rank;
  it.r0 = tile * kTileM;
  const int nk = it.Lkc > 0 ? (it.Lkc + kTileN - 1) / kTileN : 0;
  if (it.r0 >= p.Lq || nk == 0) {
    it.kbmax = -1;
  } else if (CAUSAL) {
    const long long r_last = min(it.r0 + kTileM - 1, p.Lq - 1);
    const long long lim = r_last + p.q_offset - it.koff;
    it.kbmax = lim < 0 ? -1 : static_cast<int>(lim / kTileN < nk - 1 ? lim / kTileN : nk - 1);
  } else {
    it.kbmax = nk - 1;
  }
  it.ns = (it.kbmax + 2) / 2;
  return it;
}

// The next pair of a block-sparse item's blocks (b1 = -1: b0 is alone; b0 =
// -1: none left); `cur` is the last block taken.
__device__ __forceinline__ void bm_pair(const uint32_t* bm, int words, int& cur, int& b0, int& b1) {
  b0 = bm_next(bm, words, cur);
  b1 = b0 >= 0 ? bm_next(bm, words, b0) : -1;
  cur = b1 >= 0 ? b1 : b0;
}

// One bit in `bm` (cleared) per block of the item's list: entries out of
// range are reported and skipped, and so are blocks past the last one the
// tile can see (the causal future).  Threads i0, i0 + step, ... share the
// entries.
template <bool CAUSAL>
__device__ void wide_build_bitmap(const WideItem& it, const FwdParams& p, int nk, uint32_t* bm, int i0,
                                  int step) {
  if (it.kbmax < 0) return;
  const int qb = it.r0 / kTileM;
  if (qb >= p.n_qblk) return;
  const int* rp = p.row_ptr + static_cast<size_t>(it.bh / p.heads_per_list) * (p.n_qblk + 1) + qb;
  const int beg = __ldg(rp);
  const int end = __ldg(rp + 1);
  if (beg < 0 || end < beg || end > p.nnz) {
    if (i0 == 0) record_error(p.err, ATTN_ERR_BAD_BLOCKLIST);
    return;
  }
  for (int e = beg + i0; e < end; e += step) {
    const int c = __ldg(p.col_idx + e);
    if (c < 0 || c >= nk) {
      record_error(p.err, ATTN_ERR_BAD_BLOCKLIST);
      continue;
    }
    if (c <= it.kbmax) atomicOr(bm + (c >> 5), 1u << (c & 31));
  }
}

template <bool CAUSAL, bool PARTIAL, bool SPARSE>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  static_assert(!(PARTIAL && SPARSE), "partial states of block-sparse launches are not built");
  using C = WideCfg<SPARSE>;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  const int nk_all = (p.Lk + kTileN - 1) / kTileN;   // key blocks of the launch
  const int bw = SPARSE ? (nk_all + 31) >> 5 : 0;     // bitmap words an item
  {
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if (pad > static_cast<uint32_t>(wide_slack(wide_used<SPARSE>(bw))) ||
        (SPARSE && nk_all > kWideMaxSparseBlocks)) {  // layout would not fit: report, touch nothing
      if (threadIdx.x == 0) record_error(p.err, ATTN_ERR_UNSUPPORTED);
      return;
    }
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::kTmemSlotOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);
  volatile int* next_item = reinterpret_cast<volatile int*>(smem + C::kNextItemOff);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + C::kBitmapOff);
  // the bitmap of the n-th item a CTA runs
  auto item_bm = [&](int n) -> const uint32_t* { return bitmap + (n & 1) * bw; };

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int tid = static_cast<int>(threadIdx.x);
  // A launch whose earlier CTAs already timed out stops at once.
  if (*reinterpret_cast<volatile int*>(p.err) == ATTN_ERR_TIMEOUT) return;
  const int n_tiles = (p.Lq + kTileM - 1) / kTileM;

  if (tid == 0) {
    mbar_init(bar(C::kBarQFull), 1);
    mbar_init(bar(C::kBarQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
      mbar_init(bar(C::kBarVFull + s), 1);
      mbar_init(bar(C::kBarVEmpty + s), 1);
      mbar_init(bar(C::kBarXch + s), 2 * 4 * 32);
      mbar_init(bar(C::kBarItemFull + s), 1);
      mbar_init(bar(C::kBarItemEmpty + s), C::kItemReaders);
      if (SPARSE) mbar_init(bar(C::kBarBmEmpty + s), C::kBmWalkers);
    }
    mbar_init(bar(C::kBarSFull), 1);
    mbar_init(bar(C::kBarSFree), 2 * 4 * 32);
    mbar_init(bar(C::kBarPFull + 0), 2 * 4 * 32);
    mbar_init(bar(C::kBarPFull + 1), 4 * 32);
    mbar_init(bar(C::kBarPvDone + 0), 1);
    mbar_init(bar(C::kBarPvDone + 1), 1);
    mbar_init(bar(C::kBarOFull), 1);
    mbar_init(bar(C::kBarOEmpty), 2 * 4 * 32);
    mbar_init(bar(C::kBarClc), 1);
    mbar_init(bar(C::kBarMmaDone), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + C::kTmemSlotOff, C::kTmemCols);
    tmem_relinquish();
  }
  if (SPARSE) {
    // the first item's bitmap, by every thread; later items' come from warp 3
    for (int i = tid; i < 2 * bw; i += C::kThreads) bitmap[i] = 0u;
    __syncthreads();
    wide_build_bitmap<CAUSAL>(wide_item<CAUSAL, false>(static_cast<int>(blockIdx.x), p, n_tiles), p,
                              nk_all, bitmap, tid, C::kThreads);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    regs_set<kWideLow, kWideLaunchRegs>();
    if (warp == 0) {
      // =================== TMA producer and item scheduler ===================
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        int item = static_cast<int>(blockIdx.x);
        int n = 0;              // items finished
        int ik = 0, iv = 0;     // pair stages and V tiles loaded (over all items)
        int qn = 0;             // Q tiles loaded
        int clc_k = 0;          // cancel requests answered
        bool clc_live = !SPARSE;  // a block-sparse launch's items are claimed by warp 3
        bool clc_out = false;   // a cancel request is in flight
        bool ok = true;
        auto request_item = [&]() {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bar(C::kBarClc), 16);
          clc_try_cancel(sbase + C::kClcOff, bar(C::kBarClc));
          clc_out = true;
        };
        // a pair of key blocks of the item's chunk: 2k, 2k + 1 (a block past
        // the chunk reads the next chunk's keys or the zero fill; the softmax
        // masks it), or two listed blocks (b1 = -1: b0 alone)
        auto load_k = [&](const WideItem& it, int b0, int b1) -> bool {
          const int s = ik % C::kStagesK;
          if (ik >= C::kStagesK &&
              !wait_bar(bar(C::kBarKEmpty + s), ((ik / C::kStagesK) & 1) ^ 1, abort_flag, p.err))
            return false;
          const bool two = !SPARSE || b1 >= 0;
          const uint32_t ks = sbase + C::kKOff + s * C::kPairBytes;
          mbar_arrive_expect_tx(bar(C::kBarKFull + s), two ? C::kPairBytes : C::kTileBytes);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t == 1 && !two) break;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_4d(ks + c * 2 * C::kChunkBytes + t * C::kChunkBytes, &tmK, bar(C::kBarKFull + s),
                          c * 64, it.kbase + (t ? b1 : b0) * kTileN, it.hkv, it.b);
          }
          ++ik;
          return true;
        };
        auto load_v = [&](const WideItem& it, int kb) -> bool {
          const int s = iv % C::kStagesV;
          if (iv >= C::kStagesV &&
              !wait_bar(bar(C::kBarVEmpty + s), ((iv / C::kStagesV) & 1) ^ 1, abort_flag, p.err))
            return false;
          const uint32_t vs = sbase + C::kVOff + s * C::kTileBytes;
          mbar_arrive_expect_tx(bar(C::kBarVFull + s), C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(vs + c * C::kChunkBytes, &tmV, bar(C::kBarVFull + s), c * 64,
                        it.kbase + kb * kTileN, it.hkv, it.b);
          ++iv;
          return true;
        };
        while (ok) {
          const WideItem it = wide_item<CAUSAL, PARTIAL>(item, p, n_tiles);
          const uint32_t* bm = item_bm(n);
          const int ns = SPARSE ? (bm_count(bm, bw) + 1) / 2 : it.ns;
          if (ns > 0) {
            // one Q buffer: the previous item's last S must have read it
            if (qn > 0 && !wait_bar(bar(C::kBarQEmpty), (qn - 1) & 1, abort_flag, p.err)) break;
            mbar_arrive_expect_tx(bar(C::kBarQFull), C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_4d(sbase + C::kQOff + c * C::kChunkBytes, &tmQ, bar(C::kBarQFull), c * 64, it.r0,
                          it.h, it.b);
            ++qn;
            // K runs one step ahead of V
            int cur = -1, a0 = 0, a1 = 1;   // the blocks of the pair whose K was loaded last
            if (SPARSE) bm_pair(bm, bw, cur, a0, a1);
            ok = load_k(it, a0, a1);
            for (int k = 0; k < ns && ok; ++k) {
              if (k == ns - 1 && clc_live) request_item();   // the next item, as this one's last loads go
              const int v0 = a0, v1 = a1;
              if (k + 1 < ns) {
                if (SPARSE) {
                  bm_pair(bm, bw, cur, a0, a1);
                } else {
                  a0 = 2 * k + 2;
                  a1 = 2 * k + 3;
                }
                ok = load_k(it, a0, a1);
              }
              if (ok) ok = load_v(it, v0) && ((SPARSE && v1 < 0) || load_v(it, v1));
            }
            if (!ok) break;
          }
          if (SPARSE) {
            // this item's bitmap is walked; its buffer may take the item after next
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
          if (clc_live && !clc_out) request_item();   // an item without keys
          int next = -1;
          if (clc_out) {
            if (!wait_bar(bar(C::kBarClc), clc_k & 1, abort_flag, p.err)) break;
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
          if (n >= 2 && !wait_bar(bar(C::kBarItemEmpty + s), ((n >> 1) & 1) ^ 1, abort_flag, p.err))
            break;
          next_item[s] = next;
          mbar_arrive(bar(C::kBarItemFull + s));
          ++n;
          if (next < 0) break;
          item = next;
        }
        // every copy issued has landed before the CTA may exit
        for (int j = max(0, ik - C::kStagesK); j < ik; ++j)
          drain_bar(bar(C::kBarKFull + j % C::kStagesK), (j / C::kStagesK) & 1);
        for (int j = max(0, iv - C::kStagesV); j < iv; ++j)
          drain_bar(bar(C::kBarVFull + j % C::kStagesV), (j / C::kStagesV) & 1);
        if (qn > 0) drain_bar(bar(C::kBarQFull), (qn - 1) & 1);
        if (clc_out) drain_bar(bar(C::kBarClc), clc_k & 1);
      }
    } else if (warp == 1) {
      // =================== MMA issuer (one thread) ===================
      // Per item: S_0, then for every step k: S_{k+1} (as soon as both
      // softmax warpgroups hold S_k in registers) and P_k V_k.  S, P and O
      // have columns of their own, and one thread's MMAs run in issue order.
      if (lane == 0) {
        constexpr uint32_t kIdescS = idesc_bf16_f32(kTileM, 2 * kTileN, false, false);
        constexpr uint32_t kIdescS1 = idesc_bf16_f32(kTileM, kTileN, false, false);   // a block alone
        constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileM, D, false, true);
        const uint64_t dq = sdesc_sw128(sbase + C::kQOff, 16, 1024);
        int item = static_cast<int>(blockIdx.x);
        int n = 0;              // items finished
        int ik = 0, iv = 0;     // pair stages and V tiles consumed
        int qn = 0;             // Q tiles consumed
        int sn = 0;             // S tiles issued
        int pn = 0;             // P tiles consumed
        int on = 0;             // O results handed to the epilogue
        bool ok = true;
        auto issue_s = [&](bool last, bool alone) -> bool {
          if (sn > 0 && !wait_bar(bar(C::kBarSFree), (sn - 1) & 1, abort_flag, p.err)) return false;
          const int s = ik % C::kStagesK;
          if (!wait_bar(bar(C::kBarKFull + s), (ik / C::kStagesK) & 1, abort_flag, p.err)) return false;
          tc_fence_after();
          const uint64_t dk = sdesc_sw128(sbase + C::kKOff + s * C::kPairBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qoff = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * 2 * C::kChunkBytes + (kk & 3) * 32;
            mma_ss(tmem + C::kColS, sdesc_add(dq, qoff), sdesc_add(dk, koff),
                   (SPARSE && alone) ? kIdescS1 : kIdescS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kBarSFull));
          mma_commit(bar(C::kBarKEmpty + s));
          if (last) mma_commit(bar(C::kBarQEmpty));   // Q is free for the next item
          ++ik;
          ++sn;
          return true;
        };
        // P V block by block: block X's MMAs go as soon as warpgroup X has
        // written its P, and their completion frees that block's P columns
        auto issue_pv = [&](bool first, bool alone) -> bool {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!wait_bar(bar(C::kBarPFull + t), pn & 1, abort_flag, p.err)) return false;
            tc_fence_after();
            if (t == 0 && first && on > 0) {
              // O still holds the previous item's result until its epilogue read it
              if (!wait_bar(bar(C::kBarOEmpty), (on - 1) & 1, abort_flag, p.err)) return false;
              tc_fence_after();
            }
            if (!(SPARSE && alone && t == 1)) {
              const int s = iv % C::kStagesV;
              if (!wait_bar(bar(C::kBarVFull + s), (iv / C::kStagesV) & 1, abort_flag, p.err)) return false;
              tc_fence_after();
              const uint64_t dv = sdesc_sw128(sbase + C::kVOff + s * C::kTileBytes, C::kChunkBytes, 1024);
#pragma unroll
              for (int kk = 0; kk < kTileN / 16; ++kk)
                mma_ts(tmem + C::kColO, tmem + C::kColP + (t * 8 + kk) * 8, sdesc_add(dv, kk * 16 * 128),
                       kIdescPV, (!first || t > 0 || kk > 0) ? 1u : 0u);
              mma_commit(bar(C::kBarVEmpty + s));
              ++iv;
            }
            mma_commit(bar(C::kBarPvDone + t));
          }
          ++pn;
          return true;
        };
        while (ok) {
          const WideItem it = wide_item<CAUSAL, PARTIAL>(item, p, n_tiles);
          int ns = it.ns;
          bool odd = false;     // block-sparse: the last pair is one block
          if (SPARSE) {
            const int nb = bm_count(item_bm(n), bw);
            mbar_arrive(bar(C::kBarBmEmpty + (n & 1)));
            ns = (nb + 1) / 2;
            odd = (nb & 1) != 0;
          }
          if (ns > 0) {
            if (!wait_bar(bar(C::kBarQFull), qn & 1, abort_flag, p.err)) break;
            ++qn;
            ok = issue_s(ns == 1, odd && ns == 1);
            for (int k = 0; k < ns && ok; ++k) {
              if (k + 1 < ns) ok = issue_s(k + 1 == ns - 1, odd && k + 1 == ns - 1);
              if (ok) ok = issue_pv(k == 0, odd && k == ns - 1);
            }
            if (!ok) break;
            mma_commit(bar(C::kBarOFull));
            ++on;
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
      // =================== block-sparse item preparation ===================
      // Item k (k >= 1) of this CTA: claimed by cluster launch control, its
      // bitmap built in buffer k & 1, and its index written to ring slot
      // (k - 1) & 1, which every role reads at the end of item k - 1.  The
      // buffer last held item k - 2, so the claim comes as soon as every role
      // has walked that item: about one item ahead.
      bool live = true;       // false: every item claimed
      int clc_k = 0;          // cancel requests answered
      bool clc_out = false;   // a cancel request is in flight
      for (int k = 1;; ++k) {
        const int s = (k - 1) & 1;
        const int b = k & 1;
        // the slot's previous entry (item k - 2) has been read by every role
        if (k >= 3 && !__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarItemEmpty + s),
                                                        (((k - 1) >> 1) & 1) ^ 1, abort_flag, p.err)))
          break;
        int next = -1;
        if (live) {
          // the buffer's previous item (k - 2) has been walked by every role
          if (k >= 2 && !__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarBmEmpty + b), ((k - 2) >> 1) & 1,
                                                          abort_flag, p.err)))
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
            live = false;     // nothing left to take (no request follows a failed one)
        }
        if (next >= 0) {
          uint32_t* bmk = bitmap + b * bw;
          for (int i = lane; i < bw; i += 32) bmk[i] = 0u;
          __syncwarp();
          wide_build_bitmap<CAUSAL>(wide_item<CAUSAL, false>(next, p, n_tiles), p, nk_all, bmk, lane, 32);
          __threadfence_block();
          __syncwarp();
        }
        if (lane == 0) {
          next_item[s] = next;
          mbar_arrive(bar(C::kBarItemFull + s));   // releases the bitmap built above
        }
        if (next < 0) break;
      }
      if (lane == 0 && clc_out) drain_bar(bar(C::kBarClc), clc_k & 1);
    }
  } else {
    regs_set<kWideHigh, kWideLaunchRegs>();
    // =================== softmax warpgroups: X = 0 (warps 4-7), 1 (warps 8-11) ===================
    const int X = (warp - 4) >> 2;                // key block X of every pair
    const int wq = warp & 3;                      // TMEM lane quarter of this warp
    const int row_in_tile = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kColS + X * 128;
    const uint32_t tP = tmem + lane_base + C::kColP + X * 64;
    const uint32_t tO = tmem + lane_base + C::kColO + X * 64;
    const float sl2 = p.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    float* xch = reinterpret_cast<float*>(smem + C::kXchOff);

    int item = static_cast<int>(blockIdx.x);
    int n = 0;          // items finished
    int cnt = 0;        // S tiles consumed (over all items)
    int nx = 0;         // row values exchanged
    int on = 0;         // O results read
    bool ok = true;
    // hand this row's value to the other warpgroup and take its value back
    auto exchange = [&](float v, float& other) -> bool {
      float* xb = xch + (nx & 1) * 2 * kTileM;
      xb[X * kTileM + row_in_tile] = v;
      mbar_arrive(bar(C::kBarXch + (nx & 1)));
      const bool w = __all_sync(0xFFFFFFFFu,
                                wait_bar(bar(C::kBarXch + (nx & 1)), (nx >> 1) & 1, abort_flag, p.err));
      other = xb[(1 - X) * kTileM + row_in_tile];
      ++nx;
      return w;
    };
    while (ok) {
      const WideItem it = wide_item<CAUSAL, PARTIAL>(item, p, n_tiles);
      const int row = it.r0 + row_in_tile;
      const uint32_t* bm = item_bm(n);
      const int ns = SPARSE ? (bm_count(bm, bw) + 1) / 2 : it.ns;
      int cur = -1;           // block-sparse: the last block walked
      float m2 = NEG_INF;     // reference max (log2 units), moved only by > 8
      float mt = NEG_INF;     // exact running max (log2 units)
      float l = 0.f;          // this warpgroup's part of the row sum
      for (int k = 0; k < ns; ++k) {
        int blk = 2 * k + X;  // this warpgroup's key block of the pair (-1: none)
        if (SPARSE) {
          int b0, b1;
          bm_pair(bm, bw, cur, b0, b1);
          blk = X ? b1 : b0;
        }
        if (!__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarSFull), cnt & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);
        // S is in registers: the next pair's S may overwrite its columns
        tc_fence_before();
        mbar_arrive(bar(C::kBarSFree));

        // element mask: where the block crosses the diagonal or the end of
        // the chunk (a block wholly past either, or missing from a
        // block-sparse pair, is masked out entirely)
        // (a launch with one chunk reads the key count and offset from the
        // kernel parameters)
        const int Lkc = PARTIAL ? it.Lkc : p.Lk;
        const long long koff = PARTIAL ? it.koff : p.k_offset;
        const bool none = SPARSE && blk < 0;
        const int kstart = (none ? 0 : blk) * kTileN;
        const bool edge = none || (kstart + kTileN > Lkc) ||
                          (CAUSAL && (static_cast<long long>(kstart) + kTileN - 1 + koff >
                                      static_cast<long long>(it.r0) + p.q_offset));
        if (edge) {
          long long lim = static_cast<long long>(Lkc) - 1 - kstart;
          if (CAUSAL) lim = min(lim, static_cast<long long>(row) + p.q_offset - koff - kstart);
          if (none) lim = -1;
          const int jl = static_cast<int>(max(-1ll, min(127ll, lim)));
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j > jl) s[c][j] = __float_as_uint(NEG_INF);
        }
        // row max of this block over 8 chains of three-input max
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
        const float mmine = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
        // the pair's row max: both warpgroups take the same decisions below
        float mothr;
        if (!exchange(mmine, mothr)) {
          ok = false;
          break;
        }
        const float mblk = fmaxf(mmine, mothr);
        mt = fmaxf(mt, mblk);
        float alpha = 1.f;
        bool moved = false;
        if (mblk > m2 + 8.f) {
          alpha = ex2(m2 - mblk);
          m2 = mblk;
          moved = true;
        }
        const float mu = (m2 == NEG_INF) ? 0.f : m2;
        // Where the reference max moved, this warpgroup's half of O is
        // rescaled: after the previous pair's whole P V (both blocks write
        // all of O).  Warpgroup 1 does it first and then releases block 0's
        // P V; warpgroup 0 after writing its P, before releasing it.
        const bool fix = moved && k > 0;
        const bool any_fix = __any_sync(0xFFFFFFFFu, fix);
        auto rescale_o = [&]() -> bool {
          if (!__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarPvDone + 1), (cnt - 1) & 1, abort_flag, p.err)))
            return false;
          tc_fence_after();
          const float a = fix ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * a);
            tmem_st32(tO + c * 32, o);
          }
          return true;
        };
        if (X == 1) {
          if (any_fix && !rescale_o()) {
            ok = false;
            break;
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(C::kBarPFull + 0));
        }
        // P block X is written below: the previous pair's P V of block X
        // (which reads it) must have completed
        if (cnt > 0 &&
            !__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarPvDone + X), (cnt - 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
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
        if (X == 0 && any_fix && !rescale_o()) {
          ok = false;
          break;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kBarPFull + X));
        ++cnt;
      }
      if (!ok) break;
      if (SPARSE) {
        // this item's bitmap is walked
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kBarBmEmpty + (n & 1)));
      }

      // ---- epilogue: the row sum is the two warpgroups' parts; each writes
      // its half of the row's columns ----
      uint32_t o[2][32];
      float lt = 0.f;
      if (ns > 0) {
        float lo;
        if (!exchange(l, lo)) break;
        lt = l + lo;
        if (!__all_sync(0xFFFFFFFFu, wait_bar(bar(C::kBarOFull), on & 1, abort_flag, p.err))) break;
        tc_fence_after();
        tmem_ld32(tO, o[0]);
        tmem_ld32(tO + 32, o[1]);
        tmem_ld_wait(o[0]);
        tmem_ld_wait(o[1]);
        tc_fence_before();
        mbar_arrive(bar(C::kBarOEmpty));
        ++on;
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) o[c][j] = 0u;
      }
      const bool inb = row < p.Lq;
      // the states of chunk c follow those of chunks 0 .. c-1
      const size_t rows0 = static_cast<size_t>(it.c) * p.B * p.H * p.Lq + static_cast<size_t>(it.bh) * p.Lq;
      const size_t wrow0 = rows0 + (it.r0 + wq * 32);
      if (PARTIAL) {
        // (m, l, acc) referred to the exact row max; an empty state (m = -inf)
        // is fully described by m and l, and its acc row is not written (a
        // merge never reads it)
        const float factor = (mt == NEG_INF || ns == 0) ? 0.f : ex2(m2 - mt);
        const uint32_t valid = __ballot_sync(0xFFFFFFFFu, inb && ns > 0 && mt != NEG_INF);
        if (valid) {
          uint8_t* base = reinterpret_cast<uint8_t*>(p.acc_out + wrow0 * D) + X * 256;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[c][j] = __float_as_uint(__uint_as_float(o[c][j]) * factor);
            transpose_octets(o[c], lane);
            store_octet_lines(o[c], base + c * 128, D * 4, valid, lane);
          }
        }
        if (X == 0 && inb) {
          p.m_out[rows0 + row] = (mt == NEG_INF) ? NEG_INF : mt * kLn2;
          p.l_out[rows0 + row] = lt * factor;
        }
      } else {
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const uint32_t valid = __ballot_sync(0xFFFFFFFFu, inb);
        uint8_t* base = reinterpret_cast<uint8_t*>(p.o + wrow0 * D) + X * 128;
        uint32_t w[32];
#pragma unroll
        for (int kq = 0; kq < 32; ++kq) {
          const int c = kq / 16;
          const int j = (2 * kq) % 32;
          w[kq] = pack_bf16(__uint_as_float(o[c][j]) * inv, __uint_as_float(o[c][j + 1]) * inv);
        }
        transpose_octets(w, lane);
        store_octet_lines(w, base, D * 2, valid, lane);
        if (X == 0 && inb) p.lse[rows0 + row] = lt > 0.f ? (m2 + __log2f(lt)) * kLn2 : NEG_INF;
      }
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

template <bool CAUSAL, bool PARTIAL, bool SPARSE>
cudaError_t launch_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const FwdParams& p0, cudaStream_t st) {
  using C = WideCfg<SPARSE>;
  auto kern = attn_fwd_wide_kernel<CAUSAL, PARTIAL, SPARSE>;
  FwdParams p = p0;
  const long long items =
      static_cast<long long>(p.n_chunks) * p.B * p.H * ((p.Lq + kTileM - 1) / kTileM);
  if (items > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  p.n_items = static_cast<int>(items);
  if (p.n_items == 0) return cudaSuccess;
  const int nk = (p.Lk + kTileN - 1) / kTileN;
  if (SPARSE && nk > kWideMaxSparseBlocks) return cudaErrorInvalidValue;
  const int used = wide_used<SPARSE>(SPARSE ? (nk + 31) / 32 : 0);
  const int smem = used + wide_slack(used);
  constexpr int kMaxUsed = wide_used<SPARSE>(SPARSE ? kWideMaxSparseBlocks / 32 : 0);
  constexpr int kMaxSmem = kMaxUsed + wide_slack(kMaxUsed);
  constexpr int kMaxDev = 64;
  static bool configured[kMaxDev] = {};  // the attribute is per device and function
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    if (fa.numRegs < static_cast<int>(kWideLaunchRegs)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  kern<<<p.n_items, C::kThreads, smem, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

bool fwd_wide_takes_sparse(int Lk) {
  return (static_cast<long long>(Lk) + kTileN - 1) / kTileN <= kWideMaxSparseBlocks;
}

cudaError_t launch_fwd_wide(bool causal, bool partial, bool sparse, const CUtensorMap& tq,
                            const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                            cudaStream_t st) {
  if (sparse) {
    if (partial) return cudaErrorInvalidValue;
    return causal ? launch_wide<true, false, true>(tq, tk, tv, p, st)
                  : launch_wide<false, false, true>(tq, tk, tv, p, st);
  }
  if (partial)
    return causal ? launch_wide<true, true, false>(tq, tk, tv, p, st)
                  : launch_wide<false, true, false>(tq, tk, tv, p, st);
  return causal ? launch_wide<true, false, false>(tq, tk, tv, p, st)
                : launch_wide<false, false, false>(tq, tk, tv, p, st);
}

}  // namespace bss
