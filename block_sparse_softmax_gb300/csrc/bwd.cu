// Attention backward by recomputation for sm_103a.
//
// What it computes ("Exact Blocks, Rings, and Sparsity", section 3;
// "FlashAttention: Fast and Memory Efficient Exact Attention with IO
// Awareness", section 5.3):
//   D_i  = dO_i . O_i                      (preprocess, from the saved O)
//   P    = exp(scale Q K^T - LSE)          (recomputed tile by tile, masked -> 0)
//   dV   = P^T dO,   dP = dO V^T,   dS = P o (dP - D)
//   dK   = scale dS^T Q,   dQ = scale dS K
// Three kernels run in stream order: preprocess (D, and clearing the fp32 dQ
// accumulator), the main kernel, and the dQ conversion to bf16.
//
// Main kernel design (the KV-owned traversal of section 3, 'The ownership
// conflict between dQ and dK, dV'): one CTA owns a 128-key tile of one (b, h)
// and keeps K_j, V_j in shared memory and dK_j, dV_j accumulating in TMEM
// while the query tiles stream past.  Scores are computed transposed (TMEM
// lane = key), so that one thread owns one key row:
//   S^T  = K_j Q_i^T   and   dP^T = V_j dO_i^T         (SS MMAs, M = 128 keys)
//   two warpgroups (64 query columns each) first turn S^T into P^T (bf16,
//   written back into the lower halves of S^T's own columns as the
//   tensor-memory A operand of dV), then, once dP^T is there, form dS and
//   store it (bf16) in shared memory in the 128-byte-swizzled layout of a
//   K-major tile with one key per row;
//   dV  += P^T dO_i                                     (TS MMA)
//   dK  += dS^T Q_i   (dS^T is that tile read K-major) (SS MMA)
//   dQ_i = dS K_j     (the same tile read M-major)      (SS MMA, M = queries)
//   four more warps move dQ_i out of TMEM through a shared staging buffer and
//   add it into the fp32 accumulator in global memory with bulk tensor
//   reduce-adds.
// One thread issues every MMA, in the order
//   dV(i), S^T(i+1), dQ(i), dK(i), dP^T(i+1)
// so that the tensor core works on dV(i) and S^T(i+1) while dS(i) is formed
// and on dK(i) while dQ(i) is drained: the chain that sets the pace is
// dQ(i) -> drain -> dP^T(i+1) -> dS(i+1) -> dQ(i+1), and the other MMAs fill
// its gaps.  dQ_i is written into dP^T's columns at d=128 (they are free once
// dS(i) has been formed) and into columns of its own at d=64.
// Causal: only query tiles i >= j are visited and the element mask is applied
// on the diagonal tile and on the ragged tail.
#include "common.cuh"

namespace bss {
namespace {

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = kTileM * 128;
  static constexpr int kTileBytes = kTileM * D * 2;
  static constexpr int kStagesQ = 2;                     // Q_i ring depth (S^T(i+1) and dK(i) overlap)
  static constexpr int kStagesDO = (D == 128) ? 1 : 2;    // dO_i ring depth (room for dQ staging)
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;
  static constexpr int kDOOff = kQOff + kStagesQ * kTileBytes;
  static constexpr int kDSOff = kDOOff + kStagesDO * kTileBytes;  // dS, 128 keys x 128 queries bf16
  static constexpr int kDSBytes = kTileM * kTileN * 2;
  static constexpr int kStageOff = kDSOff + kDSBytes;    // dQ staging: 128 rows x 64 fp32
  static constexpr int kStageBytes = kTileM * 64 * 4;
  static constexpr int kStatOff = kStageOff + kStageBytes;   // 2 x (lse2[128], delta[128])
  static constexpr int kColBmOff = kStatOff + 2 * 2 * 128 * 4;   // block-sparse: this key tile's column
  static constexpr int kColBmWords = kMaxKBlocks / 32;
  static constexpr int kBarOff = kColBmOff + kColBmWords * 4;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;
  static constexpr int kBarQEmpty = kBarQFull + kStagesQ;
  static constexpr int kBarDOFull = kBarQEmpty + kStagesQ;
  static constexpr int kBarDOEmpty = kBarDOFull + kStagesDO;
  static constexpr int kBarSFull = kBarDOEmpty + kStagesDO;   // S^T of a query tile in TMEM
  static constexpr int kBarDPFull = kBarSFull + 1;            // [2]: dP^T query half h in TMEM
  static constexpr int kBarPReady = kBarDPFull + 2;           // P^T written (S^T read)
  static constexpr int kBarDSReady = kBarPReady + 1;          // dS in shared memory (dP^T read)
  static constexpr int kBarDQFull = kBarDSReady + 1;
  static constexpr int kBarDQFree = kBarDQFull + 1;           // [2]: dQ d-columns [64r, 64r+64) read
  static constexpr int kBarDKVFull = kBarDQFree + 2;
  static constexpr int kBarMmaDone = kBarDKVFull + 1;
  static constexpr int kBarStat = kBarMmaDone + 1;     // [2]: LSE/D of a query tile staged
  static constexpr int kBarStaged = kBarStat + 2;      // dQ round staged (CTA-wide drain)
  static constexpr int kBarStageFree = kBarStaged + 1; // staging read by the reduce (CTA-wide drain)
  static constexpr int kNumBars = kBarStageFree + 1;
  // dQ drain: at d=128 each drain warp reduces its own 32 rows (no barrier
  // among the four warps, which frees dQ's columns for dP^T sooner); at d=64,
  // with one round per tile and a shorter period, one thread reduces all 128
  // rows in two larger boxes after a CTA-wide barrier (measured faster there).
  static constexpr bool kDrainPerWarp = (D == 128);
  static constexpr int kDrainBoxRows = kDrainPerWarp ? 32 : 128;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // Alignment slack for the 1024-byte aligned layout.  At d=128 the layout
  // leaves less than 1024 bytes: the kernel then relies on the dynamic shared
  // memory base being 1024-aligned and checks that before touching it.
  static constexpr int kPayload = kMiscOff + 16;
  static constexpr int kSlack = (kPayload + 1024 <= 232448) ? 1024 : 232448 - kPayload;
  static constexpr int kSmemBytes = kPayload + kSlack;
  static_assert(kPayload <= 232448, "backward shared memory exceeds the 227 KB a CTA may use");
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: S^T (fp32) at [0,128) and dP^T at [128,256).  Half X of the
  // P^T/dS warpgroups (query columns [64X, 64X+64)) writes its P^T (bf16
  // pairs, 32 columns) to S^T columns [64X, 64X+32), inside the range it has
  // itself already read.  dV and dK follow.  dQ of a query tile takes dP^T's
  // columns at d=128 and columns of its own, [384,448), at d=64.
  static constexpr uint32_t kColST = 0;
  static constexpr uint32_t kColDPT = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr uint32_t kColDQ = (D == 128) ? kColDPT : 384;
  static constexpr bool kDQOverDP = (kColDQ == kColDPT);
  // A operand address of query k-step kk (16 queries) inside P^T
  static __device__ __forceinline__ uint32_t pcol(int kk) { return 64 * (kk >> 2) + 8 * (kk & 3); }
  static constexpr int kThreads = 512;
};

// Register split per warpgroup (setmaxnreg): warpgroup 0 (TMA, MMA, two idle
// warps) kLow, the P/dS warpgroups 1-2 kMid (each thread keeps 64 fp32 P
// values between its two phases), the dQ warpgroup 3 kHigh.  96/160/160/96
// compiles every instantiation without register spills (88/160/160/104
// spilled a few bytes at d=128 and measured 1.9 % slower there).  Each SM
// sub-partition holds one warp of every warpgroup: kLow + 2 kMid + kHigh <= 512
// registers a lane, and the split fits the 512 * 128 registers the launch
// holds (launch_main refuses to launch if ptxas gave the kernel fewer than 128
// a thread).
template <int D>
struct BwdRegs {
  static constexpr uint32_t kLow = 96;
  static constexpr uint32_t kMid = 160;
  static constexpr uint32_t kHigh = 96;
  static constexpr uint32_t kLaunchRegs = 128;
  static_assert(kLow + 2 * kMid + kHigh <= 512, "register split exceeds an SM sub-partition");
  static_assert(128 * (kLow + 2 * kMid + kHigh) <= 512 * kLaunchRegs, "register split exceeds the launch");
};

// The key tile and (b, K/V head) of CTA x in the head-grouped order: heads in
// groups of head_group, and inside a group key tile major (under a causal mask
// the first key tiles have the most query tiles, so they start first).  The
// CTAs running at any moment then belong to a few heads, whose Q, dO and fp32
// dQ accumulator stay in L2, so the dQ reduce-adds are read-modify-writes in
// L2 rather than in DRAM.
__device__ __forceinline__ void bwd_cta_tile(int x, int nq, int head_group, int BH, int& bh,
                                             int& j) {
  const int grp = x / (head_group * nq);
  const int gsz = min(head_group, BH - grp * head_group);
  const int within = x - grp * head_group * nq;
  j = within / gsz;
  bh = grp * head_group + (within - j * gsz);
}

// The query tiles a key tile meets, in ascending order: a dense range
// [first, nq) or the set bits of the key tile's column of the block list
// (kept in shared memory).  Every role walks it identically.
struct QTiles {
  const uint32_t* bm;      // nullptr: dense range
  int first_dense, nq;
  __device__ __forceinline__ int first() const {
    if (bm == nullptr) return first_dense < nq ? first_dense : -1;
    return next(-1);
  }
  __device__ __forceinline__ int next(int i) const {
    if (bm == nullptr) return i + 1 < nq ? i + 1 : -1;
    int c = i + 1;
    while (c < nq) {
      const int w = c >> 5;
      const uint32_t bits = bm[w] & (0xFFFFFFFFu << (c & 31));
      if (bits) return (w << 5) + __ffs(bits) - 1;
      c = (w + 1) << 5;
    }
    return -1;
  }
};

// The (query head of the group, query tile) pairs a KV-head key tile meets:
// the query tiles of every query head that reads this KV head, head by head.
struct QWalk {
  QTiles qs;
  int G;                   // query heads per KV head
  __device__ __forceinline__ void start(int& g, int& i) const {
    g = 0;
    i = qs.first();
  }
  // the pair after (g, i); i < 0 at the end
  __device__ __forceinline__ void advance(int& g, int& i) const {
    i = qs.next(i);
    if (i < 0 && ++g < G) i = qs.first();
  }
};

template <int D, bool CAUSAL, bool SPARSE>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  {
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if (pad > static_cast<uint32_t>(C::kSlack)) {     // layout would not fit: report, touch nothing
      if (threadIdx.x == 0) record_error(p.err, ATTN_ERR_UNSUPPORTED);
      return;
    }
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
  float* stats = reinterpret_cast<float*>(smem + C::kStatOff);

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int tid = static_cast<int>(threadIdx.x);
  const bool tr = BSS_TRACE_ON(p, blockIdx.x);
  BSS_TRACE_EV(p, tr && tid == 0, 5, 0);             // kernel entry
  (void)tr;
  if (*reinterpret_cast<volatile int*>(p.err) == ATTN_ERR_TIMEOUT) return;

  // CTA order (bwd_cta_tile): heads in groups of p.head_group, key tile major
  // inside a group.  A block-sparse launch may instead read its order from
  // p.cta_order, which starts the few key tiles with far more query tiles
  // than the rest first and keeps the head-grouped order for the others.
  const int L = p.L;
  const int nq = (L + kTileM - 1) / kTileM;
  // heads here are K/V heads: the CTA owns a key tile of one (b, K/V head)
  // and meets the query tiles of the G query heads that read it
  const int BH = p.B * p.Hkv;
  const int G = p.H / p.Hkv;
  int j, bh;                                      // key tile owned by this CTA; (b, K/V head)
  if (SPARSE && p.cta_order != nullptr) {
    const int lin = __ldg(p.cta_order + blockIdx.x);
    bh = lin / nq;
    j = lin - bh * nq;
  } else {
    bwd_cta_tile(static_cast<int>(blockIdx.x), nq, p.head_group, BH, bh, j);
  }
  const int b = bh / p.Hkv;
  const int h = bh - b * p.Hkv;                   // K/V head
  const int hq0 = h * G;                          // first query head of the group
  const int bhq0 = b * p.H + hq0;
  // Query tiles met by this key tile: under a causal mask none before j.  A
  // block-sparse launch takes them from the key tile's column of the block
  // list (built with the causal cut already applied).
  uint32_t* col_bm = reinterpret_cast<uint32_t*>(smem + C::kColBmOff);
  QTiles qs;
  qs.bm = SPARSE ? col_bm : nullptr;
  qs.first_dense = CAUSAL ? j : 0;
  qs.nq = nq;
  int n_it = SPARSE ? 0 : nq - qs.first_dense;   // query tiles per query head
  if (SPARSE) {
    const int words = (nq + 31) / 32;
    for (int w = tid; w < words; w += C::kThreads)
      col_bm[w] = __ldg(p.col_bitmap +
                        (static_cast<size_t>(bhq0 / p.heads_per_list) * nq + j) * p.col_bitmap_words + w);
    __syncthreads();
    for (int w = 0; w < words; ++w) n_it += __popc(col_bm[w]);
  }
  n_it *= G;                                      // over all query heads of the group
  QWalk walk;
  walk.qs = qs;
  walk.G = G;

  if (tid == 0) {
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < C::kStagesQ; ++s) {
      mbar_init(bar(C::kBarQFull + s), 1);
      mbar_init(bar(C::kBarQEmpty + s), 1);
    }
    for (int s = 0; s < C::kStagesDO; ++s) {
      mbar_init(bar(C::kBarDOFull + s), 1);
      mbar_init(bar(C::kBarDOEmpty + s), 1);
    }
    mbar_init(bar(C::kBarSFull), 1);
    mbar_init(bar(C::kBarDPFull), 1);
    mbar_init(bar(C::kBarDPFull + 1), 1);
    mbar_init(bar(C::kBarPReady), 256);
    mbar_init(bar(C::kBarDSReady), 256);
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQFree), 128);
    mbar_init(bar(C::kBarDQFree + 1), 128);
    mbar_init(bar(C::kBarStaged), 128);
    mbar_init(bar(C::kBarStageFree), 1);
    mbar_init(bar(C::kBarDKVFull), 1);
    mbar_init(bar(C::kBarMmaDone), 1);
    mbar_init(bar(C::kBarStat + 0), 128);
    mbar_init(bar(C::kBarStat + 1), 128);
    *abort_flag = 0;
    fence_barrier_init();
    // K_j and V_j go out at once: their load overlaps the rest of the set-up
    mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTileBytes);
    for (int c = 0; c < C::kChunks; ++c) {
      tma_load_4d(sbase + C::kKOff + c * C::kChunkBytes, &tmK, bar(C::kBarKV), c * 64, j * kTileN, h, b);
      tma_load_4d(sbase + C::kVOff + c * C::kChunkBytes, &tmV, bar(C::kBarKV), c * 64, j * kTileN, h, b);
    }
  }
  if (warp == 0) {
    tmem_alloc(sbase + C::kMiscOff, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  BSS_TRACE_EV(p, tr && tid == 0, 5, 1);             // set-up done

  if (warp < 4) {
  regs_set<BwdRegs<D>::kLow, BwdRegs<D>::kLaunchRegs>();
  if (warp == 0) {
    // =================== TMA producer ===================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      int nq_ld = 0, ndo_ld = 0;
      int g, i;
      walk.start(g, i);
      for (int it = 0; i >= 0; walk.advance(g, i), ++it) {
        const int row = i * kTileM;
        const int hq = hq0 + g;
        const int sq = it % C::kStagesQ;
        if (it >= C::kStagesQ &&
            !wait_bar(bar(C::kBarQEmpty + sq), ((it / C::kStagesQ) & 1) ^ 1, abort_flag, p.err))
          break;
        mbar_arrive_expect_tx(bar(C::kBarQFull + sq), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sbase + C::kQOff + sq * C::kTileBytes + c * C::kChunkBytes, &tmQ,
                      bar(C::kBarQFull + sq), c * 64, row, hq, b);
        ++nq_ld;
        const int sd = it % C::kStagesDO;
        if (it >= C::kStagesDO &&
            !wait_bar(bar(C::kBarDOEmpty + sd), ((it / C::kStagesDO) & 1) ^ 1, abort_flag, p.err))
          break;
        mbar_arrive_expect_tx(bar(C::kBarDOFull + sd), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sbase + C::kDOOff + sd * C::kTileBytes + c * C::kChunkBytes, &tmDO,
                      bar(C::kBarDOFull + sd), c * 64, row, hq, b);
        ++ndo_ld;
      }
      // Drain: every load issued has landed before the CTA may exit.
      drain_bar(bar(C::kBarKV), 0);
      for (int x = max(0, nq_ld - C::kStagesQ); x < nq_ld; ++x)
        drain_bar(bar(C::kBarQFull + x % C::kStagesQ), (x / C::kStagesQ) & 1);
      for (int x = max(0, ndo_ld - C::kStagesDO); x < ndo_ld; ++x)
        drain_bar(bar(C::kBarDOFull + x % C::kStagesDO), (x / C::kStagesDO) & 1);
    }
  } else if (warp == 1) {
    // =================== MMA issuer (one thread) ===================
    // Issue order per query tile i: dV(i), S^T(i+1), dQ(i), dK(i), dP^T(i+1).
    // Every overwrite of TMEM or shared memory is ordered behind the MMAs that
    // read the old contents by issue order (the tensor core executes one
    // thread's MMAs in order) or by the barrier it waits on:
    //   S^T(i+1) over P^T(i): after dV(i);  P^T(i+1) written after S^T(i+1)
    //   completes; dQ(i) over dP^T(i): after ds_ready(i) (dP^T read);
    //   dP^T(i+1) over dQ(i): after dq_free(i); dS(i+1) written after
    //   dP^T(i+1) completes, so after dQ(i) and dK(i) read dS(i).
    if (lane == 0) {
      constexpr uint32_t kIdescT = idesc_bf16_f32(kTileM, kTileN, false, false);  // S^T, dP^T
      constexpr uint32_t kIdescKV = idesc_bf16_f32(kTileM, D, false, true);       // dV, dK
      constexpr uint32_t kIdescQ = idesc_bf16_f32(kTileM, D, true, true);         // dQ
      const uint32_t ka = sbase + C::kKOff, va = sbase + C::kVOff, dsa = sbase + C::kDSOff;
      auto qaddr = [&](int it) { return sbase + C::kQOff + (it % C::kStagesQ) * C::kTileBytes; };
      auto doaddr = [&](int it) { return sbase + C::kDOOff + (it % C::kStagesDO) * C::kTileBytes; };
      // S^T(it) = K_j Q^T
      auto issue_s = [&](int it) -> bool {
        if (!wait_bar(bar(C::kBarQFull + it % C::kStagesQ), (it / C::kStagesQ) & 1, abort_flag, p.err))
          return false;
        tc_fence_after();
        const uint32_t qa = qaddr(it);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColST, sdesc_sw128(ka + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024),
                 kIdescT, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarSFull));
        return true;
      };
      // dP^T(it) = V_j dO^T, in two halves of 64 queries (N = 64) when dQ
      // shares dP^T's columns: half h overwrites dQ's d-columns [64h, 64h+64),
      // which round h of the drain frees, and feeds P/dS half X = h alone.
      constexpr uint32_t kIdescTHalf = idesc_bf16_f32(kTileM, kTileN / 2, false, false);
      auto issue_dp_half = [&](int it, int h) -> bool {
        if (h == 0) {
          if (!wait_bar(bar(C::kBarDOFull + it % C::kStagesDO), (it / C::kStagesDO) & 1, abort_flag,
                        p.err))
            return false;
        }
        tc_fence_after();
        const uint32_t doa = doaddr(it) + h * (kTileN / 2) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColDPT + h * (kTileN / 2), sdesc_sw128(va + off, 16, 1024),
                 sdesc_sw128(doa + off, 16, 1024), kIdescTHalf, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarDPFull + h));
        return true;
      };
      // Block-sparse launches issue dP^T as one N=128 group once both halves
      // of dQ's columns are free: an N=64 MMA costs the tensor pipe nearly as
      // much as an N=128 one (93 against 102 cycles in a probe), and with a CTA's query
      // tiles spread out the halves' earlier start does not pay for the extra
      // eight (0.868 -> 0.850 ms on the L'=16320 workload; the dense and
      // causal backward measured 2.8 % slower with it, 1 % slower when the
      // single group was taken only when both halves were already free).
      constexpr bool kDPHalves = C::kDQOverDP && !SPARSE;
      auto issue_dp = [&](int it) -> bool {
        if (kDPHalves) return issue_dp_half(it, 0) && issue_dp_half(it, 1);
        if (!wait_bar(bar(C::kBarDOFull + it % C::kStagesDO), (it / C::kStagesDO) & 1, abort_flag, p.err))
          return false;
        tc_fence_after();
        const uint32_t doa = doaddr(it);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColDPT, sdesc_sw128(va + off, 16, 1024), sdesc_sw128(doa + off, 16, 1024),
                 kIdescT, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarDPFull));
        mma_commit(bar(C::kBarDPFull + 1));
        return true;
      };
      bool ok = wait_bar(bar(C::kBarKV), 0, abort_flag, p.err);
      BSS_TRACE_EV(p, tr, 5, 2);                       // K and V landed
      if (ok && n_it > 0) ok = issue_s(0) && issue_dp(0);
      int g, i;
      walk.start(g, i);
      for (int it = 0; i >= 0 && ok; walk.advance(g, i), ++it) {
        const bool more = it + 1 < n_it;               // another query tile follows
        // dV += P^T dO_i  (K dimension = the 128 queries)
        if (!wait_bar(bar(C::kBarPReady), it & 1, abort_flag, p.err)) break;
        BSS_TRACE_EV(p, tr, 1, 4 * it);
        tc_fence_after();
        const uint32_t doa = doaddr(it);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {
          mma_ts(tmem + C::kColDV, tmem + C::kColST + C::pcol(kk),
                 sdesc_sw128(doa + kk * 2048, C::kChunkBytes, 1024), kIdescKV,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(C::kBarDOEmpty + it % C::kStagesDO));   // dP^T(it) and dV(it) read dO_i
        if (more && !issue_s(it + 1)) break;
        // the P/dS warps run for a while: poll gently so that the issue slots
        // they share with this warp stay theirs
        if (!wait_bar_relaxed(bar(C::kBarDSReady), it & 1, abort_flag, p.err)) break;
        BSS_TRACE_EV(p, tr, 1, 4 * it + 1);
        tc_fence_after();
        // dQ_i = dS K_j  (M = queries, N = d, K dimension = the 128 keys); with
        // columns of its own, only after the previous dQ has been read
        if (!C::kDQOverDP && it > 0 && !wait_bar(bar(C::kBarDQFree), (it - 1) & 1, abort_flag, p.err))
          break;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          mma_ss(tmem + C::kColDQ, sdesc_sw128(dsa + kk * 2048, C::kChunkBytes, 1024),
                 sdesc_sw128(ka + kk * 2048, C::kChunkBytes, 1024), kIdescQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarDQFull));
        // dK += dS^T Q_i  (dS^T: the same tile read K-major; K dimension = queries)
        const uint32_t qa = qaddr(it);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColDK, sdesc_sw128(dsa + off, 16, 1024),
                 sdesc_sw128(qa + kk * 2048, C::kChunkBytes, 1024), kIdescKV,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(C::kBarQEmpty + it % C::kStagesQ));
        BSS_TRACE_EV(p, tr, 1, 4 * it + 2);
        if (more) {
          if (kDPHalves) {
            // dP^T(i+1) over dQ(i): each half once its columns have been read out
            if (!wait_bar(bar(C::kBarDQFree), it & 1, abort_flag, p.err)) break;
            if (!issue_dp_half(it + 1, 0)) break;
            if (!wait_bar(bar(C::kBarDQFree + 1), it & 1, abort_flag, p.err)) break;
            BSS_TRACE_EV(p, tr, 1, 4 * it + 3);
            if (!issue_dp_half(it + 1, 1)) break;
          } else if (C::kDQOverDP) {
            // one N=128 group once both halves of dQ's columns are read out
            if (!wait_bar(bar(C::kBarDQFree), it & 1, abort_flag, p.err)) break;
            if (!wait_bar(bar(C::kBarDQFree + 1), it & 1, abort_flag, p.err)) break;
            BSS_TRACE_EV(p, tr, 1, 4 * it + 3);
            if (!issue_dp(it + 1)) break;
          } else {
            BSS_TRACE_EV(p, tr, 1, 4 * it + 3);
            if (!issue_dp(it + 1)) break;
          }
        }
      }
      mma_commit(bar(C::kBarDKVFull));
      mma_commit(bar(C::kBarMmaDone));
      drain_bar(bar(C::kBarMmaDone), 0);   // every MMA issued has completed
    }
  }
#ifdef BSS_TRACE
  else if (warp == 2 && lane == 0 && tr) {
    // trace builds: watch the MMA groups complete (passive waits on the
    // barriers their commits arrive at) for the pipeline trace
    for (int it = 0; it < n_it && it < kTraceEvents / 8; ++it) {
      const bool more = it + 1 < n_it;
      if (!drain_bar(bar(C::kBarDOEmpty + it % C::kStagesDO), (it / C::kStagesDO) & 1, 1ll << 28)) break;
      BSS_TRACE_EV(p, true, 4, 8 * it + 0);          // dV(it) done
      if (more) {
        if (!drain_bar(bar(C::kBarSFull), (it + 1) & 1, 1ll << 28)) break;
        BSS_TRACE_EV(p, true, 4, 8 * it + 1);        // S^T(it+1) done
      }
      if (!drain_bar(bar(C::kBarDQFull), it & 1, 1ll << 28)) break;
      BSS_TRACE_EV(p, true, 4, 8 * it + 2);          // dQ(it) done
      if (!drain_bar(bar(C::kBarQEmpty + it % C::kStagesQ), (it / C::kStagesQ) & 1, 1ll << 28)) break;
      BSS_TRACE_EV(p, true, 4, 8 * it + 3);          // dK(it) done
      if (more) {
        if (!drain_bar(bar(C::kBarDPFull), (it + 1) & 1, 1ll << 28)) break;
        BSS_TRACE_EV(p, true, 4, 8 * it + 4);        // dP^T(it+1) half 0 done
        if (!drain_bar(bar(C::kBarDPFull + 1), (it + 1) & 1, 1ll << 28)) break;
        BSS_TRACE_EV(p, true, 4, 8 * it + 5);        // dP^T(it+1) half 1 done
      }
    }
  }
#endif
  } else if (warp < 12) {
    regs_set<BwdRegs<D>::kMid, BwdRegs<D>::kLaunchRegs>();
    // =================== P^T / dS: two warpgroups, thread = key row ===================
    // Warpgroup X (warps 4-7: X = 0, warps 8-11: X = 1) handles query columns
    // [64X, 64X + 64), 16 at a time.  Phase 1 turns S^T into P (kept in fp32
    // registers) and writes P^T (bf16) to columns [64X + 8c, 64X + 8c + 8) of
    // chunk c, which this half has already read; phase 2 forms dS from P and
    // dP^T and stores it in shared memory.
    const int X = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int kr = wq * 32 + lane;
    const int key = j * kTileN + kr;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tST = tmem + lane_base + C::kColST;
    const uint32_t tDPT = tmem + lane_base + C::kColDPT;
    const float sl2 = p.scale_log2;
    const float scale = p.scale;
    const float INF = __int_as_float(0x7f800000);
    uint8_t* ds_row = smem + C::kDSOff + X * C::kChunkBytes + kr * 128;   // this key's dS row
    // statistics of query tile i of query head hq0 + g, negated so that
    // P = ex2(S sl2 + nl2) and dP - D = dP scale + ndl are single FMAs
    auto load_stats = [&](int g, int i, float& nl2, float& ndl) {
      const int q = i * kTileM + kr;
      if (i >= 0 && i < nq && q < L) {
        const size_t stat_base = static_cast<size_t>(bhq0 + g) * L;
        const float lse = __ldg(p.lse + stat_base + q);
        nl2 = (lse == -INF) ? -INF : -(lse * kLog2e);  // an empty row contributes nothing
        ndl = -(__ldg(p.delta + stat_base + q) * scale);
      } else {
        nl2 = -INF;
        ndl = 0.f;
      }
    };
    if (X == 0) {
      float l2, dl;
      load_stats(0, qs.first(), l2, dl);
      stats[kr] = l2;
      stats[128 + kr] = dl;
      mbar_arrive(bar(C::kBarStat + 0));
    }
    // Buffer (it & 1) holds the statistics of the it-th query tile met (minus
    // the LSE in log2 units, minus scale * D).  It is rewritten (for tile it + 2) at the end of tile
    // it + 1 by half 0; by then dP^T(it + 1) has been issued, which waited for
    // dS(it) of both halves, so nobody reads it for tile it any more.
    bool ok = true;
    int g, i;
    walk.start(g, i);
    for (int it = 0; i >= 0; walk.advance(g, i), ++it) {
      const float* lse2 = stats + (it & 1) * 256 + 64 * X;
      const float* dlt = lse2 + 128;
      float l2n = 0.f, dln = 0.f;
      if (X == 0) {
        int gn = g, in = i;
        walk.advance(gn, in);
        load_stats(gn, in, l2n, dln);
      }
      if (!wait_bar(bar(C::kBarSFull), it & 1, abort_flag, p.err) ||
          !wait_bar(bar(C::kBarStat + (it & 1)), (it >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      const bool trw = tr && kr == 0 && X == 0;
      (void)trw;
      BSS_TRACE_EV(p, trw, 2, 4 * it);
      tc_fence_after();
      const bool key_ok = key < L;
      // element mask: diagonal tile (query < key) and keys past L; the ragged
      // tail (query >= L) has -lse2 = -inf, so P is 0 there already
      const bool diag = CAUSAL && (i == j);
      const bool need_mask = !key_ok || diag;
      // ---- phase 1: P (four chunks of 16 queries; chunk c+1's TMEM load is in
      // flight while chunk c is computed) ----
      float pf[4][16];
      {
        uint32_t sv[2][16];
        tmem_ld16(tST + 64 * X, sv[0]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int cur = c & 1;
          const int col = 64 * X + 16 * c;                 // first query of the chunk
          tmem_ld_wait16(sv[cur]);
          if (c + 1 < 4) tmem_ld16(tST + col + 16, sv[cur ^ 1]);
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse2 + 16 * c + e);
            float x[4];
            ffma2(x[0], x[1], __uint_as_float(sv[cur][e]), __uint_as_float(sv[cur][e + 1]), sl2,
                  sl2, l4.x, l4.y);
            ffma2(x[2], x[3], __uint_as_float(sv[cur][e + 2]), __uint_as_float(sv[cur][e + 3]),
                  sl2, sl2, l4.z, l4.w);
#pragma unroll
            for (int u = 0; u < 4; ++u) pf[c][e + u] = ex2(x[u]);
          }
          if (need_mask) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (!key_ok || col + e < kr) pf[c][e] = 0.f;
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = pack_bf16(pf[c][2 * e], pf[c][2 * e + 1]);
          tmem_st8(tST + 64 * X + 8 * c, pk);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPReady));
      BSS_TRACE_EV(p, trw, 2, 4 * it + 1);
      // ---- phase 2: dS = P o (dP - D), into shared memory ----
      if (!wait_bar(bar(C::kBarDPFull + X), it & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      BSS_TRACE_EV(p, trw, 2, 4 * it + 2);
      tc_fence_after();
      {
        uint32_t dv[2][16];
        tmem_ld16(tDPT + 64 * X, dv[0]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int cur = c & 1;
          const int col = 64 * X + 16 * c;
          tmem_ld_wait16(dv[cur]);
          if (c + 1 < 4) tmem_ld16(tDPT + col + 16, dv[cur ^ 1]);
          uint32_t dk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(dlt + 16 * c + e);
            float ds[4];
            ffma2(ds[0], ds[1], __uint_as_float(dv[cur][e]), __uint_as_float(dv[cur][e + 1]), scale,
                  scale, d4.x, d4.y);
            ffma2(ds[2], ds[3], __uint_as_float(dv[cur][e + 2]), __uint_as_float(dv[cur][e + 3]),
                  scale, scale, d4.z, d4.w);
            fmul2(ds[0], ds[1], pf[c][e], pf[c][e + 1], ds[0], ds[1]);
            fmul2(ds[2], ds[3], pf[c][e + 2], pf[c][e + 3], ds[2], ds[3]);
            dk[e / 2] = pack_bf16(ds[0], ds[1]);
            dk[e / 2 + 1] = pack_bf16(ds[2], ds[3]);
          }
          // one 128-byte row per key (queries 64X .. 64X+63), 16-byte units of
          // 8 queries swizzled by the row index: the K-major tile layout
#pragma unroll
          for (int u2 = 0; u2 < 2; ++u2) {
            const int unit = 2 * c + u2;
            *reinterpret_cast<uint4*>(ds_row + ((unit ^ (kr & 7)) * 16)) =
                make_uint4(dk[4 * u2 + 0], dk[4 * u2 + 1], dk[4 * u2 + 2], dk[4 * u2 + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::kBarDSReady));
      BSS_TRACE_EV(p, trw, 2, 4 * it + 3);
      if (X == 0) {
        // statistics of the next query tile
        float* nxt = stats + ((it + 1) & 1) * 256;
        nxt[kr] = l2n;
        nxt[128 + kr] = dln;
        mbar_arrive(bar(C::kBarStat + ((it + 1) & 1)));
      }
    }
    // ---- epilogue: half 0 stores dK rows, half 1 stores dV rows ----
    if (ok) ok = wait_bar(bar(C::kBarDKVFull), 0, abort_flag, p.err);
    BSS_TRACE_EV(p, tr && kr == 0 && X == 0, 5, 3);   // dK and dV complete
    tc_fence_after();
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (ok) {
      // one 128-byte line (64 columns as bf16 pairs) of this thread's key row
      // at a time; after the octet transpose every store writes whole lines
      const uint32_t tsrc = tmem + lane_base + (X == 0 ? C::kColDK : C::kColDV);
      const int wrow0 = j * kTileN + wq * 32;          // this warp's first key row
      const uint32_t valid = __ballot_sync(0xFFFFFFFFu, key < L);
      uint8_t* base = reinterpret_cast<uint8_t*>((X == 0 ? p.dk : p.dv) +
                                                 (static_cast<size_t>(bh) * L + wrow0) * D);
#pragma unroll 1
      for (int g2 = 0; g2 < D / 64; ++g2) {
        uint32_t a[32], c[32];
        if (n_it > 0) {
          tmem_ld32(tsrc + g2 * 64, a);
          tmem_ld32(tsrc + g2 * 64 + 32, c);
          tmem_ld_wait(a);
          tmem_ld_wait(c);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = c[e] = 0u;
        }
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          w[k] = pack_bf16(__uint_as_float(a[2 * k]), __uint_as_float(a[2 * k + 1]));
          w[16 + k] = pack_bf16(__uint_as_float(c[2 * k]), __uint_as_float(c[2 * k + 1]));
        }
        transpose_octets(w, lane);
        store_octet_lines(w, base + g2 * 128, D * 2, valid, lane);
      }
    }
  } else {
    regs_set<BwdRegs<D>::kHigh, BwdRegs<D>::kLaunchRegs>();
    // =================== dQ: warps 12-15, thread = query row ===================
    // Each round moves 64 d-columns of the tile's dQ from TMEM to a
    // 128-byte-swizzled fp32 staging buffer, from which bulk tensor
    // reduce-adds (boxes of 32 columns) add it into the fp32 accumulator in
    // global memory; dQ's TMEM columns of a round are handed back right after
    // their reads.  Per-warp drain (d=128): each warp reduces its own 32 rows
    // and reuses its staging rows once its own previous reduces have read them
    // (bulk groups are per thread).  CTA-wide drain (d=64): one thread reduces
    // the 128 rows after all four warps have staged them.  (On the bench
    // shapes, vector red.global from registers, for all of dQ or for one
    // round, measured slower: the reduce stream sets the pace.)
    constexpr bool kPerWarp = C::kDrainPerWarp;
    const int wq = warp & 3;
    const int qr = wq * 32 + lane;
    const uint32_t tDQ = tmem + (static_cast<uint32_t>(wq * 32) << 16) + C::kColDQ;
    constexpr int kRounds = D / 64;
    constexpr int kBoxBytes = kTileM * 32 * 4;    // 128 rows x 32 fp32: one box column
    static_assert(2 * kBoxBytes == C::kStageBytes, "two box columns fill the staging buffer");
    const uint32_t stage = sbase + C::kStageOff + (kPerWarp ? wq * 32 * 128 : 0);
    uint8_t* stage_ptr = smem + C::kStageOff;
    bool ok = true;
    int g = 0;                                    // staged rounds (CTA-wide drain)
    int gq, i;                                    // query head of the group, query tile
    walk.start(gq, i);
    for (int it = 0; i >= 0 && ok; walk.advance(gq, i), ++it) {
      if (!wait_bar_relaxed(bar(C::kBarDQFull), it & 1, abort_flag, p.err)) break;
      BSS_TRACE_EV(p, tr && qr == 0, 3, 3 * it);
      tc_fence_after();
      for (int r = 0; r < kRounds; ++r, ++g) {
        uint32_t v0[32], v1[32];
        tmem_ld32(tDQ + 64 * r, v0);
        tmem_ld32(tDQ + 64 * r + 32, v1);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
        // d-columns [64r, 64r + 64) of this tile are read (at d=128 dP^T's
        // half r may overwrite them; at d=64 the next dQ may)
        tc_fence_before();
        mbar_arrive(bar(C::kBarDQFree + r));
        if (r == kRounds - 1) BSS_TRACE_EV(p, tr && qr == 0, 3, 3 * it + 1);
        // the staging rows must have been read by the reduces that used them
        if constexpr (kPerWarp) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        } else if (g > 0) {
          if (qr == 0) {
            bulk_wait_read_all();
            mbar_arrive(bar(C::kBarStageFree));
          }
          if (!wait_bar(bar(C::kBarStageFree), (g - 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {               // box column 0: columns 0..31 of the round
          *reinterpret_cast<uint4*>(stage_ptr + qr * 128 + ((u ^ (qr & 7)) * 16)) =
              make_uint4(v0[4 * u], v0[4 * u + 1], v0[4 * u + 2], v0[4 * u + 3]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {               // box column 1: columns 32..63
          *reinterpret_cast<uint4*>(stage_ptr + kBoxBytes + qr * 128 + ((u ^ (qr & 7)) * 16)) =
              make_uint4(v1[4 * u], v1[4 * u + 1], v1[4 * u + 2], v1[4 * u + 3]);
        }
        fence_proxy_async_smem();
        if constexpr (kPerWarp) {
          __syncwarp();
          if (lane == 0) {
            const int row = i * kTileM + wq * 32;
            tma_reduce_add_4d(&tmDQ, stage, 64 * r, row, hq0 + gq, b);
            tma_reduce_add_4d(&tmDQ, stage + kBoxBytes, 64 * r + 32, row, hq0 + gq, b);
            bulk_commit_group();
          }
        } else {
          mbar_arrive(bar(C::kBarStaged));
          if (qr == 0) {
            if (!wait_bar(bar(C::kBarStaged), g & 1, abort_flag, p.err)) {
              ok = false;
              break;
            }
            const int row = i * kTileM;
            tma_reduce_add_4d(&tmDQ, stage, 64 * r, row, hq0 + gq, b);
            tma_reduce_add_4d(&tmDQ, stage + kBoxBytes, 64 * r + 32, row, hq0 + gq, b);
            bulk_commit_group();
          }
        }
        __syncwarp();                               // reconverge before the next TMEM load
      }
      BSS_TRACE_EV(p, tr && qr == 0, 3, 3 * it + 2);
    }
    if (kPerWarp ? lane == 0 : qr == 0) bulk_wait_all();   // every reduction has landed
  }

  tc_fence_before();
  __syncthreads();
  BSS_TRACE_EV(p, tr && tid == 0, 5, 4);             // every role done
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// D_i = dO_i . O_i for every row, and the fp32 dQ accumulator cleared.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(const BwdParams p) {
  constexpr int G = D / 8;                           // threads per row, 16 bytes each
  const long long rows = static_cast<long long>(p.B) * p.H * p.L;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  const int g = static_cast<int>(threadIdx.x % G);
  for (long long r = tid / G;; r += nthreads / G) {
    const bool active = r < rows;
    if (__all_sync(0xFFFFFFFFu, !active)) break;     // every lane of the warp is done
    uint4 o = make_uint4(0u, 0u, 0u, 0u), d = o;
    if (active) {
      o = __ldg(reinterpret_cast<const uint4*>(p.o + r * D) + g);
      d = __ldg(reinterpret_cast<const uint4*>(p.dout + r * D) + g);
    }
    float s = bf16lo(o.x) * bf16lo(d.x) + bf16hi(o.x) * bf16hi(d.x);
    s = fmaf(bf16lo(o.y), bf16lo(d.y), s);
    s = fmaf(bf16hi(o.y), bf16hi(d.y), s);
    s = fmaf(bf16lo(o.z), bf16lo(d.z), s);
    s = fmaf(bf16hi(o.z), bf16hi(d.z), s);
    s = fmaf(bf16lo(o.w), bf16lo(d.w), s);
    s = fmaf(bf16hi(o.w), bf16hi(d.w), s);
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off, G);
    if (active && g == 0) p.delta[r] = s;
  }
  float4* acc = reinterpret_cast<float4*>(p.dq_acc);
  const long long n4 = rows * D / 4;
  for (long long x = tid; x < n4; x += nthreads) acc[x] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ (bf16) from the fp32 accumulator; the scale was applied to dS already.
__global__ void __launch_bounds__(256) attn_bwd_dq_convert_kernel(const float* acc, __nv_bfloat16* dq,
                                                                  long long n8) {
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long x = tid; x < n8; x += nthreads) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc) + 2 * x);
    const float4 b = __ldg(reinterpret_cast<const float4*>(acc) + 2 * x + 1);
    uint4 w;
    w.x = pack_bf16(a.x, a.y);
    w.y = pack_bf16(a.z, a.w);
    w.z = pack_bf16(b.x, b.y);
    w.w = pack_bf16(b.z, b.w);
    reinterpret_cast<uint4*>(dq)[x] = w;
  }
}

template <int D, bool CAUSAL, bool SPARSE>
cudaError_t launch_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                        cudaStream_t st) {
  using C = BwdCfg<D>;
  auto kern = attn_bwd_main_kernel<D, CAUSAL, SPARSE>;
  constexpr int kMaxDev = 64;
  static bool configured[kMaxDev] = {};  // the attribute is per device and function
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    if (fa.numRegs < static_cast<int>(BwdRegs<D>::kLaunchRegs)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int n_cta = p.B * p.Hkv * ((p.L + kTileN - 1) / kTileN);
  kern<<<n_cta, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, tdo, tdq, p);
  return cudaGetLastError();
}

unsigned grid_for(long long work, int per_block) {
  long long blocks = (work + per_block - 1) / per_block;
  const long long cap = 152LL * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

// Key-major bitmaps of the block lists: bit i of column c of list l is set
// when query block i of list l lists key block c.  Duplicates collapse, the
// order of a row is irrelevant, and under a causal mask a key block after the
// query block is left out (it holds no allowed pair).  One thread per (list,
// query block); malformed rows and entries are skipped and reported.
__global__ void __launch_bounds__(256) attn_blocklist_columns_kernel(
    const int* row_ptr, const int* col_idx, int n_lists, int n_qblk, int nnz, int causal,
    uint32_t* bm, int words, int* err) {
  const long long total = static_cast<long long>(n_lists) * n_qblk;
  for (long long x = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; x < total;
       x += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int list = static_cast<int>(x / n_qblk);
    const int i = static_cast<int>(x - static_cast<long long>(list) * n_qblk);
    const int* rp = row_ptr + static_cast<size_t>(list) * (n_qblk + 1);
    const int beg = __ldg(rp + i);
    const int end = __ldg(rp + i + 1);
    if (beg < 0 || end < beg || end > nnz) {
      record_error(err, ATTN_ERR_BAD_BLOCKLIST);
      continue;
    }
    uint32_t* lbm = bm + static_cast<size_t>(list) * n_qblk * words;
    for (int e = beg; e < end; ++e) {
      const int c = __ldg(col_idx + e);
      if (c < 0 || c >= n_qblk) {
        record_error(err, ATTN_ERR_BAD_BLOCKLIST);
        continue;
      }
      if (causal && c > i) continue;
      atomicOr(lbm + static_cast<size_t>(c) * words + (i >> 5), 1u << (i & 31));
    }
  }
}

// Launch order of the block-sparse backward's CTAs.  A key tile's CTA walks
// the query tiles that list it, one after another, so a column listed by far
// more query blocks than the others (a global block every row lists) runs
// many times longer than the rest; started late in the head-grouped order it
// would finish alone at the end.  Longest-first scheduling bounds that tail:
// the columns whose length exceeds 4 times the mean (and 8 query tiles) go
// first, in the head-grouped order, then all the others in that same order,
// which keeps their heads' Q, dO and dQ accumulator together in L2.  One CTA
// partitions the n_cta entries stably with block-wide prefix sums.
constexpr int kOrderThreads = 1024;

__device__ __forceinline__ int bwd_column_len(const uint32_t* bm, int words, int nq, int H, int G,
                                              int Hkv, int heads_per_list, int bh, int j) {
  const int b = bh / Hkv;
  const int h = bh - b * Hkv;
  const size_t list = static_cast<size_t>(b * H + h * G) / heads_per_list;
  const uint32_t* col = bm + (list * nq + j) * words;
  int n = 0;
  for (int w = 0; w < words; ++w) n += __popc(__ldg(col + w));
  return n;
}

// Exclusive prefix sum of one int per thread over the block; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < kOrderThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;                      // inclusive sums of the warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[kOrderThreads / 32 - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kOrderThreads) attn_bwd_cta_order_kernel(
    const uint32_t* bm, int words, int nq, int B, int H, int Hkv, int heads_per_list,
    int head_group, int* order) {
  __shared__ int warp_sums[32];
  const int G = H / Hkv;
  const int BH = B * Hkv;
  const int n_cta = BH * nq;
  // pass 1: total query tiles over all CTAs
  long long total = 0;
  for (int x0 = 0; x0 < n_cta; x0 += kOrderThreads) {
    const int x = x0 + static_cast<int>(threadIdx.x);
    int len = 0;
    if (x < n_cta) {
      int bh, j;
      bwd_cta_tile(x, nq, head_group, BH, bh, j);
      len = bwd_column_len(bm, words, nq, H, G, Hkv, heads_per_list, bh, j);
    }
    int t;
    block_exclusive_scan(len, warp_sums, &t);
    total += t;
  }
  // pass 2: the long columns, then the others, each in the head-grouped order
  int n_long = 0;
  for (int pass = 0; pass < 2; ++pass) {
    int base = pass == 0 ? 0 : n_long;
    for (int x0 = 0; x0 < n_cta; x0 += kOrderThreads) {
      const int x = x0 + static_cast<int>(threadIdx.x);
      int bh = 0, j = 0, sel = 0;
      if (x < n_cta) {
        bwd_cta_tile(x, nq, head_group, BH, bh, j);
        const int len = bwd_column_len(bm, words, nq, H, G, Hkv, heads_per_list, bh, j);
        const bool is_long = len >= 8 && static_cast<long long>(len) * n_cta > 4 * total;
        sel = (pass == 0) == is_long ? 1 : 0;
      }
      int cnt;
      const int pos = block_exclusive_scan(sel, warp_sums, &cnt);
      if (sel) order[base + pos] = bh * nq + j;
      base += cnt;
    }
    if (pass == 0) n_long = base;
  }
}

}  // namespace

cudaError_t launch_bwd_cta_order(const uint32_t* bitmap, int words, int nq, int B, int H, int Hkv,
                                 int heads_per_list, int head_group, int* order, cudaStream_t st) {
  attn_bwd_cta_order_kernel<<<1, kOrderThreads, 0, st>>>(bitmap, words, nq, B, H, Hkv,
                                                         heads_per_list, head_group, order);
  return cudaGetLastError();
}

int bwd_dq_box_rows(int d) {
  return d == 128 ? BwdCfg<128>::kDrainBoxRows : BwdCfg<64>::kDrainBoxRows;
}

cudaError_t launch_blocklist_columns(const int* row_ptr, const int* col_idx, int n_lists, int n_qblk,
                                     int nnz, int causal, uint32_t* bitmap, int words, int* err,
                                     cudaStream_t st) {
  const size_t bytes = static_cast<size_t>(n_lists) * n_qblk * words * 4;
  cudaError_t e = cudaMemsetAsync(bitmap, 0, bytes, st);
  if (e != cudaSuccess) return e;
  attn_blocklist_columns_kernel<<<grid_for(static_cast<long long>(n_lists) * n_qblk, 256), 256, 0, st>>>(
      row_ptr, col_idx, n_lists, n_qblk, nnz, causal, bitmap, words, err);
  return cudaGetLastError();
}

cudaError_t launch_bwd(int d, bool sparse, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                       const BwdParams& p, cudaStream_t st, cudaEvent_t main_begin,
                       cudaEvent_t main_end) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.L;
  cudaError_t e;
  if (d == 64) {
    attn_bwd_preprocess_kernel<64><<<grid_for(rows * 8, 256), 256, 0, st>>>(p);
  } else if (d == 128) {
    attn_bwd_preprocess_kernel<128><<<grid_for(rows * 16, 256), 256, 0, st>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // optional timing of the main kernel alone (attn_bwd_time_main)
  if (main_begin && (e = cudaEventRecord(main_begin, st)) != cudaSuccess) return e;
#define BSS_BWD_CASE(DD, CA, SP)                                  \
  if (d == DD && (p.causal != 0) == CA && sparse == SP)           \
    e = launch_main<DD, CA, SP>(tq, tk, tv, tdo, tdq, p, st);
  e = cudaErrorInvalidValue;
  BSS_BWD_CASE(64, false, false)
  BSS_BWD_CASE(64, true, false)
  BSS_BWD_CASE(128, false, false)
  BSS_BWD_CASE(128, true, false)
  BSS_BWD_CASE(64, false, true)
  BSS_BWD_CASE(64, true, true)
  BSS_BWD_CASE(128, false, true)
  BSS_BWD_CASE(128, true, true)
#undef BSS_BWD_CASE
  if (e != cudaSuccess) return e;
  if (main_end && (e = cudaEventRecord(main_end, st)) != cudaSuccess) return e;
  const long long n8 = rows * d / 8;
  attn_bwd_dq_convert_kernel<<<grid_for(n8, 256), 256, 0, st>>>(p.dq_acc, p.dq, n8);
  return cudaGetLastError();
}

}  // namespace bss
