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
//   * one CTA owns TWO consecutive 128-row query tiles of one (b, h) that share
//     a single K/V stream: each K/V tile is loaded once for 256 query rows;
//   * warp 0 issues TMA loads (128-byte swizzled boxes of 128 rows x 64 d) into
//     a ring of K and V stages; warp 1 (one thread) issues every tcgen05.mma;
//     warpgroups 1 and 2 (warps 4-7, 8-11) run the online softmax of tile 0
//     and tile 1, one thread per query row (TMEM lane = row), with a larger
//     register budget handed over from warpgroup 0 (setmaxnreg);
//   * TMEM (512 columns): S0 | S1 | O0 | O1.  S = Q K^T is written by an SS
//     MMA; the softmax warpgroup reads its row, writes P (bf16) back into the
//     upper half of the same S columns, and P V accumulates into O by a TS MMA
//     with P as the tensor-memory A operand;
//   * the two tiles alternate on the tensor core (P V of tile 0, S of tile 0's
//     next block, P V of tile 1, S of tile 1's next block), so one warpgroup's
//     exponentials overlap the other tile's MMAs;
//   * exponentials are base 2 with scale*log2(e) folded in; the running max is
//     only moved (and O rescaled in TMEM) when it grows by more than 2^8, which
//     keeps the result exact because l and A always share the same reference m;
//   * causal: blocks wholly in the future are never visited, the element mask
//     is applied only where a block crosses the diagonal or the sequence end;
//   * block-sparse: each CTA turns its two CSR rows into bitmaps in shared
//     memory (duplicates collapse, order is irrelevant) and visits the union,
//     each tile computing only the blocks of its own list.
#include "common.cuh"

namespace bss {
namespace {

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;                   // 128-byte swizzle atoms across d
  static constexpr int kChunkBytes = kTileM * 128;         // 128 rows x 128 bytes
  static constexpr int kTileBytes = kTileM * D * 2;
  static constexpr int kStagesK = (D == 128) ? 2 : 4;
  static constexpr int kStagesV = (D == 128) ? 3 : 4;   // V is consumed last: deeper prefetch
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStagesK * kTileBytes;
  static constexpr int kBarOff = kVOff + kStagesV * kTileBytes;
  // q_full[2] k_full[SK] k_empty[SK] v_full[SV] v_empty[SV] s_full[2] p_full[2] o_full[2] mma_done
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKFull = 2;
  static constexpr int kBarKEmpty = kBarKFull + kStagesK;
  static constexpr int kBarVFull = kBarKEmpty + kStagesK;
  static constexpr int kBarVEmpty = kBarVFull + kStagesV;
  static constexpr int kBarSFull = kBarVEmpty + kStagesV;
  static constexpr int kBarPFull = kBarSFull + 2;
  static constexpr int kBarOFull = kBarPFull + 2;
  static constexpr int kBarMmaDone = kBarOFull + 2;
  static constexpr int kNumBars = kBarMmaDone + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBitmapWords = kMaxKBlocks / 32;
  static constexpr int kBitmapOff = kMiscOff + 16;
  static constexpr int kSmemBytes = kBitmapOff + 2 * kBitmapWords * 4 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;                      // S_t at t*128
  static constexpr uint32_t kColP = 64;                     // P_t at S_t + 64 (bf16 pairs)
  static constexpr uint32_t kColO = 256;                    // O_t at 256 + t*D
  static constexpr int kThreads = 384;
  // Register split per warpgroup (setmaxnreg): warpgroup 0 (TMA, MMA, two idle
  // warps) keeps kRegsLow, the two softmax warpgroups get kRegsHigh.  Each SM
  // sub-partition holds one warp of every warpgroup: 88 + 2 * 200 = 488 <= 512
  // registers per lane there, and the whole split 128*88 + 256*200 = 62464 fits
  // the 384 * R registers the launch holds for any ptxas assignment R >= 163
  // (the build asserts R = 168).
  static constexpr uint32_t kRegsLow = 88;
  static constexpr uint32_t kRegsHigh = 200;
};

// The ordered list of key blocks this CTA visits and which of its two tiles
// takes part in each.  Every role walks it identically.
struct Schedule {
  int kbmax0, kbmax1;          // last block a tile can see (-1: none)
  const uint32_t* bm0;         // block-sparse bitmaps (nullptr: dense prefix)
  const uint32_t* bm1;

  __device__ __forceinline__ int member(int kb) const {
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
};

template <int D, bool CAUSAL, bool SPARSE, bool PARTIAL>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + C::kBarOff;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + C::kBitmapOff);

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  const int tid = static_cast<int>(threadIdx.x);
  const bool tr = BSS_TRACE_ON(p, blockIdx.y * gridDim.x + blockIdx.x);
  (void)tr;
  // A launch whose earlier CTAs already timed out stops at once instead of
  // timing out CTA by CTA.
  if (*reinterpret_cast<volatile int*>(p.err) == ATTN_ERR_TIMEOUT) return;

  const int bh = blockIdx.x;
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int pair = CAUSAL ? (p.n_pairs - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
  const int r0_0 = pair * 2 * kTileM;
  const int r0[2] = {r0_0, r0_0 + kTileM};
  const int nk = (p.Lk + kTileN - 1) / kTileN;

  // Last key block each tile can see.
  int kbmax[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    if (r0[t] >= p.Lq) {
      kbmax[t] = -1;
    } else if (CAUSAL) {
      const long long r_last = min(r0[t] + kTileM - 1, p.Lq - 1);
      const long long lim = r_last + p.q_offset - p.k_offset;
      kbmax[t] = lim < 0 ? -1 : static_cast<int>(lim / kTileN < nk - 1 ? lim / kTileN : nk - 1);
    } else {
      kbmax[t] = nk - 1;
    }
  }

  // A dense-mode CTA whose rows see no key (all rows before a chunk's first
  // key, or past the end) writes the empty state of its rows and leaves
  // without setting anything up.
  if (!SPARSE && kbmax[0] < 0 && kbmax[1] < 0) {
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int nrows = max(0, min(2 * kTileM, p.Lq - r0[0]));
    const size_t row0 = static_cast<size_t>(bh) * p.Lq + r0[0];
    for (int r = tid; r < nrows; r += C::kThreads) {
      if (PARTIAL) {
        p.m_out[row0 + r] = NEG_INF;
        p.l_out[row0 + r] = 0.f;
      } else {
        p.lse[row0 + r] = NEG_INF;
      }
    }
    if (!PARTIAL) {
      uint4* o4 = reinterpret_cast<uint4*>(p.o + row0 * D);
      const int n16 = nrows * D / 8;
      for (int x = tid; x < n16; x += C::kThreads) o4[x] = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }

  // ---- set-up: barriers, tensor memory, block-sparse bitmaps -------------
  if (tid == 0) {
    mbar_init(bar(C::kBarQFull + 0), 1);
    mbar_init(bar(C::kBarQFull + 1), 1);
    for (int s = 0; s < C::kStagesK; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
    }
    for (int s = 0; s < C::kStagesV; ++s) {
      mbar_init(bar(C::kBarVFull + s), 1);
      mbar_init(bar(C::kBarVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kBarSFull + t), 1);
      mbar_init(bar(C::kBarPFull + t), 4 * 32);
      mbar_init(bar(C::kBarOFull + t), 1);
    }
    mbar_init(bar(C::kBarMmaDone), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + C::kMiscOff, C::kTmemCols);
    tmem_relinquish();
  }
  BSS_TRACE_EV(p, tr && tid == 0, 6, 0);
  if (SPARSE) {
    for (int i = tid; i < 2 * C::kBitmapWords; i += C::kThreads) bitmap[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int qb = r0[t] / kTileM;
      if (r0[t] >= p.Lq || qb >= p.n_qblk) continue;
      const int beg = __ldg(p.row_ptr + qb);
      const int end = __ldg(p.row_ptr + qb + 1);
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
        atomicOr(bitmap + t * C::kBitmapWords + (c >> 5), 1u << (c & 31));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  Schedule sch;
  sch.kbmax0 = kbmax[0];
  sch.kbmax1 = kbmax[1];
  sch.bm0 = SPARSE ? bitmap : nullptr;
  sch.bm1 = SPARSE ? bitmap + C::kBitmapWords : nullptr;

  if (warp < 4) {
  regs_dec<C::kRegsLow>();
  if (warp == 0) {
    // =================== TMA producer ===================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      bool qloaded[2] = {false, false};
      int i = 0;
      bool ok = true;
      for (int kb = sch.next(-1); kb >= 0 && ok; kb = sch.next(kb), ++i) {
        const int mask = sch.member(kb);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (((mask >> t) & 1) && !qloaded[t]) {
            const uint32_t qs = sbase + C::kQOff + t * C::kTileBytes;
            mbar_arrive_expect_tx(bar(C::kBarQFull + t), C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_4d(qs + c * C::kChunkBytes, &tmQ, bar(C::kBarQFull + t), c * 64, r0[t], h, b);
            qloaded[t] = true;
          }
        }
        const int sk = i % C::kStagesK;
        if (i >= C::kStagesK &&
            !wait_bar(bar(C::kBarKEmpty + sk), ((i / C::kStagesK) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        BSS_TRACE_EV(p, tr, 0, 2 * i);
        const uint32_t ks = sbase + C::kKOff + sk * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kBarKFull + sk), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(ks + c * C::kChunkBytes, &tmK, bar(C::kBarKFull + sk), c * 64, kb * kTileN, h, b);
        const int sv = i % C::kStagesV;
        if (i >= C::kStagesV &&
            !wait_bar(bar(C::kBarVEmpty + sv), ((i / C::kStagesV) & 1) ^ 1, abort_flag, p.err)) {
          ++i;  // the K load of this step is in flight
          ok = false;
          break;
        }
        BSS_TRACE_EV(p, tr, 0, 2 * i + 1);
        const uint32_t vs = sbase + C::kVOff + sv * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kBarVFull + sv), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(vs + c * C::kChunkBytes, &tmV, bar(C::kBarVFull + sv), c * 64, kb * kTileN, h, b);
      }
      // Drain: every load issued has landed before the CTA may exit (in the
      // normal path these waits return at once).
      const long long drain = 1ll << 26;
      for (int j = max(0, i - C::kStagesK); j < i; ++j)
        wait_bar(bar(C::kBarKFull + j % C::kStagesK), (j / C::kStagesK) & 1, abort_flag, p.err, drain);
      for (int j = max(0, i - C::kStagesV); j < i; ++j)
        wait_bar(bar(C::kBarVFull + j % C::kStagesV), (j / C::kStagesV) & 1, abort_flag, p.err, drain);
      for (int t = 0; t < 2; ++t)
        if (qloaded[t]) wait_bar(bar(C::kBarQFull + t), 0, abort_flag, p.err, drain);
    }
  } else if (warp == 1) {
    // =================== MMA issuer (one thread) ===================
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(kTileM, kTileN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileM, D, false, true);
      bool qready[2] = {false, false};
      bool ostarted[2] = {false, false};
      int pcount[2] = {0, 0};
      bool ok = true;

      auto issue_qk = [&](int t, int sk) -> bool {
        if (!qready[t]) {
          if (!wait_bar(bar(C::kBarQFull + t), 0, abort_flag, p.err)) return false;
          qready[t] = true;
        }
        const uint32_t qa = sbase + C::kQOff + t * C::kTileBytes;
        const uint32_t ka = sbase + C::kKOff + sk * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColS + t * 128, sdesc_sw128(qa + off, 16, 1024),
                 sdesc_sw128(ka + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarSFull + t));
        return true;
      };
      auto issue_pv = [&](int t, int sv) {
        const uint32_t va = sbase + C::kVOff + sv * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          mma_ts(tmem + C::kColO + t * D, tmem + C::kColS + t * 128 + C::kColP + kk * 8,
                 sdesc_sw128(va + kk * 16 * 128, C::kChunkBytes, 1024), kIdescPV,
                 (ostarted[t] || kk > 0) ? 1u : 0u);
        }
        ostarted[t] = true;
      };

      int kb = sch.next(-1);
      int mask = kb >= 0 ? sch.member(kb) : 0;
      if (kb >= 0) {
        ok = wait_bar(bar(C::kBarKFull + 0), 0, abort_flag, p.err);
        if (ok) {
          tc_fence_after();
          for (int t = 0; t < 2 && ok; ++t)
            if ((mask >> t) & 1) ok = issue_qk(t, 0);
          mma_commit(bar(C::kBarKEmpty + 0));
        }
      }
      int i = 0;
      while (kb >= 0 && ok) {
        const int nkb = sch.next(kb);
        const int nmask = nkb >= 0 ? sch.member(nkb) : 0;
        const int sv = i % C::kStagesV;
        const int skn = (i + 1) % C::kStagesK;
        if (!wait_bar(bar(C::kBarVFull + sv), (i / C::kStagesV) & 1, abort_flag, p.err)) break;
        BSS_TRACE_EV(p, tr, 1, 4 * i);
        tc_fence_after();
        bool kready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if ((mask >> t) & 1) {
            if (!wait_bar(bar(C::kBarPFull + t), pcount[t] & 1, abort_flag, p.err)) {
              ok = false;
              break;
            }
            ++pcount[t];
            BSS_TRACE_EV(p, tr, 1, 4 * i + 1 + t);
            tc_fence_after();
            issue_pv(t, sv);
          }
          if ((nmask >> t) & 1) {
            if (!kready) {
              if (!wait_bar(bar(C::kBarKFull + skn), ((i + 1) / C::kStagesK) & 1, abort_flag, p.err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              kready = true;
            }
            ok = issue_qk(t, skn);
          }
        }
        if (!ok) break;
        BSS_TRACE_EV(p, tr, 1, 4 * i + 3);
        mma_commit(bar(C::kBarVEmpty + sv));
        if (nkb >= 0) mma_commit(bar(C::kBarKEmpty + skn));
        kb = nkb;
        mask = nmask;
        ++i;
      }
      for (int t = 0; t < 2; ++t)
        if (ostarted[t]) mma_commit(bar(C::kBarOFull + t));
      mma_commit(bar(C::kBarMmaDone));
      wait_bar(bar(C::kBarMmaDone), 0, abort_flag, p.err);
    }
  }
  } else {
    regs_inc<C::kRegsHigh>();
    // =================== softmax warpgroups (warps 4-7: tile 0, 8-11: tile 1) ===================
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;                      // TMEM lane quarter of this warp
    const int row_in_tile = wq * 32 + lane;
    const int row = r0[t] + row_in_tile;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::kColS + t * 128;
    const uint32_t tP = tS + C::kColP;
    const uint32_t tO = tmem + lane_base + C::kColO + t * D;
    const float sl2 = p.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);

    float m2 = NEG_INF;     // reference max (log2 units), moved only by > 8
    float mt = NEG_INF;     // exact running max (log2 units)
    float l = 0.f;
    int cnt = 0;
    bool ok = true;
    for (int kb = sch.next(-1); kb >= 0; kb = sch.next(kb)) {
      if (!((sch.member(kb) >> t) & 1)) continue;
      if (!wait_bar(bar(C::kBarSFull + t), cnt & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      const bool trw = tr && lane == 0 && wq == 0;
      BSS_TRACE_EV(p, trw, 2 + t, 4 * cnt);
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);

      // element mask: only where the block crosses the diagonal or the end
      const int kstart = kb * kTileN;
      const bool edge = (kstart + kTileN > p.Lk) ||
                        (CAUSAL && (static_cast<long long>(kstart) + kTileN - 1 + p.k_offset >
                                    static_cast<long long>(r0[t]) + p.q_offset));
      if (edge) {
        long long lim = static_cast<long long>(p.Lk) - 1 - kstart;
        if (CAUSAL) lim = min(lim, static_cast<long long>(row) + p.q_offset - p.k_offset - kstart);
        const int jl = static_cast<int>(max(-1ll, min(127ll, lim)));
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j > jl) s[c][j] = __float_as_uint(NEG_INF);
      }
      // row max over 8 independent chains (short dependency chains)
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(s[0][u]);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = (c == 0 ? 8 : 0); j < 32; j += 8)
#pragma unroll
          for (int u = 0; u < 8; ++u) mx[u] = fmaxf(mx[u], __uint_as_float(s[c][j + u]));
      const float mblk =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
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
      float rs[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) rs[u] = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = half * 2 + c2;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float p0 = ex2(fmaf(__uint_as_float(s[c][j]), sl2, -mu));
            const float p1 = ex2(fmaf(__uint_as_float(s[c][j + 1]), sl2, -mu));
            rs[(j >> 1) & 3] += p0 + p1;
            pk[c2 * 16 + j / 2] = pack_bf16(p0, p1);
          }
        }
        tmem_st32(tP + half * 32, pk);
      }
      l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
      BSS_TRACE_EV(p, trw, 2 + t, 4 * cnt + 2);
      // rescale O when this row's reference max moved and O already holds data
      const bool fix = moved && cnt > 0;
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
    }

    // ---- epilogue ----
    if (ok && cnt > 0) {
      ok = wait_bar(bar(C::kBarOFull + t), 0, abort_flag, p.err);
      tc_fence_after();
    }
    BSS_TRACE_EV(p, tr && lane == 0 && wq == 0, 4 + t, 0);
    if (ok) {
      const bool inb = row < p.Lq;
      const size_t row_g = static_cast<size_t>(bh) * p.Lq + (inb ? row : 0);
      if (PARTIAL) {
        // An empty state (m = -inf) is fully described by m and l; its acc row
        // is not written (a merge never reads it).
        const float factor = (mt == NEG_INF || cnt == 0) ? 0.f : ex2(m2 - mt);
        float* dst = p.acc_out + row_g * D;
#pragma unroll 1
        for (int c = 0; c < D / 32 && cnt > 0; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
          if (inb && mt != NEG_INF) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float4 v4 = make_float4(__uint_as_float(o[j]) * factor, __uint_as_float(o[j + 1]) * factor,
                                      __uint_as_float(o[j + 2]) * factor, __uint_as_float(o[j + 3]) * factor);
              *reinterpret_cast<float4*>(dst + c * 32 + j) = v4;
            }
          }
        }
        if (inb) {
          p.m_out[row_g] = (mt == NEG_INF) ? NEG_INF : mt * kLn2;
          p.l_out[row_g] = l * factor;
        }
      } else {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* dst = p.o + row_g * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          if (cnt > 0) {
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0u;
          }
          if (inb) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 w;
              w.x = pack_bf16(__uint_as_float(o[j + 0]) * inv, __uint_as_float(o[j + 1]) * inv);
              w.y = pack_bf16(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
              w.z = pack_bf16(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv);
              w.w = pack_bf16(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + c * 32 + j) = w;
            }
          }
        }
        if (inb) p.lse[row_g] = l > 0.f ? (m2 + __log2f(l)) * kLn2 : NEG_INF;
      }
    }
  }

  if (warp >= 4) BSS_TRACE_EV(p, tr && lane == 0 && (warp & 3) == 0, 4 + ((warp - 4) >> 2), 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool SPARSE, bool PARTIAL>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t st) {
  using C = FwdCfg<D>;
  auto kern = attn_fwd_kernel<D, CAUSAL, SPARSE, PARTIAL>;
  static bool configured = false;  // per-process; the attribute is per function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.B * p.H, p.n_pairs);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, bool causal, bool sparse, bool partial, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                       cudaStream_t st) {
#define BSS_FWD_CASE(DD, CA, SP, PA)                                   \
  if (d == DD && causal == CA && sparse == SP && partial == PA)        \
    return launch_one<DD, CA, SP, PA>(tq, tk, tv, p, st);
  BSS_FWD_CASE(64, false, false, false)
  BSS_FWD_CASE(64, true, false, false)
  BSS_FWD_CASE(128, false, false, false)
  BSS_FWD_CASE(128, true, false, false)
  BSS_FWD_CASE(64, false, false, true)
  BSS_FWD_CASE(64, true, false, true)
  BSS_FWD_CASE(128, false, false, true)
  BSS_FWD_CASE(128, true, false, true)
  BSS_FWD_CASE(64, false, true, false)
  BSS_FWD_CASE(64, true, true, false)
  BSS_FWD_CASE(128, false, true, false)
  BSS_FWD_CASE(128, true, true, false)
#undef BSS_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace bss
