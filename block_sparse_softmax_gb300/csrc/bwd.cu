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
// while the query tiles stream past.  Everything is computed transposed
// (TMEM lane = key), so that one thread owns one key row:
//   S^T  = K_j Q_i^T   and   dP^T = V_j dO_i^T         (SS MMAs, M = 128 keys)
//   the "softmax" warpgroup turns them into P^T and dS^T (bf16), written back
//   into the lower halves of the same TMEM columns (tensor-memory A operands)
//   and dS^T also into shared memory in the layout the dQ MMA reads;
//   dV  += P^T dO_i,  dK += dS^T Q_i                   (TS MMAs)
//   dQ_i = dS K_j     (SS, M = 128 queries) into the freed upper halves of the
//   S^T and dP^T columns; a second warpgroup reads it and adds it into the
//   fp32 accumulator in global memory with vector atomics.
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
  static constexpr int kStages = (D == 64) ? 2 : 1;       // Q_i / dO_i ring depth
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;
  static constexpr int kDOOff = kQOff + kStages * kTileBytes;
  static constexpr int kDSOff = kDOOff + kStages * kTileBytes;   // dS, 128 x 128 bf16
  static constexpr int kDSBytes = kTileM * kTileN * 2;
  static constexpr int kStatOff = kDSOff + kDSBytes;             // 2 x (lse2[128], delta[128])
  static constexpr int kBarOff = kStatOff + 2 * 2 * 128 * 4;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;
  static constexpr int kBarQEmpty = kBarQFull + kStages;
  static constexpr int kBarSFull = kBarQEmpty + kStages;
  static constexpr int kBarDSReady = kBarSFull + 1;
  static constexpr int kBarDQFull = kBarDSReady + 1;
  static constexpr int kBarDQFree = kBarDQFull + 1;
  static constexpr int kBarDKVFull = kBarDQFree + 1;
  static constexpr int kBarMmaDone = kBarDKVFull + 1;
  static constexpr int kBarStat = kBarMmaDone + 1;   // [2]: LSE/D of a query tile staged
  static constexpr int kNumBars = kBarStat + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColST = 0;      // S^T (fp32, 128); P^T bf16 in [0,64); dQ half 0 in [64,128)
  static constexpr uint32_t kColDPT = 128;   // dP^T (fp32, 128); dS^T bf16 in [128,192); dQ half 1 in [192,256)
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr int kThreads = 384;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
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
  if (*reinterpret_cast<volatile int*>(p.err) == ATTN_ERR_TIMEOUT) return;

  const int bh = blockIdx.x;
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int j = blockIdx.y;                       // key tile owned by this CTA
  const int L = p.L;
  const int nq = (L + kTileM - 1) / kTileM;
  const int i0 = CAUSAL ? j : 0;                  // first query tile that sees these keys
  const int n_it = nq - i0;

  if (tid == 0) {
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarQFull + s), 1);
      mbar_init(bar(C::kBarQEmpty + s), 1);
    }
    mbar_init(bar(C::kBarSFull), 1);
    mbar_init(bar(C::kBarDSReady), 128);
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQFree), 128);
    mbar_init(bar(C::kBarDKVFull), 1);
    mbar_init(bar(C::kBarMmaDone), 1);
    mbar_init(bar(C::kBarStat + 0), 128);
    mbar_init(bar(C::kBarStat + 1), 128);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + C::kMiscOff, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // =================== TMA producer ===================
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d(sbase + C::kKOff + c * C::kChunkBytes, &tmK, bar(C::kBarKV), c * 64, j * kTileN, h, b);
        tma_load_4d(sbase + C::kVOff + c * C::kChunkBytes, &tmV, bar(C::kBarKV), c * 64, j * kTileN, h, b);
      }
      int it = 0;
      for (; it < n_it; ++it) {
        const int s = it % C::kStages;
        if (it >= C::kStages &&
            !wait_bar(bar(C::kBarQEmpty + s), ((it / C::kStages) & 1) ^ 1, abort_flag, p.err))
          break;
        const int row = (i0 + it) * kTileM;
        mbar_arrive_expect_tx(bar(C::kBarQFull + s), 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_4d(sbase + C::kQOff + s * C::kTileBytes + c * C::kChunkBytes, &tmQ,
                      bar(C::kBarQFull + s), c * 64, row, h, b);
          tma_load_4d(sbase + C::kDOOff + s * C::kTileBytes + c * C::kChunkBytes, &tmDO,
                      bar(C::kBarQFull + s), c * 64, row, h, b);
        }
      }
      const long long drain = 1ll << 26;
      wait_bar(bar(C::kBarKV), 0, abort_flag, p.err, drain);
      for (int x = max(0, it - C::kStages); x < it; ++x)
        wait_bar(bar(C::kBarQFull + x % C::kStages), (x / C::kStages) & 1, abort_flag, p.err, drain);
    }
  } else if (warp == 1) {
    // =================== MMA issuer ===================
    if (lane == 0) {
      constexpr uint32_t kIdescT = idesc_bf16_f32(kTileM, kTileN, false, false);  // S^T, dP^T
      constexpr uint32_t kIdescKV = idesc_bf16_f32(kTileM, D, false, true);       // dV, dK
      constexpr uint32_t kIdescQ = idesc_bf16_f32(kTileM, 64, true, true);        // dQ halves
      bool ok = wait_bar(bar(C::kBarKV), 0, abort_flag, p.err);
      const uint32_t ka = sbase + C::kKOff, va = sbase + C::kVOff, dsa = sbase + C::kDSOff;
      for (int it = 0; it < n_it && ok; ++it) {
        const int s = it % C::kStages;
        const uint32_t qa = sbase + C::kQOff + s * C::kTileBytes;
        const uint32_t doa = sbase + C::kDOOff + s * C::kTileBytes;
        if (!wait_bar(bar(C::kBarQFull + s), (it / C::kStages) & 1, abort_flag, p.err)) break;
        // S^T and dP^T reuse the columns that held dQ of the previous tile
        if (it > 0 && !wait_bar(bar(C::kBarDQFree), (it - 1) & 1, abort_flag, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColST, sdesc_sw128(ka + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024),
                 kIdescT, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColDPT, sdesc_sw128(va + off, 16, 1024),
                 sdesc_sw128(doa + off, 16, 1024), kIdescT, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBarSFull));
        if (!wait_bar(bar(C::kBarDSReady), it & 1, abort_flag, p.err)) break;
        tc_fence_after();
        // dV += P^T dO_i ; dK += dS^T Q_i   (K dimension = the 128 queries)
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {
          mma_ts(tmem + C::kColDV, tmem + C::kColST + kk * 8,
                 sdesc_sw128(doa + kk * 2048, C::kChunkBytes, 1024), kIdescKV,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {
          mma_ts(tmem + C::kColDK, tmem + C::kColDPT + kk * 8,
                 sdesc_sw128(qa + kk * 2048, C::kChunkBytes, 1024), kIdescKV,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
        // dQ_i = dS K_j  (M = queries, K dimension = the 128 keys), one N=64 MMA per d-half
#pragma unroll
        for (int hh = 0; hh < C::kChunks; ++hh) {
          const uint32_t dcol = hh == 0 ? C::kColST + 64 : C::kColDPT + 64;
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk) {
            mma_ss(tmem + dcol, sdesc_sw128(dsa + kk * 2048, C::kChunkBytes, 1024),
                   sdesc_sw128(ka + hh * C::kChunkBytes + kk * 2048, C::kChunkBytes, 1024), kIdescQ,
                   kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(C::kBarDQFull));
        mma_commit(bar(C::kBarQEmpty + s));
      }
      mma_commit(bar(C::kBarDKVFull));
      mma_commit(bar(C::kBarMmaDone));
      wait_bar(bar(C::kBarMmaDone), 0, abort_flag, p.err);
    }
  } else if (warp >= 4 && warp < 8) {
    // =================== P^T / dS^T warpgroup (thread = key row) ===================
    const int wq = warp & 3;
    const int kr = wq * 32 + lane;
    const int key = j * kTileN + kr;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tST = tmem + lane_base + C::kColST;
    const uint32_t tDPT = tmem + lane_base + C::kColDPT;
    const float sl2 = p.scale_log2;
    const float scale = p.scale;
    const float INF = __int_as_float(0x7f800000);
    const size_t stat_base = static_cast<size_t>(bh) * L;
    uint8_t* ds_smem = smem + C::kDSOff;
    auto load_stats = [&](int i, float& l2, float& dl) {
      const int q = i * kTileM + kr;
      if (i < nq && q < L) {
        const float lse = __ldg(p.lse + stat_base + q);
        l2 = (lse == -INF) ? INF : lse * kLog2e;      // an empty row contributes nothing
        dl = __ldg(p.delta + stat_base + q);
      } else {
        l2 = INF;
        dl = 0.f;
      }
    };
    {
      float l2, dl;
      load_stats(i0, l2, dl);
      stats[kr] = l2;
      stats[128 + kr] = dl;
      mbar_arrive(bar(C::kBarStat + 0));
    }
    // Buffer (it & 1) holds the statistics of query tile i0 + it.  It is
    // rewritten (for tile it + 2) only after S^T of tile it + 1 is ready, which
    // implies every thread has finished reading it for tile it.
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int i = i0 + it;
      const float* lse2 = stats + (it & 1) * 256;
      const float* dlt = lse2 + 128;
      float l2n, dln;
      load_stats(i + 1, l2n, dln);
      if (!wait_bar(bar(C::kBarSFull), it & 1, abort_flag, p.err) ||
          !wait_bar(bar(C::kBarStat + (it & 1)), (it >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool key_ok = key < L;
      // element mask: diagonal tile (query < key) or ragged tail (query >= L: its
      // lse2 is +inf, so P is 0 there already)
      const bool diag = CAUSAL && (i == j);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sv[32], dv[32];
        tmem_ld32(tST + c * 32, sv);
        tmem_ld32(tDPT + c * 32, dv);
        tmem_ld_wait(sv);
        tmem_ld_wait(dv);
        uint32_t pk[16], dk[16];
        float dsv[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int ql = c * 32 + e;                       // query within the tile
          float pv = ex2(fmaf(__uint_as_float(sv[e]), sl2, -lse2[ql]));
          if (!key_ok || (diag && ql < kr)) pv = 0.f;
          const float ds = pv * (__uint_as_float(dv[e]) - dlt[ql]) * scale;
          dsv[e] = ds;
          if (e & 1) {
            pk[e >> 1] = pack_bf16(__uint_as_float(sv[e - 1]), pv);
          } else {
            sv[e] = __float_as_uint(pv);
          }
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) dk[e] = pack_bf16(dsv[2 * e], dsv[2 * e + 1]);
        // P^T -> columns [16c, 16c+16) of S^T (already read); dS^T likewise in dP^T
        uint32_t lo[32];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          lo[e] = pk[e];
          lo[16 + e] = dk[e];
        }
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tST + c * 16),
            "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3]), "r"(lo[4]), "r"(lo[5]), "r"(lo[6]),
            "r"(lo[7]), "r"(lo[8]), "r"(lo[9]), "r"(lo[10]), "r"(lo[11]), "r"(lo[12]), "r"(lo[13]),
            "r"(lo[14]), "r"(lo[15])
            : "memory");
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15, %16};" ::"r"(tDPT + c * 16),
            "r"(lo[16]), "r"(lo[17]), "r"(lo[18]), "r"(lo[19]), "r"(lo[20]), "r"(lo[21]),
            "r"(lo[22]), "r"(lo[23]), "r"(lo[24]), "r"(lo[25]), "r"(lo[26]), "r"(lo[27]),
            "r"(lo[28]), "r"(lo[29]), "r"(lo[30]), "r"(lo[31])
            : "memory");
        // dS into shared memory as the M-major A operand of the dQ MMA: queries
        // 64*mc .. 64*mc+63 form chunk mc, one 128-byte row per key, 16-byte
        // units swizzled by the row index.
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const int mc = c >> 1;
          const int unit = (c & 1) * 4 + u4;
          uint4 w = make_uint4(dk[u4 * 4 + 0], dk[u4 * 4 + 1], dk[u4 * 4 + 2], dk[u4 * 4 + 3]);
          *reinterpret_cast<uint4*>(ds_smem + mc * C::kChunkBytes + kr * 128 + ((unit ^ (kr & 7)) * 16)) = w;
        }
      }
      tmem_st_wait();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(bar(C::kBarDSReady));
      // statistics of the next query tile
      float* nxt = stats + ((it + 1) & 1) * 256;
      nxt[kr] = l2n;
      nxt[128 + kr] = dln;
      mbar_arrive(bar(C::kBarStat + ((it + 1) & 1)));
    }
    // ---- epilogue: dK, dV rows of this key tile ----
    if (ok) ok = wait_bar(bar(C::kBarDKVFull), 0, abort_flag, p.err);
    tc_fence_after();
    if (ok) {
      const size_t row_g = static_cast<size_t>(bh) * L + (key < L ? key : 0);
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t tsrc = tmem + lane_base + (which == 0 ? C::kColDK : C::kColDV);
        __nv_bfloat16* dst = (which == 0 ? p.dk : p.dv) + row_g * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          if (n_it > 0) {
            tmem_ld32(tsrc + c * 32, o);
            tmem_ld_wait(o);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          if (key < L) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 w;
              w.x = pack_bf16(__uint_as_float(o[e + 0]), __uint_as_float(o[e + 1]));
              w.y = pack_bf16(__uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
              w.z = pack_bf16(__uint_as_float(o[e + 4]), __uint_as_float(o[e + 5]));
              w.w = pack_bf16(__uint_as_float(o[e + 6]), __uint_as_float(o[e + 7]));
              *reinterpret_cast<uint4*>(dst + c * 32 + e) = w;
            }
          }
        }
      }
    }
  } else if (warp >= 8) {
    // =================== dQ accumulation warpgroup (thread = query row) ===================
    const int wq = warp & 3;
    const int qr = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    for (int it = 0; it < n_it; ++it) {
      if (!wait_bar(bar(C::kBarDQFull), it & 1, abort_flag, p.err)) break;
      tc_fence_after();
      uint32_t a[32], c2[32];
      tmem_ld32(tmem + lane_base + C::kColST + 64, a);
      tmem_ld32(tmem + lane_base + C::kColST + 96, c2);
      tmem_ld_wait(a);
      tmem_ld_wait(c2);
      uint32_t e2[32], f2[32];
      if (D == 128) {
        tmem_ld32(tmem + lane_base + C::kColDPT + 64, e2);
        tmem_ld32(tmem + lane_base + C::kColDPT + 96, f2);
        tmem_ld_wait(e2);
        tmem_ld_wait(f2);
      }
      tc_fence_before();
      mbar_arrive(bar(C::kBarDQFree));
      const int q = (i0 + it) * kTileM + qr;
      if (q < L) {
        float4* dst = reinterpret_cast<float4*>(p.dq_acc + (static_cast<size_t>(bh) * L + q) * D);
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          atomicAdd(dst + e / 4, make_float4(__uint_as_float(a[e]), __uint_as_float(a[e + 1]),
                                             __uint_as_float(a[e + 2]), __uint_as_float(a[e + 3])));
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          atomicAdd(dst + 8 + e / 4, make_float4(__uint_as_float(c2[e]), __uint_as_float(c2[e + 1]),
                                                 __uint_as_float(c2[e + 2]), __uint_as_float(c2[e + 3])));
        if (D == 128) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            atomicAdd(dst + 16 + e / 4, make_float4(__uint_as_float(e2[e]), __uint_as_float(e2[e + 1]),
                                                    __uint_as_float(e2[e + 2]), __uint_as_float(e2[e + 3])));
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            atomicAdd(dst + 24 + e / 4, make_float4(__uint_as_float(f2[e]), __uint_as_float(f2[e + 1]),
                                                    __uint_as_float(f2[e + 2]), __uint_as_float(f2[e + 3])));
        }
      }
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

template <int D, bool CAUSAL>
cudaError_t launch_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const BwdParams& p, cudaStream_t st) {
  using C = BwdCfg<D>;
  auto kern = attn_bwd_main_kernel<D, CAUSAL>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.B * p.H, (p.L + kTileN - 1) / kTileN);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

unsigned grid_for(long long work, int per_block) {
  long long blocks = (work + per_block - 1) / per_block;
  const long long cap = 152LL * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, cudaStream_t st) {
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
  if (d == 64)
    e = p.causal ? launch_main<64, true>(tq, tk, tv, tdo, p, st) : launch_main<64, false>(tq, tk, tv, tdo, p, st);
  else
    e = p.causal ? launch_main<128, true>(tq, tk, tv, tdo, p, st) : launch_main<128, false>(tq, tk, tv, tdo, p, st);
  if (e != cudaSuccess) return e;
  const long long n8 = rows * d / 8;
  attn_bwd_dq_convert_kernel<<<grid_for(n8, 256), 256, 0, st>>>(p.dq_acc, p.dq, n8);
  return cudaGetLastError();
}

}  // namespace bss
