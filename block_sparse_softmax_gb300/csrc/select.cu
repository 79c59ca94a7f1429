// Mean-pooled block selector: the block lists the block-sparse kernels visit.
//
// What it computes ("Exact Blocks, Rings, and Sparsity", section 5, 'Why the
// sparse unit is usually a block' and 'Fixed pooling: a cheap proxy, not the
// true block mass'; section 6 on grouped heads sharing one block choice):
//   kbar_c = mean of the key rows of block c, qbar_a likewise for queries;
//   score(a, c) = sum over the heads sharing a list of scale * qbar_a . kbar_c
//   (the mean logit of the block pair, added over the heads);
//   row a keeps the local window a, a-1, .., a-local+1 and the top_r other
//   candidates (under a causal mask blocks 0..a), ties to the lower index,
//   in ascending order.
// Two kernels: the block means of Q and K (HBM-bound: both are read once),
// then one warp per (list, query block) that scores its candidates, picks the
// top_r by repeated warp-wide arg-max and writes its row and row offset.
//
// Also here: the accounting of a block list (attn_blocklist_stats), which
// reports what a list asks the block-sparse kernels to do (block-sparse
// attention patterns page, 'Count active blocks and acknowledge the changed
// operator': logical allowed pairs beside the executed tiles, and listed
// blocks wholly in the causal future, which contribute nothing).
#include "common.cuh"

namespace bss {
namespace {

constexpr int kPoolThreads = 256;

// Block means of Q and of K in one launch: CTA x < n_q_items pools block
// (bh, c) of q into qbar, the rest pool k into kbar.  out[bh][c][:] = mean of
// rows c*128 .. min(L, c*128+128)-1 (bf16 -> fp32).  Each thread owns one
// 8-column slice (16-byte loads) of every RG-th row, so a CTA has all of its
// 32 KB (d=128) in flight at once; the RG partial sums meet in shared memory.
template <int D>
__global__ void __launch_bounds__(kPoolThreads) pool_blocks_kernel(const __nv_bfloat16* q,
                                                                   const __nv_bfloat16* k,
                                                                   float* qbar, float* kbar,
                                                                   int L, int n,
                                                                   long long n_q_items) {
  constexpr int kVec = 8;                       // bf16 per 16-byte load
  constexpr int kSlices = D / kVec;             // 16-byte slices per row
  constexpr int kRG = kPoolThreads / kSlices;   // row groups
  __shared__ float part[kRG][D];
  long long item = blockIdx.x;
  const __nv_bfloat16* x = q;
  float* out = qbar;
  if (item >= n_q_items) {
    item -= n_q_items;
    x = k;
    out = kbar;
  }
  const long long bh = item / n;
  const int c = static_cast<int>(item - bh * n);
  const int r0 = c * kTileN;
  const int rows = min(L, r0 + kTileN) - r0;
  const int slice = threadIdx.x % kSlices;
  const int rg = threadIdx.x / kSlices;
  const __nv_bfloat16* base = x + (bh * L + r0) * D + slice * kVec;
  float acc[kVec];
#pragma unroll
  for (int e = 0; e < kVec; ++e) acc[e] = 0.f;
  constexpr int kPerThread = kTileN / kRG;
  uint4 v[kPerThread];
#pragma unroll
  for (int t = 0; t < kPerThread; ++t) {
    const int r = rg + t * kRG;
    v[t] = r < rows ? __ldg(reinterpret_cast<const uint4*>(base + static_cast<long long>(r) * D))
                    : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int t = 0; t < kPerThread; ++t) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[t]);
#pragma unroll
    for (int e = 0; e < kVec / 2; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      acc[2 * e] += f.x;
      acc[2 * e + 1] += f.y;
    }
  }
#pragma unroll
  for (int e = 0; e < kVec; ++e) part[rg][slice * kVec + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < kRG; ++g) s += part[g][threadIdx.x];
    out[(bh * n + c) * D + threadIdx.x] = s / static_cast<float>(rows);
  }
}

// Keys a row keeps: the window and min(top_r, other candidates).
__device__ __host__ __forceinline__ int select_row_count(int a, int n, int top_r, int local,
                                                        int causal) {
  const int last = causal ? a : n - 1;
  const int window = min(a + 1, local);
  return window + min(top_r, last + 1 - window);
}

// True when (v1, i1) ranks before (v2, i2): larger score, then lower index.
__device__ __forceinline__ bool ranks_before(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// One CTA per (list l, kSelWarps consecutive query blocks a0 .. a0+7).
//   * The list's query heads l*hpl .. l*hpl+hpl-1 read K/V heads
//     (b*H + h) / group, a run kv0 .. kv1 of consecutive K/V heads.  For each,
//     warp w adds the query means of the heads sharing it into row w of qs;
//     then warp w copies the key means of candidates c0 + 16*w .. +15 into its
//     slice of shared memory (one coalesced 512-byte row per load, rows padded
//     by 4 floats so that 16-byte reads of eight consecutive rows hit distinct
//     banks), and lane i takes candidate c0 + 16*w + i%16 and half i/16 of the
//     d dimensions and accumulates it against all eight query rows, so each
//     key value feeds eight fused multiply-adds.  The two halves meet by one
//     shuffle and the scores land in the rows' score arrays:
//     score(a, c) = scale * sum_j qsum_j . kbar[kv0 + j][c].
//   * Warp w then owns query block a0 + w: top_r rounds of warp-wide arg-max
//     (larger score, then lower index); a picked block is marked NaN in the
//     row, which no later round takes (scores themselves are NaN-free: a NaN
//     score becomes -FLT_MAX).
//   * The row (window and picks) is written in ascending order with ballots;
//     row_ptr[l][a] = l * total + entries of rows 0 .. a-1, both counted here
//     from the closed-form row sizes.
constexpr int kSelWarps = 8;
constexpr int kSelRows = 16;                        // candidates per warp and pass
constexpr int kSelPass = kSelWarps * kSelRows;      // candidates scored per pass

template <int D>
__host__ __device__ constexpr int select_kstride() { return D + 4; }

template <int D>
__host__ __device__ constexpr size_t select_smem_bytes(int n) {
  return (static_cast<size_t>(kSelWarps) * kSelRows * select_kstride<D>() +
          static_cast<size_t>(kSelWarps) * D + static_cast<size_t>(kSelWarps) * n) * sizeof(float);
}

template <int D>
__global__ void __launch_bounds__(kSelWarps * 32) select_kernel(
    const float* qbar, const float* kbar, int* row_ptr, int* col_idx, int n, int hpl, int top_r,
    int local, int causal, float scale, int group) {
  constexpr int kHalf = D / 2;
  constexpr int kStride = select_kstride<D>();
  extern __shared__ float sel_smem[];
  float* ks = sel_smem;                                   // [kSelWarps][kSelRows][D+4] key means
  float* qs = ks + kSelWarps * kSelRows * kStride;        // [kSelWarps][D] summed query means
  float* scs = qs + kSelWarps * D;                        // [kSelWarps][n] score rows
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int tiles = (n + kSelWarps - 1) / kSelWarps;
  const int l = blockIdx.x / tiles;
  const int a0 = (blockIdx.x - l * tiles) * kSelWarps;
  const int a = a0 + warp;
  const bool active = a < n;                              // tail warps only help score
  float* sc = scs + static_cast<size_t>(warp) * n;        // this warp's score row
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int last = causal ? a : n - 1;
  const int n_cand = last + 1;
  const int n_stage = causal ? min(n, a0 + kSelWarps) : n;   // candidates any row scores
  const int rows = min(kSelWarps, n - a0);
  const long long h_lo = static_cast<long long>(l) * hpl;
  const int kv0 = static_cast<int>(h_lo / group);
  const int kv1 = static_cast<int>((h_lo + hpl - 1) / group);
  const int half = lane >> 4;

  for (int kvh = kv0; kvh <= kv1; ++kvh) {
    if (active) {
      const long long x0 = max(h_lo, static_cast<long long>(kvh) * group);
      const long long x1 = min(h_lo + hpl, static_cast<long long>(kvh + 1) * group);
      for (int e = lane; e < D; e += 32) {
        float sum = 0.f;
        for (long long x = x0; x < x1; ++x) sum += __ldg(qbar + (x * n + a) * D + e);
        qs[warp * D + e] = sum;
      }
    }
    __syncthreads();                    // qs complete
    const float* kb = kbar + static_cast<size_t>(kvh) * n * D;
    float* kw = ks + warp * kSelRows * kStride;
    for (int c0 = 0; c0 < n_stage; c0 += kSelPass) {
      const int cw = c0 + warp * kSelRows;               // this warp's first candidate
      if (cw >= n_stage) continue;
      {
        if constexpr (D == 128) {
          float4 t[kSelRows];
#pragma unroll
          for (int i = 0; i < kSelRows; ++i)
            t[i] = __ldg(reinterpret_cast<const float4*>(
                kb + static_cast<size_t>(min(cw + i, n - 1)) * D + lane * 4));
#pragma unroll
          for (int i = 0; i < kSelRows; ++i)
            *reinterpret_cast<float4*>(kw + i * kStride + lane * 4) = t[i];
        } else {
          // D = 64: a row is 16 float4, two rows per load
          float4 t[kSelRows / 2];
#pragma unroll
          for (int i = 0; i < kSelRows / 2; ++i) {
            const int row = 2 * i + (lane >> 4);
            t[i] = __ldg(reinterpret_cast<const float4*>(
                kb + static_cast<size_t>(min(cw + row, n - 1)) * D + (lane & 15) * 4));
          }
#pragma unroll
          for (int i = 0; i < kSelRows / 2; ++i) {
            const int row = 2 * i + (lane >> 4);
            *reinterpret_cast<float4*>(kw + row * kStride + (lane & 15) * 4) = t[i];
          }
        }
      }
      __syncwarp();
      const int c = cw + (lane & 15);
      const float* kr = kw + (lane & 15) * kStride + half * kHalf;
      float acc[kSelWarps];
#pragma unroll
      for (int r = 0; r < kSelWarps; ++r) acc[r] = 0.f;
#pragma unroll 4
      for (int e = 0; e < kHalf; e += 4) {
        const float4 kv = *reinterpret_cast<const float4*>(kr + e);
#pragma unroll
        for (int r = 0; r < kSelWarps; ++r) {
          const float4 qv = *reinterpret_cast<const float4*>(qs + r * D + half * kHalf + e);
          acc[r] = fmaf(qv.x, kv.x, acc[r]);
          acc[r] = fmaf(qv.y, kv.y, acc[r]);
          acc[r] = fmaf(qv.z, kv.z, acc[r]);
          acc[r] = fmaf(qv.w, kv.w, acc[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < kSelWarps; ++r) acc[r] += __shfl_xor_sync(0xFFFFFFFFu, acc[r], 16);
      if (half == 0 && c < n_stage) {
#pragma unroll
        for (int r = 0; r < kSelWarps; ++r) {
          if (r < rows) {
            float* dst = scs + static_cast<size_t>(r) * n + c;
            *dst = kvh == kv0 ? acc[r] : *dst + acc[r];
          }
        }
      }
      __syncwarp();                     // kw is refilled by the next pass
    }
    __syncthreads();                    // scores of this K/V head in; qs reusable
  }
  if (!active) return;

  // row offsets: entries of rows 0 .. a-1 and of the whole list
  int before = 0, total = 0;
  for (int r = lane; r < n; r += 32) {
    const int cnt = select_row_count(r, n, top_r, local, causal);
    total += cnt;
    if (r < a) before += cnt;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    before += __shfl_xor_sync(0xFFFFFFFFu, before, off);
    total += __shfl_xor_sync(0xFFFFFFFFu, total, off);
  }
  const long long list_base = static_cast<long long>(l) * total;
  if (lane == 0) {
    row_ptr[static_cast<size_t>(l) * (n + 1) + a] = static_cast<int>(list_base + before);
    if (a == n - 1) row_ptr[static_cast<size_t>(l) * (n + 1) + n] = static_cast<int>(list_base + total);
  }

  // final scores; window and non-candidates are -inf
  const int wlo = max(0, a - local + 1);
  for (int c = lane; c < n; c += 32) {
    float v = NEG_INF;
    if (c < n_cand && !(c >= wlo && c <= a)) {
      v = scale * sc[c];
      // a NaN or -inf score ranks last among candidates (and stays one)
      if (!(v == v) || v == NEG_INF) v = -3.402823466e38f;
    }
    sc[c] = v;
  }
  __syncwarp();
  const int window = min(a + 1, local);
  const int k = min(top_r, n_cand - window);
  const float NAN_MARK = __int_as_float(0x7fc00000);
  for (int round = 0; round < k; ++round) {
    float bv = NEG_INF;
    int bi = 0x7fffffff;
    for (int c = lane; c < n_cand; c += 32) {
      const float v = sc[c];
      if (v != NEG_INF && ranks_before(v, c, bv, bi)) {   // NaN (picked) never ranks
        bv = v;
        bi = c;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (ranks_before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0 && bi < n_cand) sc[bi] = NAN_MARK;
    __syncwarp();
  }
  // ascending write of the window and the picks
  int* dst = col_idx + list_base + before;
  int written = 0;
  for (int c0 = 0; c0 < n_cand; c0 += 32) {
    const int c = c0 + lane;
    bool keep = false;
    if (c < n_cand) {
      const float v = sc[c];
      keep = (c >= wlo && c <= a) || !(v == v);
    }
    const unsigned ballot = __ballot_sync(0xFFFFFFFFu, keep);
    if (keep) dst[written + __popc(ballot & ((1u << lane) - 1u))] = c;
    written += __popc(ballot);
  }
}

template <int D>
cudaError_t launch_select_d(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H, int Hkv,
                            int L, int n_lists, int top_r, int local, int causal, float scale,
                            int* row_ptr, int* col_idx, float* qbar, float* kbar,
                            cudaStream_t st) {
  const int n = (L + kTileN - 1) / kTileN;
  const long long bhn = static_cast<long long>(B) * H * n;
  const long long bkvn = static_cast<long long>(B) * Hkv * n;
  pool_blocks_kernel<D><<<static_cast<unsigned>(bhn + bkvn), kPoolThreads, 0, st>>>(
      q, k, qbar, kbar, L, n, bhn);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int group = H / Hkv;
  const int hpl = static_cast<int>(static_cast<long long>(B) * H / n_lists);
  const size_t smem = select_smem_bytes<D>(n);
  auto kern = select_kernel<D>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem))) != cudaSuccess)
    return e;
  const long long tiles = (n + kSelWarps - 1) / kSelWarps;
  kern<<<static_cast<unsigned>(n_lists * tiles), kSelWarps * 32, smem, st>>>(
      qbar, kbar, row_ptr, col_idx, n, hpl, top_r, local, causal, scale, group);
  return cudaGetLastError();
}

// Block-list accounting: one CTA per list, one warp per query block at a
// time.  The warp turns the row's raw entries into a bitmap in shared memory
// (duplicates collapse, order is irrelevant), then walks the set bits.  On the
// square, unshifted sequence of the block-sparse kernels a listed block c of
// query block a is wholly in the causal future exactly when c > a; every other
// listed block holds allowed pairs: all (rows x keys) pairs before the
// diagonal, n (n + 1) / 2 on the diagonal block of n tokens.  Malformed rows and
// entries are skipped and reported as the block-sparse kernels report them.
constexpr int kStatWarps = 8;
constexpr int kStatWords = kMaxKBlocks / 32;

__global__ void __launch_bounds__(kStatWarps * 32) blocklist_stats_kernel(
    const int* row_ptr, const int* col_idx, int n, int nnz, int L, int causal,
    long long* stats, int* err) {
  __shared__ uint32_t bm[kStatWarps][kStatWords];
  __shared__ unsigned long long part[kStatWarps][4];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int list = blockIdx.x;
  const int* rp = row_ptr + static_cast<size_t>(list) * (n + 1);
  const int words = (n + 31) / 32;
  unsigned long long listed = 0, executed = 0, future = 0, pairs = 0;
  for (int a = warp; a < n; a += kStatWarps) {
    for (int w = lane; w < words; w += 32) bm[warp][w] = 0u;
    __syncwarp();
    const int beg = __ldg(rp + a);
    const int end = __ldg(rp + a + 1);
    if (beg < 0 || end < beg || end > nnz) {
      if (lane == 0) record_error(err, ATTN_ERR_BAD_BLOCKLIST);
    } else {
      for (int e = beg + lane; e < end; e += 32) {
        const int c = __ldg(col_idx + e);
        if (c < 0 || c >= n) {
          record_error(err, ATTN_ERR_BAD_BLOCKLIST);
          continue;
        }
        atomicOr(&bm[warp][c >> 5], 1u << (c & 31));
      }
    }
    __syncwarp();
    const long long nq = min(L, (a + 1) * kTileN) - a * kTileN;
    for (int w = lane; w < words; w += 32) {
      uint32_t bits = bm[warp][w];
      while (bits) {
        const int c = 32 * w + __ffs(bits) - 1;
        bits &= bits - 1u;
        ++listed;
        if (causal && c > a) {
          ++future;
          continue;
        }
        ++executed;
        const long long nk = min(L, (c + 1) * kTileN) - c * kTileN;
        pairs += (causal && c == a) ? nq * (nq + 1) / 2 : nq * nk;
      }
    }
    __syncwarp();
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    listed += __shfl_xor_sync(0xFFFFFFFFu, listed, o);
    executed += __shfl_xor_sync(0xFFFFFFFFu, executed, o);
    future += __shfl_xor_sync(0xFFFFFFFFu, future, o);
    pairs += __shfl_xor_sync(0xFFFFFFFFu, pairs, o);
  }
  if (lane == 0) {
    part[warp][0] = listed;
    part[warp][1] = executed;
    part[warp][2] = future;
    part[warp][3] = pairs;
  }
  __syncthreads();
  if (threadIdx.x < 4) {
    unsigned long long t = 0;
    for (int w = 0; w < kStatWarps; ++w) t += part[w][threadIdx.x];
    stats[static_cast<size_t>(list) * 4 + threadIdx.x] = static_cast<long long>(t);
  }
}

}  // namespace

cudaError_t launch_blocklist_stats(const int* row_ptr, const int* col_idx, int n_lists, int n,
                                   int nnz, int L, int causal, long long* stats, int* err,
                                   cudaStream_t st) {
  if (n_lists <= 0) return cudaSuccess;
  blocklist_stats_kernel<<<static_cast<unsigned>(n_lists), kStatWarps * 32, 0, st>>>(
      row_ptr, col_idx, n, nnz, L, causal, stats, err);
  return cudaGetLastError();
}

int select_row_entries(int L, int top_r, int local, int causal) {
  const int n = (L + kTileN - 1) / kTileN;
  int acc = 0;
  for (int a = 0; a < n; ++a) acc += select_row_count(a, n, top_r, local, causal);
  return acc;
}

cudaError_t launch_select(int d, const void* q, const void* k, int B, int H, int Hkv, int L,
                          int n_lists, int top_r, int local, int causal, float scale, int* row_ptr,
                          int* col_idx, float* qbar, float* kbar, cudaStream_t st) {
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  const auto* kk = static_cast<const __nv_bfloat16*>(k);
  if (d == 64)
    return launch_select_d<64>(qq, kk, B, H, Hkv, L, n_lists, top_r, local, causal, scale, row_ptr,
                               col_idx, qbar, kbar, st);
  if (d == 128)
    return launch_select_d<128>(qq, kk, B, H, Hkv, L, n_lists, top_r, local, causal, scale, row_ptr,
                                col_idx, qbar, kbar, st);
  return cudaErrorInvalidValue;
}

}  // namespace bss
