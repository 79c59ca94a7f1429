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
// Three small kernels: the block means (HBM-bound: Q and K are read once),
// the row offsets (which depend on the shapes only), and one CTA per
// (list, query block) that scores its candidates and picks the top_r by
// repeated block-wide arg-max.
#include "common.cuh"

namespace bss {
namespace {

constexpr int kSelThreads = 256;

// out[bh][c][:] = mean of rows c*128 .. min(L, c*128+128)-1 of x[bh] (bf16 -> fp32).
template <int D>
__global__ void __launch_bounds__(D) pool_blocks_kernel(const __nv_bfloat16* x, float* out, int L,
                                                        int n) {
  const long long bhc = blockIdx.x;
  const long long bh = bhc / n;
  const int c = static_cast<int>(bhc - bh * n);
  const int r0 = c * kTileN;
  const int r1 = min(L, r0 + kTileN);
  const __nv_bfloat16* src = x + (bh * L + r0) * D + threadIdx.x;
  float s = 0.f;
  for (int r = r0; r < r1; ++r, src += D) s += __bfloat162float(*src);
  out[bhc * D + threadIdx.x] = s / static_cast<float>(r1 - r0);
}

// Keys a row keeps: the window and min(top_r, other candidates).
__device__ __host__ __forceinline__ int select_row_count(int a, int n, int top_r, int local,
                                                        int causal) {
  const int last = causal ? a : n - 1;
  const int window = min(a + 1, local);
  return window + min(top_r, last + 1 - window);
}

// prefix[a] = entries of rows 0..a-1 of one list; row_ptr[l][a] = l*prefix[n] + prefix[a].
__global__ void __launch_bounds__(kSelThreads) select_rowptr_kernel(int* prefix, int* row_ptr,
                                                                   int n_lists, int n, int top_r,
                                                                   int local, int causal) {
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int a = 0; a < n; ++a) {
      prefix[a] = acc;
      acc += select_row_count(a, n, top_r, local, causal);
    }
    prefix[n] = acc;
  }
  __syncthreads();
  const long long total = static_cast<long long>(n_lists) * (n + 1);
  for (long long x = threadIdx.x; x < total; x += blockDim.x) {
    const int l = static_cast<int>(x / (n + 1));
    const int a = static_cast<int>(x - static_cast<long long>(l) * (n + 1));
    row_ptr[x] = l * prefix[n] + prefix[a];
  }
}

// True when (v1, i1) ranks before (v2, i2): larger score, then lower index.
__device__ __forceinline__ bool ranks_before(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

template <int D>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const float* qbar, const float* kbar,
                                                            const int* prefix, int* col_idx, int n,
                                                            int hpl, int top_r, int local,
                                                            int causal, float scale, int H,
                                                            int group) {
  extern __shared__ float sel_smem[];
  float* qs = sel_smem;               // [hpl][D] query block means of the list's heads
  float* sc = sel_smem + hpl * D;     // [n] candidate scores (-inf: not a candidate)
  __shared__ float red_v[kSelThreads / 32];
  __shared__ int red_i[kSelThreads / 32];
  __shared__ int picked[256];
  const int l = blockIdx.x / n;
  const int a = blockIdx.x - l * n;
  const int tid = threadIdx.x;
  const float NEG_INF = -__int_as_float(0x7f800000);
  for (int i = tid; i < hpl * D; i += kSelThreads) {
    const int x = i / D;
    qs[i] = qbar[((static_cast<size_t>(l) * hpl + x) * n + a) * D + (i - x * D)];
  }
  __syncthreads();
  const int last = causal ? a : n - 1;
  const int wlo = max(0, a - local + 1);
  for (int c = tid; c < n; c += kSelThreads) {
    float v = NEG_INF;
    if (c <= last && !(c >= wlo && c <= a)) {
      v = 0.f;
      for (int x = 0; x < hpl; ++x) {
        // query head (b, hq) = l*hpl + x reads the block means of K/V head hq / group
        const int bhq = l * hpl + x;
        const int bq = bhq / H;
        const size_t bkv = static_cast<size_t>(bq) * (H / group) + (bhq - bq * H) / group;
        const float* kr = kbar + (bkv * n + c) * D;
        const float* qr = qs + x * D;
        float dot = 0.f;
#pragma unroll 8
        for (int e = 0; e < D; ++e) dot = fmaf(qr[e], __ldg(kr + e), dot);
        v += scale * dot;
      }
      if (!(v == v)) v = -3.402823466e38f;   // a NaN score ranks last among candidates
    }
    sc[c] = v;
  }
  __syncthreads();
  const int window = min(a + 1, local);
  const int k = min(top_r, last + 1 - window);
  for (int round = 0; round < k; ++round) {
    float bv = NEG_INF;
    int bi = 0x7fffffff;
    for (int c = tid; c <= last; c += kSelThreads) {
      const float v = sc[c];
      if (v != NEG_INF && ranks_before(v, c, bv, bi)) {
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
    if ((tid & 31) == 0) {
      red_v[tid >> 5] = bv;
      red_i[tid >> 5] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kSelThreads / 32; ++w)
        if (ranks_before(red_v[w], red_i[w], bv, bi)) {
          bv = red_v[w];
          bi = red_i[w];
        }
      picked[round] = bi;
      sc[bi] = NEG_INF;
    }
    __syncthreads();
  }
  if (tid == 0) {
    // window then picks, sorted ascending (insertion sort of at most 256)
    int row[256];
    int m = 0;
    for (int c = wlo; c <= a && c <= last; ++c) row[m++] = c;
    for (int r = 0; r < k; ++r) {
      const int v = picked[r];
      int j = m++;
      while (j > 0 && row[j - 1] > v) {
        row[j] = row[j - 1];
        --j;
      }
      row[j] = v;
    }
    int* dst = col_idx + static_cast<size_t>(l) * prefix[n] + prefix[a];
    for (int j = 0; j < m; ++j) dst[j] = row[j];
  }
}

template <int D>
cudaError_t launch_select_d(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H, int Hkv,
                            int L, int n_lists, int top_r, int local, int causal, float scale,
                            int* row_ptr, int* col_idx, float* qbar, float* kbar, int* prefix,
                            cudaStream_t st) {
  const int n = (L + kTileN - 1) / kTileN;
  const long long bhn = static_cast<long long>(B) * H * n;
  const long long bkvn = static_cast<long long>(B) * Hkv * n;
  pool_blocks_kernel<D><<<static_cast<unsigned>(bhn), D, 0, st>>>(q, qbar, L, n);
  pool_blocks_kernel<D><<<static_cast<unsigned>(bkvn), D, 0, st>>>(k, kbar, L, n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  select_rowptr_kernel<<<1, kSelThreads, 0, st>>>(prefix, row_ptr, n_lists, n, top_r, local, causal);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int hpl = static_cast<int>(static_cast<long long>(B) * H / n_lists);
  const size_t smem = (static_cast<size_t>(hpl) * D + n) * sizeof(float);
  auto kern = select_kernel<D>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem))) != cudaSuccess)
    return e;
  kern<<<static_cast<unsigned>(static_cast<long long>(n_lists) * n), kSelThreads, smem, st>>>(
      qbar, kbar, prefix, col_idx, n, hpl, top_r, local, causal, scale, H, H / Hkv);
  return cudaGetLastError();
}

}  // namespace

int select_row_entries(int L, int top_r, int local, int causal) {
  const int n = (L + kTileN - 1) / kTileN;
  int acc = 0;
  for (int a = 0; a < n; ++a) acc += select_row_count(a, n, top_r, local, causal);
  return acc;
}

cudaError_t launch_select(int d, const void* q, const void* k, int B, int H, int Hkv, int L,
                          int n_lists, int top_r, int local, int causal, float scale, int* row_ptr,
                          int* col_idx, float* qbar, float* kbar, int* prefix, cudaStream_t st) {
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  const auto* kk = static_cast<const __nv_bfloat16*>(k);
  if (d == 64)
    return launch_select_d<64>(qq, kk, B, H, Hkv, L, n_lists, top_r, local, causal, scale, row_ptr,
                               col_idx, qbar, kbar, prefix, st);
  if (d == 128)
    return launch_select_d<128>(qq, kk, B, H, Hkv, L, n_lists, top_r, local, causal, scale, row_ptr,
                                col_idx, qbar, kbar, prefix, st);
  return cudaErrorInvalidValue;
}

}  // namespace bss
