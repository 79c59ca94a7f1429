// Merge of C partial online-softmax states into the final output, and the
// watchdog self-test kernel.
//
// "Exact Blocks, Rings, and Sparsity", section 4: two states over disjoint key
// sets combine by rescaling both to the larger maximum and adding their l and A
// terms; the operator is associative, so C states merge in one pass with
// m* = max_c m_c, l* = sum_c e^{m_c - m*} l_c, A* = sum_c e^{m_c - m*} A_c,
// O = A*/l*, LSE = m* + ln l*.
//
// The kernel is bound by HBM bandwidth: every row reads C (m, l) pairs and the
// A rows of its non-empty states (an empty state, m = -inf, is never read) and
// writes one bf16 O row and one LSE.  D/4 threads cover one row with 16-byte
// loads, so a warp reads 512 contiguous bytes per state; a grid-stride loop
// over rows keeps several independent loads per thread in flight.
#include "common.cuh"

namespace bss {
namespace {

template <int D>
__global__ void __launch_bounds__(256) merge_states_kernel(const MergeParams p) {
  constexpr int G = D / 4;                       // threads per row
  const int g = static_cast<int>(threadIdx.x) % G;
  const long long first = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / G;
  const long long step = (static_cast<long long>(gridDim.x) * blockDim.x) / G;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const long long rows = p.rows;
  for (long long r = first; r < rows; r += step) {
    float ms = NEG_INF;
#pragma unroll 8
    for (int c = 0; c < p.C; ++c) ms = fmaxf(ms, __ldg(p.m + c * rows + r));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float ls = 0.f;
    if (ms != NEG_INF) {
#pragma unroll 8
      for (int c = 0; c < p.C; ++c) {
        const float mc = __ldg(p.m + c * rows + r);
        if (mc == NEG_INF) continue;
        const float w = ex2((mc - ms) * kLog2e);
        ls = fmaf(w, __ldg(p.l + c * rows + r), ls);
        const float4 a = __ldg(reinterpret_cast<const float4*>(p.acc + (c * rows + r) * D) + g);
        acc.x = fmaf(w, a.x, acc.x);
        acc.y = fmaf(w, a.y, acc.y);
        acc.z = fmaf(w, a.z, acc.z);
        acc.w = fmaf(w, a.w, acc.w);
      }
    }
    const float inv = ls > 0.f ? 1.f / ls : 0.f;
    uint2 out;
    out.x = pack_bf16(acc.x * inv, acc.y * inv);
    out.y = pack_bf16(acc.z * inv, acc.w * inv);
    *(reinterpret_cast<uint2*>(p.o + r * D) + g) = out;
    if (g == 0) p.lse[r] = ls > 0.f ? ms + __logf(ls) : NEG_INF;
  }
}

__global__ void watchdog_selftest_kernel(unsigned long long cycles, int* err) {
  __shared__ __align__(8) uint64_t never_arrived;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&never_arrived), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    wait_bar(smem_u32(&never_arrived), 0, &abort_flag, err, static_cast<long long>(cycles));
}

// Exponential-unit rate: every thread runs eight independent chains of
// y <- 2^(-y - 1/2), whose values stay in [2^-1.5, 2^-0.5], so the number of
// ex2.approx instructions in flight, not their latency, sets the time.  Each
// thread evaluates 8 * iters exponentials.  `sink` is written only when the
// sum is negative, which it never is; the branch keeps the work alive.
__global__ void __launch_bounds__(256) ex2_rate_kernel(float* sink, int iters) {
  float y[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) y[k] = 0.5f + 0.03125f * static_cast<float>(k) +
                                     1e-4f * static_cast<float>(threadIdx.x & 31);
  for (int n = 0; n < iters; ++n) {
#pragma unroll
    for (int k = 0; k < 8; ++k) y[k] = ex2(-y[k] - 0.5f);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += y[k];
  if (s < 0.f) *sink = s;
}

}  // namespace

cudaError_t launch_ex2_rate(float* sink, int blocks, int iters, cudaStream_t st) {
  ex2_rate_kernel<<<blocks, 256, 0, st>>>(sink, iters);
  return cudaGetLastError();
}

cudaError_t launch_merge(int d, const MergeParams& p, int* err, cudaStream_t st) {
  (void)err;
  if (p.rows == 0) return cudaSuccess;
  const int G = d / 4;
  const long long threads = p.rows * G;
  long long blocks = (threads + 255) / 256;
  const long long cap = 152LL * 16;
  if (blocks > cap) blocks = cap;
  if (d == 64)
    merge_states_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, st>>>(p);
  else if (d == 128)
    merge_states_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, st>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(unsigned long long cycles, int* err, cudaStream_t st) {
  watchdog_selftest_kernel<<<1, 32, 0, st>>>(cycles, err);
  return cudaGetLastError();
}

}  // namespace bss
