// Shared definitions of the device code: launch parameters, status codes,
// and the bounded-wait watchdog every spin in this library goes through.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/bss_attn.h"
#include "ptx.cuh"

namespace bss {

constexpr int kTileM = 128;      // query rows per tile (TMEM lanes)
constexpr int kTileN = 128;      // keys per KV tile
constexpr int kMaxKBlocks = 4096;  // key blocks a block-sparse launch can address
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// Watchdog: a wait that has not completed after this many SM cycles (about a
// second at GB300 clocks) gives up, records ATTN_ERR_TIMEOUT and the kernel
// unwinds.
constexpr long long kWaitLimitCycles = 1ll << 31;
constexpr uint32_t kWaitSuspendNs = 20000;   // longest single hardware suspension of a wait

// Record the first error code in the library's device status word.
__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Bounded wait on phase `parity` of an mbarrier.  Returns false (and raises the
// CTA's abort flag) when the limit expires or another role already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* err, long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    // suspended until the phase completes (or ~20 us pass): no polling traffic
    if (mbar_try_wait_suspend(bar, parity, kWaitSuspendNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      record_error(err, ATTN_ERR_TIMEOUT);
      return false;
    }
  }
}

// Row-per-thread to line-coalesced stores.  In the epilogue lane l of a warp
// holds row l of the warp's 32 rows; a store of 16 bytes per lane would touch
// 32 cache lines per instruction.  An in-register 8x8 transpose of 16-byte
// segments inside each lane octet (8g..8g+7) turns that around: before it,
// lane 8g+i holds segments 0..7 (v[4s..4s+3]) of one 128-byte line of its own
// row; after it, the same lane holds segment i of that line of rows 8g+0..7
// (row 8g+k at v[4k..4k+3]).  Each of the three butterfly stages swaps one
// bit between the row and the segment index.
__device__ __forceinline__ void transpose_octets(uint32_t (&v)[32], int lane) {
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (s & m) continue;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t a = v[4 * s + r];
        const uint32_t b = v[4 * (s | m) + r];
        const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, hi ? a : b, m);
        v[4 * s + r] = hi ? recv : a;
        v[4 * (s | m) + r] = hi ? b : recv;
      }
    }
  }
}

// Store one 128-byte line per row for the warp's 32 rows after
// transpose_octets: each instruction writes 4 whole lines.  `base` points at
// byte `line_off` of the warp's first row, rows are `row_bytes` apart, and
// only rows whose bit is set in `valid` are written.
__device__ __forceinline__ void store_octet_lines(const uint32_t (&v)[32], uint8_t* base,
                                                  size_t row_bytes, uint32_t valid, int lane) {
  const int g = lane >> 3;
  const int i = lane & 7;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int r = 8 * g + k;
    if ((valid >> r) & 1u)
      *reinterpret_cast<uint4*>(base + r * row_bytes + 16 * i) =
          make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
}

// Bounded wait used while unwinding: ignores the abort flag so that copies
// and MMAs already in flight land before the CTA releases its shared and
// tensor memory.  Gives up silently after `limit` cycles.
__device__ __forceinline__ bool drain_bar(uint32_t bar, uint32_t parity,
                                          long long limit = 1ll << 26) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (clock64() - t0 <= limit) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}

// Optional pipeline trace for performance work.  Off unless the library is
// built with -DBSS_TRACE: then the roles of one chosen CTA record clock64()
// timestamps of their pipeline events into trace[role * kTraceEvents + i]
// (a device buffer registered with attn_trace_set, trace builds only).  The
// default build compiles every trace point away.
constexpr int kTraceRoles = 8;
constexpr int kTraceEvents = 1024;
#ifdef BSS_TRACE
#define BSS_TRACE_ON(p, cta_linear) ((p).trace != nullptr && static_cast<int>(cta_linear) == (p).trace_cta)
#define BSS_TRACE_EV(p, on, role, idx)                                                  \
  do {                                                                                  \
    if ((on) && (idx) < kTraceEvents) (p).trace[(role) * kTraceEvents + (idx)] = clock64(); \
  } while (0)
#else
#define BSS_TRACE_ON(p, cta_linear) false
#define BSS_TRACE_EV(p, on, role, idx) ((void)0)
#endif

// Bounded wait for roles off the critical path: the thread is suspended in
// hardware for up to kSleepNs at a time, so that waiting warps leave the
// issue slots and the shared-memory pipe to the computing ones.
template <unsigned kSleepNs = kWaitSuspendNs>
__device__ __forceinline__ bool wait_bar_relaxed(uint32_t bar, uint32_t parity,
                                                 volatile int* abort_flag, int* err,
                                                 long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_suspend(bar, parity, kSleepNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      record_error(err, ATTN_ERR_TIMEOUT);
      return false;
    }
  }
}

struct FwdParams {
  int B, H, Lq, Lk;
  int Hkv;                 // K/V heads; query head h reads K/V head h / (H / Hkv)
  float scale_log2;        // scale * log2(e): scores are exponentiated in base 2
  long long q_offset, k_offset;
  int causal;
  // regular output
  __nv_bfloat16* o;        // [B,H,Lq,d]
  float* lse;              // [B,H,Lq]
  // partial-state output
  float* m_out;            // [B,H,Lq]
  float* l_out;            // [B,H,Lq]
  float* acc_out;          // [B,H,Lq,d]
  // block-sparse list (device CSR over 128-blocks)
  const int* row_ptr;      // [n_lists][n_qblk + 1], offsets into col_idx
  const int* col_idx;
  int n_qblk, nnz;
  int heads_per_list;      // head (b*H + h) uses list (b*H + h) / heads_per_list
  int n_pairs;             // query-row pairs per head: ceil(Lq / 256)
  int n_chunks;            // key chunks, each with its own partial state (1: none)
  int chunk_len;           // keys per chunk (a multiple of 128 when n_chunks > 1)
  int n_items;             // work items (= CTAs launched): n_chunks * B * H * n_pairs
  int head_group;          // query heads whose items are numbered together (fwd_item)
  int* err;
  long long* trace;        // trace builds only (nullptr otherwise)
  int trace_cta;
};

struct MergeParams {
  int C;
  long long rows;          // B*H*L
  const float* m;          // [C, rows]
  const float* l;          // [C, rows]
  const float* acc;        // [C, rows, d]
  __nv_bfloat16* o;        // [rows, d]
  float* lse;              // [rows]
};

struct BwdParams {
  int B, H, L;
  int Hkv;                 // K/V heads; query head h reads K/V head h / (H / Hkv)
  float scale, scale_log2;
  int causal;
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  float* delta;
  float* dq_acc;           // fp32 [B,H,L,d] workspace
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int head_group;          // heads whose key tiles are launched together (see attn_bwd_main_kernel)
  // block-sparse: key-major bitmap of the block list (bit i of column c: query
  // block i lists key block c), col_bitmap_words words per column
  const uint32_t* col_bitmap;   // [n_lists][n_kblk][col_bitmap_words]
  int col_bitmap_words;
  int heads_per_list;           // head (b*H + h) uses list (b*H + h) / heads_per_list
  // block-sparse: CTA x owns key tile j of (b, K/V head) bh, cta_order[x] =
  // bh * nq + j (nullptr: the head-grouped order)
  const int* cta_order;
  int* err;
  long long* trace;        // trace builds only (nullptr otherwise)
  int trace_cta;
};

}  // namespace bss

// Host-side launchers (defined in the .cu files, called by api.cpp).
namespace bss {
cudaError_t launch_fwd(int d, bool causal, bool sparse, bool partial, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                       cudaStream_t st);
// The forward with 256-key score tiles (fwd_wide.cu): d = 128, dense, causal
// or block-sparse, a bf16 output or (partial, not block-sparse) fp32 partial
// states per key chunk.  launch_fwd picks it; fwd_wide_takes_sparse tells
// whether its block-sparse bitmaps cover a key range of Lk.
bool fwd_wide_takes_sparse(int Lk);
cudaError_t launch_fwd_wide(bool causal, bool partial, bool sparse, const CUtensorMap& tq,
                            const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                            cudaStream_t st);
cudaError_t launch_merge(int d, const MergeParams& p, int* err, cudaStream_t st);
cudaError_t launch_bwd(int d, bool sparse, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                       const BwdParams& p, cudaStream_t st, cudaEvent_t main_begin = nullptr,
                       cudaEvent_t main_end = nullptr);
cudaError_t launch_bwd_cta_order(const uint32_t* bitmap, int words, int nq, int B, int H, int Hkv,
                                 int heads_per_list, int head_group, int* order, cudaStream_t st);
cudaError_t launch_blocklist_columns(const int* row_ptr, const int* col_idx, int n_lists, int n_qblk,
                                     int nnz, int causal, uint32_t* bitmap, int words, int* err,
                                     cudaStream_t st);
cudaError_t launch_watchdog_selftest(unsigned long long cycles, int* err, cudaStream_t st);
cudaError_t launch_blocklist_stats(const int* row_ptr, const int* col_idx, int n_lists, int n,
                                   int nnz, int L, int causal, long long* stats, int* err,
                                   cudaStream_t st);
int select_row_entries(int L, int top_r, int local, int causal);
// Sets the calling thread's text of attn_last_error_message (api.cu).
void set_error_text(const char* text);
// Rows of the dQ accumulator's tensor-map box that the backward's drain
// reduces with one bulk copy at head dimension d.
int bwd_dq_box_rows(int d);
cudaError_t launch_select(int d, const void* q, const void* k, int B, int H, int Hkv, int L,
                          int n_lists, int top_r, int local, int causal, float scale, int* row_ptr,
                          int* col_idx, float* qbar, float* kbar, cudaStream_t st);
}  // namespace bss
