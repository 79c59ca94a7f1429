// The C ABI of libbss_attn.so: argument validation, TMA descriptor encoding,
// the device status word, and the host-side block-list normalisation.  Every
// arithmetic step of the attention path runs in the kernels of fwd.cu,
// merge.cu and bwd.cu; this file only checks, describes and launches.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace bss {
namespace {

// First error recorded by any kernel of this library on a device (0 = none).
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {nullptr};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

thread_local char g_last_error[256] = {0};

// attn_bwd_time_main: events recorded around each backward's main kernel
// (process-wide; NULL when off)
cudaEvent_t g_bwd_main_ev[2] = {nullptr, nullptr};

#ifdef BSS_TRACE
long long* g_trace_buf = nullptr;
int g_trace_cta = 0;
#endif

void set_error(const char* where, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
}

// Device address of the status word for the current device.
attn_status_t status_word(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice", e);
    return ATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(g_last_error, sizeof(g_last_error),
             "device %d is beyond the %d devices this library keeps state for", dev, kMaxDevices);
    return ATTN_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) {
      set_error("cudaGetSymbolAddress", e);
      return ATTN_ERR_CUDA;
    }
    g_status_ptr[dev] = static_cast<int*>(ptr);
  }
  *out = g_status_ptr[dev];
  return ATTN_OK;
}

attn_status_t get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return ATTN_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
    set_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", e);
    return ATTN_ERR_CUDA;
  }
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return ATTN_OK;
}

// [B, H, L, d] bf16 contiguous, viewed as a 4-D tensor (d, L, H, B) with boxes
// of 64 d-elements (128 bytes, swizzled) by 128 rows.  Rows beyond L (the
// ragged tail of a head) are zero-filled by the copy engine.
attn_status_t make_map(CUtensorMap* map, const void* ptr, int B, int H, long long L, int d) {
  if (L < 1) L = 1;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(L) * d * 2,
                           static_cast<cuuint64_t>(H) * L * d * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed (%d)",
             static_cast<int>(r));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// The fp32 dQ accumulator [B, H, L, d] as a 4-D tensor (d, L, H, B) with boxes
// of 32 fp32 (128 bytes, swizzled) by `box_rows` rows, the target of the
// backward's bulk reduce-adds (rows past L are never written).
attn_status_t make_map_f32(CUtensorMap* map, void* ptr, int B, int H, long long L, int d,
                           int box_rows) {
  if (L < 1) L = 1;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(L) * d * 4,
                           static_cast<cuuint64_t>(H) * L * d * 4};
  cuuint32_t box[4] = {32, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled (fp32) failed (%d)",
             static_cast<int>(r));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// K/V heads: 1 <= Hkv <= H and Hkv divides H (query head h reads K/V head
// h / (H / Hkv)).
bool valid_kv_heads(int H, int Hkv) { return Hkv >= 1 && Hkv <= H && H % Hkv == 0; }

attn_status_t check_common(int B, int H, long long Lq, long long Lk, int d, float scale) {
  if (B < 1 || H < 1 || Lq < 0 || Lk < 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((Lq + 127) / 128) > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn_status_t cuda_status(const char* where, cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  set_error(where, e);
  return ATTN_ERR_CUDA;
}

attn_status_t fwd_common(const void* q, const void* k, const void* v, int B, int H, int Hkv,
                         int Lq, int Lk, int d, float scale, int causal, long long q_offset,
                         long long k_offset, bool sparse, bool partial, FwdParams& p,
                         void* stream) {
  attn_status_t s = check_common(B, H, Lq, Lk, d, scale);
  if (s != ATTN_OK) return s;
  if (!valid_kv_heads(H, Hkv)) return ATTN_ERR_INVALID_ARG;
  if (q_offset < 0 || k_offset < 0) return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v)) return ATTN_ERR_INVALID_ARG;
  if (Lq == 0) return ATTN_OK;
  if ((s = get_encoder()) != ATTN_OK) return s;
  if ((s = status_word(&p.err)) != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  if ((s = make_map(&tq, q, B, H, Lq, d)) != ATTN_OK) return s;
  if ((s = make_map(&tk, k, B, Hkv, Lk, d)) != ATTN_OK) return s;
  if ((s = make_map(&tv, v, B, Hkv, Lk, d)) != ATTN_OK) return s;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.scale_log2 = scale * kLog2e;
  p.q_offset = q_offset;
  p.k_offset = k_offset;
  p.causal = causal ? 1 : 0;
  p.n_pairs = (Lq + 255) / 256;
  if (p.n_chunks <= 0) {            // no key split: one chunk holding every key
    p.n_chunks = 1;
    p.chunk_len = Lk;
  }
  if (static_cast<long long>(p.n_chunks) * B * H * p.n_pairs > 0x7FFFFFFFll) return ATTN_ERR_UNSUPPORTED;
  p.n_items = p.n_chunks * B * H * p.n_pairs;
  // Items in groups of query heads whose K and V (4 Lk d bytes per K/V head)
  // take about 64 MiB, so that the K/V tiles the running items stream stay in
  // L2 (which holds 129 MB): whole sets of the query heads that share a K/V
  // head, at least two waves of items per group on the 152 SMs, and groups of
  // nearly equal size (a small last group would start its longest items
  // late and leave a tail).  Measured: at B=2 H=16 L=16384 the DRAM reads
  // fell from 5x to 1.5x the algorithmic bytes at the same speed, and the
  // 8-chunk split of B=1 H=8 L=131072 ran 6 % faster; 32 MiB groups were
  // 6 % slower at L=16384.
  {
    const long long G = H / Hkv;
    const long long kvh = static_cast<long long>(B) * Hkv;
    const long long kv_bytes = 4ll * (Lk > 0 ? Lk : 1) * d;
    long long g_kv = (64ll << 20) / kv_bytes;
    const long long per_kv_items = static_cast<long long>(p.n_chunks) * p.n_pairs * G;
    const long long min_kv = (2ll * 152 + per_kv_items - 1) / per_kv_items;
    if (g_kv < min_kv) g_kv = min_kv;
    if (g_kv < 1) g_kv = 1;
    // a block-sparse launch reads only the listed blocks: all heads side by
    // side (grouping measured 5 % slower there)
    if (sparse) g_kv = kvh;
    long long n_groups = (kvh + g_kv / 2) / g_kv;          // nearest whole number of groups
    if (n_groups < 1) n_groups = 1;
    g_kv = (kvh + n_groups - 1) / n_groups;
    p.head_group = static_cast<int>(g_kv * G);
  }
#ifdef BSS_TRACE
  p.trace = g_trace_buf;
  p.trace_cta = g_trace_cta;
#endif
  return cuda_status("attn fwd launch",
                     launch_fwd(d, causal != 0, sparse, partial, tq, tk, tv, p,
                                static_cast<cudaStream_t>(stream)));
}

// Workspace of the block-sparse backward: the fp32 dQ accumulator, then (at a
// 256-byte boundary) the key-major bitmap of the block list.
size_t bwd_bitmap_offset(size_t acc_bytes) { return (acc_bytes + 255) & ~static_cast<size_t>(255); }
// Heads per block list: n_lists lists share the B*H heads in consecutive
// groups (1 list: every head uses it); 0 when n_lists does not divide B*H.
long long heads_per_list(int B, int H, int n_lists) {
  const long long bh = static_cast<long long>(B) * H;
  if (n_lists < 1 || bh % n_lists != 0) return 0;
  return bh / n_lists;
}

size_t bwd_bitmap_bytes(int L) {
  const size_t nblk = (static_cast<size_t>(L < 0 ? 0 : L) + 127) / 128;
  return nblk * ((nblk + 31) / 32) * 4;
}
// The block-sparse backward's CTA order (int32, one per (b, head, key tile))
// follows the bitmaps at a 256-byte boundary.
size_t bwd_order_offset(size_t bitmap_bytes) { return (bitmap_bytes + 255) & ~static_cast<size_t>(255); }

// The backward of attn_bwd and attn_bwd_blocksparse (row_ptr == nullptr: dense
// or causal); the workspace size has been checked by the caller.
attn_status_t bwd_common(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         float* delta, void* workspace, int B, int H, int Hkv, int L, int d, float scale,
                         int causal, const int32_t* row_ptr, const int32_t* col_idx, int n_lists,
                         int nnz, void* stream) {
  attn_status_t s = check_common(B, H, L, L, d, scale);
  if (s != ATTN_OK) return s;
  if (!valid_kv_heads(H, Hkv)) return ATTN_ERR_INVALID_ARG;
  const void* ptrs16[] = {q, k, v, o, dout, dq, dk, dv, workspace};
  for (const void* ptr : ptrs16)
    if (!ptr || !aligned16(ptr)) return ATTN_ERR_INVALID_ARG;
  if (!lse || !delta || !aligned4(lse) || !aligned4(delta)) return ATTN_ERR_INVALID_ARG;
  if (L == 0) return ATTN_OK;
  if ((s = get_encoder()) != ATTN_OK) return s;
  BwdParams p{};
  if ((s = status_word(&p.err)) != ATTN_OK) return s;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if ((s = make_map(&tq, q, B, H, L, d)) != ATTN_OK) return s;
  if ((s = make_map(&tk, k, B, Hkv, L, d)) != ATTN_OK) return s;
  if ((s = make_map(&tv, v, B, Hkv, L, d)) != ATTN_OK) return s;
  if ((s = make_map(&tdo, dout, B, H, L, d)) != ATTN_OK) return s;
  if ((s = make_map_f32(&tdq, workspace, B, H, L, d, bwd_dq_box_rows(d))) != ATTN_OK) return s;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.L = L;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.causal = causal ? 1 : 0;
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.delta = delta;
  p.dq_acc = static_cast<float*>(workspace);
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  // K/V heads launched together: about 2 groups run at once, each K/V head
  // holding Q, dO (bf16) and the dQ accumulator (fp32) of its H/Hkv query
  // heads, 8 L d bytes each; keep the pair of groups near 64 MiB, well inside L2.
  {
    const long long per_head = 8ll * L * d * (H / Hkv);
    long long g = (64ll << 20) / (2 * per_head);
    if (g < 1) g = 1;
    if (g > static_cast<long long>(B) * Hkv) g = static_cast<long long>(B) * Hkv;
    p.head_group = static_cast<int>(g);
  }
#ifdef BSS_TRACE
  p.trace = g_trace_buf;
  p.trace_cta = g_trace_cta;
#endif
  const bool sparse = row_ptr != nullptr;
  if (sparse) {
    const int nblk = (L + 127) / 128;
    uint32_t* bm = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) +
                                               bwd_bitmap_offset(attn_bwd_workspace_bytes(B, H, L, d)));
    p.col_bitmap = bm;
    p.col_bitmap_words = (nblk + 31) / 32;
    p.heads_per_list = static_cast<int>(heads_per_list(B, H, n_lists));
    // a K/V key tile walks the lists of all its query heads at once: they must
    // be one list (lists shared by whole groups of query heads)
    if (p.heads_per_list % (H / Hkv) != 0) return ATTN_ERR_BAD_BLOCKLIST;
    s = cuda_status("attn_bwd_blocksparse block-list transpose",
                    launch_blocklist_columns(row_ptr, col_idx, n_lists, nblk, nnz, causal, bm,
                                             p.col_bitmap_words, p.err,
                                             static_cast<cudaStream_t>(stream)));
    if (s != ATTN_OK) return s;
    // the CTA launch order (longest key-tile columns first), after the bitmaps
    int* order = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bm) +
                                        bwd_order_offset(static_cast<size_t>(n_lists) * bwd_bitmap_bytes(L)));
    p.cta_order = order;
    s = cuda_status("attn_bwd_blocksparse CTA order",
                    launch_bwd_cta_order(bm, p.col_bitmap_words, nblk, B, H, Hkv, p.heads_per_list,
                                         p.head_group, order, static_cast<cudaStream_t>(stream)));
    if (s != ATTN_OK) return s;
  }
  return cuda_status("attn_bwd launch", launch_bwd(d, sparse, tq, tk, tv, tdo, tdq, p,
                                                   static_cast<cudaStream_t>(stream),
                                                   g_bwd_main_ev[0], g_bwd_main_ev[1]));
}

// Split-KV forward: keys in chunks of a multiple of 128, each chunk's partial
// states in the workspace as acc [C, B*H*Lq, d] | m [C, B*H*Lq] | l [C, B*H*Lq]
// (each part at a 256-byte boundary).
struct SplitLayout {
  int chunk_len, chunks;
  size_t rows, acc_off, m_off, l_off, bytes;
};
SplitLayout split_layout(int B, int H, int Lq, int Lk, int d, int n_chunks) {
  SplitLayout s{};
  const long long per = (static_cast<long long>(Lk) + n_chunks - 1) / n_chunks;
  s.chunk_len = static_cast<int>(per <= 0 ? 128 : ((per + 127) / 128) * 128);
  s.chunks = Lk <= 0 ? 1 : static_cast<int>((static_cast<long long>(Lk) + s.chunk_len - 1) / s.chunk_len);
  s.rows = static_cast<size_t>(B) * H * (Lq < 0 ? 0 : Lq);
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  s.acc_off = 0;
  s.m_off = up(s.chunks * s.rows * static_cast<size_t>(d) * 4);
  s.l_off = s.m_off + up(s.chunks * s.rows * 4);
  s.bytes = s.l_off + up(s.chunks * s.rows * 4);
  return s;
}

}  // namespace

// The calling thread's error text (read by attn_last_error_message), for the
// entry points defined in other files.
void set_error_text(const char* text) { snprintf(g_last_error, sizeof(g_last_error), "%s", text); }

// the exponential-unit rate kernel (merge.cu, beside the other small kernels)
cudaError_t launch_ex2_rate(float* sink, int blocks, int iters, cudaStream_t st);

}  // namespace bss

using namespace bss;

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_BAD_BLOCKLIST: return "ATTN_ERR_BAD_BLOCKLIST";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

const char* attn_last_error_message(void) { return g_last_error; }

int attn_version(void) { return 100; }

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int H_kv, int Lq, int Lk, int d, float scale, int causal,
                       int64_t q_offset, int64_t k_offset, void* stream) {
  if (!o || !lse || !aligned16(o) || !aligned4(lse)) return ATTN_ERR_INVALID_ARG;
  FwdParams p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  return fwd_common(q, k, v, B, H, H_kv, Lq, Lk, d, scale, causal, q_offset, k_offset, false,
                    false, p, stream);
}

attn_status_t attn_fwd_partial(const void* q, const void* k, const void* v, float* m, float* l,
                               float* acc, int B, int H, int H_kv, int Lq, int Lk, int d,
                               float scale, int causal, int64_t q_offset, int64_t k_offset,
                               void* stream) {
  if (!m || !l || !acc || !aligned4(m) || !aligned4(l) || !aligned16(acc))
    return ATTN_ERR_INVALID_ARG;
  FwdParams p{};
  p.m_out = m;
  p.l_out = l;
  p.acc_out = acc;
  return fwd_common(q, k, v, B, H, H_kv, Lq, Lk, d, scale, causal, q_offset, k_offset, false,
                    true, p, stream);
}

size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int Lq, int Lk, int d, int n_chunks) {
  if (B < 1 || H < 1 || Lq < 0 || Lk < 0 || d < 1 || n_chunks < 1 || n_chunks > 64) return 0;
  return split_layout(B, H, Lq, Lk, d, n_chunks).bytes;
}

attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               void* workspace, size_t workspace_bytes, int B, int H, int H_kv,
                               int Lq, int Lk, int d, float scale, int causal, int64_t q_offset,
                               int64_t k_offset, int n_chunks, void* stream) {
  if (n_chunks < 1 || n_chunks > 64) return ATTN_ERR_INVALID_ARG;
  if (!o || !lse || !aligned16(o) || !aligned4(lse)) return ATTN_ERR_INVALID_ARG;
  attn_status_t s = check_common(B, H, Lq, Lk, d, scale);
  if (s != ATTN_OK) return s;
  const SplitLayout lay = split_layout(B, H, Lq, Lk, d, n_chunks);
  if (!workspace || !aligned16(workspace)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < lay.bytes) return ATTN_ERR_WORKSPACE;
  if (Lq == 0) return ATTN_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  FwdParams p{};
  p.acc_out = reinterpret_cast<float*>(ws + lay.acc_off);
  p.m_out = reinterpret_cast<float*>(ws + lay.m_off);
  p.l_out = reinterpret_cast<float*>(ws + lay.l_off);
  p.n_chunks = lay.chunks;
  p.chunk_len = lay.chunk_len;
  s = fwd_common(q, k, v, B, H, H_kv, Lq, Lk, d, scale, causal, q_offset, k_offset, false, true, p,
                 stream);
  if (s != ATTN_OK) return s;
  return attn_merge_states(lay.chunks, p.m_out, p.l_out, p.acc_out, o, lse, B, H, Lq, d, stream);
}

attn_status_t attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int H_kv, int L, int d, float scale,
                                   int causal,
                                   int block, const int32_t* row_ptr, const int32_t* col_idx,
                                   int n_lists, int n_qblk, int nnz, void* stream) {
  if (!o || !lse || !aligned16(o) || !aligned4(lse)) return ATTN_ERR_INVALID_ARG;
  if (block != 128) return ATTN_ERR_UNSUPPORTED;
  if (L < 0) return ATTN_ERR_INVALID_ARG;
  const long long nblk = (static_cast<long long>(L) + 127) / 128;
  if (nblk > kMaxKBlocks) return ATTN_ERR_UNSUPPORTED;
  if (n_qblk != nblk || nnz < 0) return ATTN_ERR_BAD_BLOCKLIST;
  const long long hpl = heads_per_list(B, H, n_lists);
  if (hpl == 0) return ATTN_ERR_BAD_BLOCKLIST;
  if (!row_ptr || (nnz > 0 && !col_idx) || !aligned4(row_ptr) || !aligned4(col_idx))
    return ATTN_ERR_INVALID_ARG;
  FwdParams p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.row_ptr = row_ptr;
  p.col_idx = col_idx;
  p.n_qblk = n_qblk;
  p.nnz = nnz;
  p.heads_per_list = static_cast<int>(hpl);
  return fwd_common(q, k, v, B, H, H_kv, L, L, d, scale, causal, 0, 0, true, false, p, stream);
}

attn_status_t attn_blocklist_stats(const int32_t* row_ptr, const int32_t* col_idx, int n_lists,
                                   int n_qblk, int nnz, int L, int causal, int block,
                                   int64_t* stats, void* stream) {
  if (block != 128) return ATTN_ERR_UNSUPPORTED;
  if (L < 0 || n_lists < 1) return ATTN_ERR_INVALID_ARG;
  const long long nblk = (static_cast<long long>(L) + 127) / 128;
  if (nblk > kMaxKBlocks) return ATTN_ERR_UNSUPPORTED;
  if (n_qblk != nblk || nnz < 0) return ATTN_ERR_BAD_BLOCKLIST;
  if (!row_ptr || (nnz > 0 && !col_idx) || !aligned4(row_ptr) || !aligned4(col_idx))
    return ATTN_ERR_INVALID_ARG;
  if (!stats || (reinterpret_cast<uintptr_t>(stats) & 7u) != 0) return ATTN_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (L == 0)
    return cuda_status("attn_blocklist_stats clear",
                       cudaMemsetAsync(stats, 0, static_cast<size_t>(n_lists) * 4 * sizeof(int64_t),
                                       st));
  int* err = nullptr;
  attn_status_t s = status_word(&err);
  if (s != ATTN_OK) return s;
  return cuda_status("attn_blocklist_stats launch",
                     launch_blocklist_stats(row_ptr, col_idx, n_lists, n_qblk, nnz, L,
                                            causal ? 1 : 0, reinterpret_cast<long long*>(stats),
                                            err, st));
}

attn_status_t attn_merge_states(int C, const float* m, const float* l, const float* acc, void* o,
                                float* lse, int B, int H, int L, int d, void* stream) {
  if (C < 1 || C > 64 || B < 1 || H < 1 || L < 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!m || !l || !acc || !o || !lse || !aligned16(acc) || !aligned16(o) || !aligned4(m) ||
      !aligned4(l) || !aligned4(lse))
    return ATTN_ERR_INVALID_ARG;
  int* err = nullptr;
  attn_status_t s = status_word(&err);
  if (s != ATTN_OK) return s;
  MergeParams p{};
  p.C = C;
  p.rows = static_cast<long long>(B) * H * L;
  p.m = m;
  p.l = l;
  p.acc = acc;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  return cuda_status("attn_merge_states launch",
                     launch_merge(d, p, err, static_cast<cudaStream_t>(stream)));
}

size_t attn_select_blocks_workspace_bytes(int B, int H, int L, int d) {
  if (B < 1 || H < 1 || L < 0 || d < 1) return 0;
  const size_t n = (static_cast<size_t>(L) + 127) / 128;
  const size_t pooled = static_cast<size_t>(B) * H * n * d * 4;
  return 2 * ((pooled + 255) & ~static_cast<size_t>(255));
}

int64_t attn_select_blocks_nnz(int L, int top_r, int local_blocks, int causal, int n_lists) {
  if (L < 0 || top_r < 0 || local_blocks < 0 || n_lists < 1) return -1;
  return static_cast<int64_t>(n_lists) * select_row_entries(L, top_r, local_blocks, causal ? 1 : 0);
}

attn_status_t attn_select_blocks(const void* q, const void* k, int B, int H, int H_kv, int L, int d,
                                 float scale, int causal, int block, int top_r, int local_blocks,
                                 int n_lists, int32_t* row_ptr, int32_t* col_idx, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  attn_status_t s = check_common(B, H, L, L, d, scale);
  if (s != ATTN_OK) return s;
  if (!valid_kv_heads(H, H_kv)) return ATTN_ERR_INVALID_ARG;
  if (block != 128) return ATTN_ERR_UNSUPPORTED;
  if (top_r < 0 || local_blocks < 0 || top_r + local_blocks > 256) return ATTN_ERR_INVALID_ARG;
  const long long n = (static_cast<long long>(L) + 127) / 128;
  if (n > kMaxKBlocks) return ATTN_ERR_UNSUPPORTED;
  const long long hpl = heads_per_list(B, H, n_lists);
  if (hpl == 0) return ATTN_ERR_BAD_BLOCKLIST;
  if (static_cast<long long>(n_lists) * select_row_entries(L, top_r, local_blocks, causal ? 1 : 0) >
      INT_MAX)
    return ATTN_ERR_UNSUPPORTED;   // int32 row offsets
  if (!q || !k || !aligned16(q) || !aligned16(k) || !row_ptr || !aligned4(row_ptr)) return ATTN_ERR_INVALID_ARG;
  if (!col_idx || !aligned4(col_idx) || !workspace || !aligned16(workspace)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_select_blocks_workspace_bytes(B, H, L, d)) return ATTN_ERR_WORKSPACE;
  if (L == 0) return ATTN_OK;
  const size_t pooled = static_cast<size_t>(B) * H * n * d * 4;
  const size_t pooled_up = (pooled + 255) & ~static_cast<size_t>(255);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return cuda_status("attn_select_blocks launch",
                     launch_select(d, q, k, B, H, H_kv, L, n_lists, top_r, local_blocks, causal ? 1 : 0,
                                   scale, row_ptr, col_idx, reinterpret_cast<float*>(ws),
                                   reinterpret_cast<float*>(ws + pooled_up),
                                   static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_blocklist_normalize(const int32_t* row_ptr, const int32_t* col_idx, int n_qblk,
                                       int n_kblk, int32_t* out_row_ptr, int32_t* out_col_idx,
                                       int32_t* out_nnz) {
  if (n_qblk < 0 || n_kblk < 0 || !row_ptr || !out_row_ptr || !out_nnz)
    return ATTN_ERR_INVALID_ARG;
  if (row_ptr[0] != 0) return ATTN_ERR_BAD_BLOCKLIST;
  for (int a = 0; a < n_qblk; ++a)
    if (row_ptr[a + 1] < row_ptr[a]) return ATTN_ERR_BAD_BLOCKLIST;
  const int32_t total = row_ptr[n_qblk];
  if (total > 0 && (!col_idx || !out_col_idx)) return ATTN_ERR_INVALID_ARG;
  for (int32_t e = 0; e < total; ++e)
    if (col_idx[e] < 0 || col_idx[e] >= n_kblk) return ATTN_ERR_BAD_BLOCKLIST;
  std::vector<int32_t> row;
  int32_t w = 0;
  out_row_ptr[0] = 0;
  for (int a = 0; a < n_qblk; ++a) {
    row.assign(col_idx + row_ptr[a], col_idx + row_ptr[a + 1]);
    std::sort(row.begin(), row.end());
    row.erase(std::unique(row.begin(), row.end()), row.end());
    for (int32_t c : row) out_col_idx[w++] = c;
    out_row_ptr[a + 1] = w;
  }
  *out_nnz = w;
  return ATTN_OK;
}

size_t attn_bwd_workspace_bytes(int B, int H, int L, int d) {
  if (B < 1 || H < 1 || L < 0 || d < 1) return 0;
  return static_cast<size_t>(B) * H * static_cast<size_t>(L) * d * sizeof(float);
}

size_t attn_bwd_blocksparse_workspace_bytes(int B, int H, int L, int d, int n_lists) {
  const size_t acc = attn_bwd_workspace_bytes(B, H, L, d);
  if ((acc == 0 && L != 0) || heads_per_list(B, H, n_lists) == 0) return 0;
  const size_t nblk = (static_cast<size_t>(L) + 127) / 128;
  return bwd_bitmap_offset(acc) + bwd_order_offset(static_cast<size_t>(n_lists) * bwd_bitmap_bytes(L)) +
         static_cast<size_t>(B) * H * nblk * sizeof(int32_t);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       float* delta, void* workspace, size_t workspace_bytes, int B, int H,
                       int H_kv, int L, int d, float scale, int causal, void* stream) {
  if (workspace_bytes < attn_bwd_workspace_bytes(B, H, L, d)) return ATTN_ERR_WORKSPACE;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, delta, workspace, B, H, H_kv, L, d, scale,
                    causal, nullptr, nullptr, 1, 0, stream);
}

attn_status_t attn_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o,
                                   const float* lse, const void* dout, void* dq, void* dk,
                                   void* dv, float* delta, void* workspace, size_t workspace_bytes,
                                   int B, int H, int H_kv, int L, int d, float scale, int causal,
                                   int block,
                                   const int32_t* row_ptr, const int32_t* col_idx, int n_lists,
                                   int n_qblk, int nnz, void* stream) {
  if (block != 128) return ATTN_ERR_UNSUPPORTED;
  if (L < 0) return ATTN_ERR_INVALID_ARG;
  const long long nblk = (static_cast<long long>(L) + 127) / 128;
  if (nblk > kMaxKBlocks) return ATTN_ERR_UNSUPPORTED;
  if (n_qblk != nblk || nnz < 0 || heads_per_list(B, H, n_lists) == 0) return ATTN_ERR_BAD_BLOCKLIST;
  if (!row_ptr || (nnz > 0 && !col_idx) || !aligned4(row_ptr) || !aligned4(col_idx))
    return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_blocksparse_workspace_bytes(B, H, L, d, n_lists))
    return ATTN_ERR_WORKSPACE;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, delta, workspace, B, H, H_kv, L, d, scale,
                    causal, row_ptr, col_idx, n_lists, nnz, stream);
}

attn_status_t attn_poll_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status("cudaStreamSynchronize", e);
  int* word = nullptr;
  attn_status_t s = status_word(&word);
  if (s != ATTN_OK) return s;
  int value = 0;
  e = cudaMemcpy(&value, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status("status read", e);
  if (value != 0) {
    const int zero = 0;
    e = cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_status("status reset", e);
  }
  return static_cast<attn_status_t>(value);
}

attn_status_t attn_bwd_time_main(void* begin, void* end) {
  if ((begin == nullptr) != (end == nullptr)) return ATTN_ERR_INVALID_ARG;
  g_bwd_main_ev[0] = static_cast<cudaEvent_t>(begin);
  g_bwd_main_ev[1] = static_cast<cudaEvent_t>(end);
  return ATTN_OK;
}

attn_status_t attn_probe_ex2_rate(float* sink, int blocks, int iters, void* stream) {
  if (!sink || !aligned4(sink) || blocks <= 0 || iters <= 0) return ATTN_ERR_INVALID_ARG;
  return cuda_status("ex2 rate probe launch",
                     launch_ex2_rate(sink, blocks, iters, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_watchdog_selftest(unsigned long long timeout_cycles, void* stream) {
  int* err = nullptr;
  attn_status_t s = status_word(&err);
  if (s != ATTN_OK) return s;
  return cuda_status("watchdog selftest launch",
                     launch_watchdog_selftest(timeout_cycles, err, static_cast<cudaStream_t>(stream)));
}

#ifdef BSS_TRACE
// Trace builds only: register a device buffer of kTraceRoles * kTraceEvents
// int64 for the pipeline events of CTA `cta` (linear block index) of the
// following launches; NULL switches tracing off.
void attn_trace_set(void* dev_buf, int cta) {
  g_trace_buf = static_cast<long long*>(dev_buf);
  g_trace_cta = cta;
}
#endif

}  // extern "C"
