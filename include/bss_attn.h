/*
 * bss_attn.h - C ABI of libbss_attn.so: exact, causal, block-sparse and
 * chunk-merged softmax attention on GB300 (sm_103a), forward and backward.
 *
 * Operation.  For every batch b and head h, with Q [Lq, d], K and V [Lk, d]:
 *     S = scale * Q K^T,   O = softmax_row(S over the allowed keys) V,
 *     LSE_i = ln sum_{j allowed} exp(S_ij)
 * computed tile by tile with the online-softmax state (m, l, A) so that S and
 * P never reach device memory ("Exact Blocks, Rings, and Sparsity", sections 1
 * and 2; "FlashAttention: Fast and Memory Efficient Exact Attention with IO
 * Awareness", section 5.2 and Theorem 1).
 *
 * Conventions shared by every entry point.
 *   - Tensors are contiguous row-major [B, H, L, d] (d fastest), bf16 unless
 *     stated; LSE, partial states and delta are fp32.  d must be 64 or 128.
 *   - Grouped heads: H query heads read H_kv K/V heads (1 <= H_kv <= H, H_kv
 *     divides H; H_kv = H is ordinary multi-head attention).  q, o, dout, dq,
 *     lse and delta have H heads; k, v, dk and dv have H_kv heads, and query
 *     head h reads K/V head h / (H / H_kv) ("Exact Blocks, Rings, and
 *     Sparsity", section 6: query heads that share one physical KV head).
 *     dk and dv are summed over the query heads of their group.  Otherwise
 *     ATTN_ERR_INVALID_ARG.
 *   - All pointers to tensors are DEVICE pointers, 16-byte aligned, owned by
 *     the caller.  The library never allocates, frees or synchronises device
 *     memory (attn_poll_status excepted) and keeps no pointer after a call
 *     returns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is only
 *     enqueued; results are ready when the stream reaches it.
 *   - Masks follow the pages' semantics: a masked pair contributes exactly
 *     zero; a query row with no allowed key gets O = 0 and LSE = -inf (and
 *     zero gradient); causal visibility is key + k_offset <= query + q_offset.
 *   - LSE is the natural log of the normaliser of the scaled logits.
 *   - Every call returns an attn_status_t; nothing is thrown or aborted across
 *     the ABI.  Errors found inside a kernel (a block index out of range, a
 *     watchdog timeout) are recorded in a per-library device word read by
 *     attn_poll_status.
 */
#ifndef BSS_ATTN_H_
#define BSS_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, non-finite or non-positive scale */
  ATTN_ERR_UNSUPPORTED = 2,   /* d not in {64,128}, block != 128, size beyond a stated limit */
  ATTN_ERR_BAD_BLOCKLIST = 3, /* malformed CSR: row_ptr not monotone, index out of range, nnz mismatch */
  ATTN_ERR_CUDA = 4,          /* a CUDA runtime/driver call or kernel launch failed */
  ATTN_ERR_TIMEOUT = 5,       /* a kernel's bounded wait expired (watchdog); the kernel returned early */
  ATTN_ERR_WORKSPACE = 6      /* workspace missing or smaller than attn_bwd_workspace_bytes() */
} attn_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* attn_status_string(int status);

/* Library ABI version (major*100 + minor). */
int attn_version(void);

/* Text of the last CUDA/driver failure seen by this thread (for ATTN_ERR_CUDA
 * diagnostics); empty string if none.  Static per-thread storage. */
const char* attn_last_error_message(void);

/*
 * attn_fwd - exact attention forward, dense or causal.
 * "Exact Blocks, Rings, and Sparsity", section 2 ('What the forward kernel
 * keeps on chip'); causal element mask on the diagonal tiles only, tiles wholly
 * in the future skipped (section 4, last paragraph).
 *   q [B,H,Lq,d], k/v [B,H,Lk,d] bf16 in; o [B,H,Lq,d] bf16 out; lse [B,H,Lq] fp32 out.
 *   causal != 0 applies key + k_offset <= query + q_offset (offsets >= 0).
 *   scale must be finite and > 0 (the pages use d^-1/2).
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int H_kv, int Lq, int Lk, int d, float scale, int causal,
                       int64_t q_offset, int64_t k_offset, void* stream);

/*
 * attn_fwd_partial - unnormalised online-softmax state over one KV chunk.
 * "Exact Blocks, Rings, and Sparsity", section 2 (state m, l, A and its merge
 * invariant) and section 4 (one Ring-Attention step on a KV block).
 *   Writes, per query row, m = max allowed scaled logit (natural-log units),
 *   l = sum exp(s - m), acc = sum exp(s - m) V over the keys of this chunk.
 *   Rows with no allowed key get the empty state m = -inf, l = 0; their acc
 *   row is left untouched (an empty state is identified by m = -inf and is
 *   never read by attn_merge_states).
 *   m, l: fp32 [B,H,Lq]; acc: fp32 [B,H,Lq,d].  Other arguments as attn_fwd;
 *   k_offset is the absolute position of the chunk's first key.
 */
attn_status_t attn_fwd_partial(const void* q, const void* k, const void* v,
                               float* m, float* l, float* acc,
                               int B, int H, int H_kv, int Lq, int Lk, int d, float scale,
                               int causal,
                               int64_t q_offset, int64_t k_offset, void* stream);

/*
 * attn_merge_states - combine C partial states over disjoint key sets.
 * "Exact Blocks, Rings, and Sparsity", section 4 (the associative merge of two
 * ring steps); "FlashAttention ..." section 5.1 (block-wise m and l).
 *   m, l: fp32 [C,B,H,L]; acc: fp32 [C,B,H,L,d] (as written by attn_fwd_partial,
 *   chunk-major).  Out: o bf16 [B,H,L,d] = A* / l*, lse fp32 [B,H,L] = m* + ln l*.
 *   Empty states (m = -inf) are skipped without reading their acc rows; a row
 *   whose states are all empty gets O = 0, LSE = -inf.  1 <= C <= 64.
 */
attn_status_t attn_merge_states(int C, const float* m, const float* l, const float* acc,
                                void* o, float* lse, int B, int H, int L, int d, void* stream);

/*
 * attn_fwd_splitkv_workspace_bytes - workspace of attn_fwd_splitkv: the fp32
 * partial states (m, l, acc) of every key chunk, 0 for invalid arguments.
 */
size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int Lq, int Lk, int d, int n_chunks);

/*
 * attn_fwd_splitkv - exact attention with the keys split into chunks whose
 * partial states are computed in one launch and then merged: the split-KV
 * (decode-shaped) forward.
 * "Exact Blocks, Rings, and Sparsity", section 4 (each Ring step folds one KV
 * block into the state (m, l, A); the merge is associative and order-free)
 * and section 2 (the merge invariant).
 *   Arguments and results as attn_fwd; n_chunks in [1, 64].  The keys are cut
 *   into chunks of ceil(Lk / n_chunks) keys rounded up to a multiple of 128
 *   (so there may be fewer chunks than asked), each read in place from k and
 *   v.  A chunk wholly in the causal future of a query tile is skipped for
 *   that tile (its state is empty and the merge ignores it).  Meant for
 *   shapes with few query tiles against many keys, e.g. decoding: Lq of one
 *   to a few hundred queries against a long cache, q_offset = Lk - Lq under a
 *   causal mask.
 *   workspace: device, 16-byte aligned, >= attn_fwd_splitkv_workspace_bytes
 *   bytes; contents on entry irrelevant.  Two launches on the stream: the
 *   partial states, then attn_merge_states.
 */
attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               void* workspace, size_t workspace_bytes, int B, int H, int H_kv,
                               int Lq,
                               int Lk, int d, float scale, int causal, int64_t q_offset,
                               int64_t k_offset, int n_chunks, void* stream);

/*
 * attn_blocklist_normalize - HOST function: canonical form of a CSR block list.
 * Block-sparse attention patterns page, 'Count active blocks and acknowledge the
 * changed operator' (duplicate entries never count twice; order carries no meaning).
 *   In: row_ptr[n_qblk+1], col_idx[row_ptr[n_qblk]] (host memory, any order,
 *   duplicates allowed).  Out: out_row_ptr[n_qblk+1] and out_col_idx (capacity
 *   >= row_ptr[n_qblk]) hold each row's set of key blocks in ascending order;
 *   *out_nnz = total unique entries.  Returns ATTN_ERR_BAD_BLOCKLIST if row_ptr
 *   does not start at 0, decreases, or an index is outside [0, n_kblk).
 */
attn_status_t attn_blocklist_normalize(const int32_t* row_ptr, const int32_t* col_idx,
                                       int n_qblk, int n_kblk, int32_t* out_row_ptr,
                                       int32_t* out_col_idx, int32_t* out_nnz);

/*
 * attn_fwd_blocksparse - attention over a per-query-block list of key blocks,
 * renormalised over the sparse domain.
 * "Exact Blocks, Rings, and Sparsity", section 5 ('Why the sparse unit is
 * usually a block': the outer loop visits only the listed tiles) and section 6
 * (drop-and-renormalise); block-sparse attention patterns page (triangular
 * element mask inside diagonal blocks, partial blocks, duplicates, empty rows).
 *   q/k/v/o/lse as attn_fwd with Lq = Lk = L.  block must be 128.
 *   row_ptr [n_lists][n_qblk+1], col_idx [nnz]: DEVICE int32 CSR, n_qblk =
 *   ceil(L/128), raw form accepted (any order, duplicates counted once).
 *   n_lists >= 1 lists share the B*H heads in consecutive groups: head
 *   (b*H + h) uses list (b*H + h) / (B*H / n_lists), so n_lists must divide
 *   B*H (1: one list for every head; B*H: one per head; B*H_kv with grouped
 *   query heads: one per KV head).  Each list's row_ptr holds offsets into
 *   the one col_idx array (else ATTN_ERR_BAD_BLOCKLIST).  A listed block
 *   wholly in the causal future contributes nothing (attn_blocklist_stats
 *   counts such blocks, with the list's pairs and tiles).  An entry outside
 *   [0, ceil(L/128)) is ignored and reported as ATTN_ERR_BAD_BLOCKLIST by
 *   attn_poll_status; so is a row whose row_ptr range is not inside [0, nnz]
 *   (that row is then treated as empty).  A query block with an empty list
 *   gets O = 0, LSE = -inf.  L <= 4096*128 (at most 4096 key blocks).
 *   Lists of one set (any order, any duplicates) give bit-identical results.
 *   At d = 128 with at most 2048 key blocks the launch runs the kernel with
 *   256-key score tiles, otherwise the two-tile kernel (speed only: both
 *   agree with the dense forward within rounding).
 */
attn_status_t attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int H_kv, int L, int d, float scale,
                                   int causal, int block, const int32_t* row_ptr,
                                   const int32_t* col_idx, int n_lists, int n_qblk, int nnz,
                                   void* stream);

/*
 * attn_blocklist_stats - what a block list asks the block-sparse kernels to do.
 * Block-sparse attention patterns page, 'Count active blocks and acknowledge the
 * changed operator' (report the logical allowed pairs beside the executed tile
 * work; under a causal mask the token rule applies inside every listed block,
 * so a listed block wholly in the causal future contributes nothing: it is
 * flagged here, not rejected).
 *   row_ptr, col_idx, n_lists, n_qblk, nnz, L, causal, block: as
 *   attn_fwd_blocksparse (DEVICE int32 CSR, raw form accepted, block 128).
 *   Out: stats, DEVICE int64 [n_lists][4], 8-byte aligned, per list:
 *     [0] listed (query block, key block) pairs, duplicates counted once;
 *     [1] executed tiles: listed pairs holding at least one allowed pair;
 *     [2] listed pairs wholly in the causal future (key block after query
 *         block; 0 without a causal mask), which the kernels skip;
 *     [3] logical allowed (query, key) pairs of the realised mask.
 *   [0] = [1] + [2].  Malformed rows and entries are skipped and reported as
 *   ATTN_ERR_BAD_BLOCKLIST by attn_poll_status, as in attn_fwd_blocksparse.
 *   One launch on the stream; stats is fully written (zeros when L = 0).
 */
attn_status_t attn_blocklist_stats(const int32_t* row_ptr, const int32_t* col_idx, int n_lists,
                                   int n_qblk, int nnz, int L, int causal, int block,
                                   int64_t* stats, void* stream);

/*
 * attn_select_blocks - block lists for attn_fwd_blocksparse from mean-pooled
 * scores (a selector that needs no trained weights).
 * "Exact Blocks, Rings, and Sparsity", section 5 ('Why the sparse unit is
 * usually a block': the selector must score something cheaper than Q K^T, and
 * it chooses an exact set: selected blocks united with a mandatory local
 * window; 'Fixed pooling: a cheap proxy, not the true block mass') and
 * section 6 (query heads that share a KV head share the block choice).
 *   q [B,H,L,d], k [B,H_kv,L,d] bf16 (device).  Per 128-row block the query
 *   and key rows are averaged (fp32); query block a scores key block c by the
 *   sum, over the query heads that share a list, of scale * qbar_a . kbar_c
 *   (the block pair's mean logit), query head h pooling the keys of K/V head
 *   h / (H / H_kv).  Row a keeps the local window a, a-1, .., a-local_blocks+1
 *   (those >= 0) and the top_r other candidates (under a causal mask only
 *   blocks <= a), larger score first, the lower index on equal scores, listed
 *   in ascending order.  n_lists as in attn_fwd_blocksparse.
 *   Out (device): row_ptr [n_lists][n+1] (offsets into col_idx),
 *   col_idx [attn_select_blocks_nnz(...)] int32 - the input format of
 *   attn_fwd_blocksparse and attn_bwd_blocksparse.
 *   block must be 128; top_r + local_blocks <= 256; ceil(L/128) <= 4096 and
 *   n_lists * entries per list < 2^31 (else ATTN_ERR_UNSUPPORTED).
 *   workspace: device, 16-byte aligned, >= attn_select_blocks_workspace_bytes.
 */
size_t attn_select_blocks_workspace_bytes(int B, int H, int L, int d);
int64_t attn_select_blocks_nnz(int L, int top_r, int local_blocks, int causal, int n_lists);
attn_status_t attn_select_blocks(const void* q, const void* k, int B, int H, int H_kv, int L,
                                 int d,
                                 float scale, int causal, int block, int top_r, int local_blocks,
                                 int n_lists, int32_t* row_ptr, int32_t* col_idx, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * attn_bwd_workspace_bytes - size of the caller-provided workspace of attn_bwd
 * (an fp32 dQ accumulator of B*H*L*d elements).
 */
size_t attn_bwd_workspace_bytes(int B, int H, int L, int d);

/*
 * attn_bwd - gradients by recomputation from the saved LSE.
 * "Exact Blocks, Rings, and Sparsity", section 3 (D_i = dO_i . O_i;
 * P = exp(S - LSE); dS = P o (dP - D); dQ = scale dS K; dK = scale dS^T Q;
 * dV = P^T dO; KV-owned traversal with accumulated dQ, 'The ownership
 * conflict between dQ and dK, dV'); "FlashAttention ..." section 5.3.
 *   q,k,v,o,dout bf16 [B,H,L,d]; lse fp32 [B,H,L] from attn_fwd with the same
 *   scale and mask.  Out: dq, dk, dv bf16 [B,H,L,d]; delta fp32 [B,H,L].
 *   workspace: device, >= attn_bwd_workspace_bytes(B,H,L,d) bytes, contents
 *   on entry irrelevant (it is cleared on the stream).
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       float* delta, void* workspace, size_t workspace_bytes,
                       int B, int H, int H_kv, int L, int d, float scale, int causal,
                       void* stream);

/*
 * attn_bwd_blocksparse_workspace_bytes - size of the caller-provided workspace
 * of attn_bwd_blocksparse: the fp32 dQ accumulator (B*H*L*d elements, rounded
 * up to 256 bytes), a key-major bitmap of each of the n_lists block lists
 * (ceil(L/128) columns of ceil(ceil(L/128)/32) 32-bit words, rounded up to
 * 256 bytes) and the launch order of the key tiles (B*H*ceil(L/128) int32);
 * 0 when n_lists does not divide B*H.
 */
size_t attn_bwd_blocksparse_workspace_bytes(int B, int H, int L, int d, int n_lists);

/*
 * attn_bwd_blocksparse - gradients of attn_fwd_blocksparse by recomputation.
 * "Exact Blocks, Rings, and Sparsity", section 3 (the backward of section 2
 * over the same allowed set) and section 6 (gradients flow only through the
 * kept blocks: the dropped ones have P = 0, and renormalising over the sparse
 * domain is what the saved LSE already encodes); block-sparse attention
 * patterns page (compare gradients too, duplicates counted once, empty rows).
 *   Arguments as attn_bwd plus the block list of attn_fwd_blocksparse (block
 *   128, DEVICE int32 CSR, raw form accepted) and the same causal flag; lse
 *   must come from attn_fwd_blocksparse with that list.  Each key tile walks
 *   the query blocks that list it (the list's transpose, built in the
 *   workspace on the stream, with the key tiles' launch order: columns far
 *   longer than the mean first).  A key block no query block lists gets
 *   dK = dV = 0; a query block with an empty list gets dQ = 0.  Malformed
 *   entries are handled and reported as in attn_fwd_blocksparse.  With
 *   grouped heads the query heads of one K/V head must share one list
 *   (B*H/n_lists a multiple of H/H_kv), else ATTN_ERR_BAD_BLOCKLIST.
 *   workspace: device, >= attn_bwd_blocksparse_workspace_bytes(B,H,L,d,n_lists).
 */
attn_status_t attn_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o,
                                   const float* lse, const void* dout, void* dq, void* dk,
                                   void* dv, float* delta, void* workspace, size_t workspace_bytes,
                                   int B, int H, int H_kv, int L, int d, float scale, int causal,
                                   int block,
                                   const int32_t* row_ptr, const int32_t* col_idx, int n_lists,
                                   int n_qblk, int nnz, void* stream);

/*
 * attn_bwd_noalloc - attn_bwd for callers that cannot allocate device memory.
 * The source pages have no counterpart: this entry exists for callers that
 * may not call cudaMalloc or own a workspace (an allocator that forbids new
 * device allocations, a host process that hands out none).  The fp32 dQ
 * accumulator lives in a static device array inside the library, 32 MiB
 * (8388608 floats).  Arguments and results are those of attn_bwd without the
 * workspace.
 *   - B*H*L*d above 8388608 is rejected with ATTN_ERR_WORKSPACE before any
 *     device work (attn_last_error_message says why).
 *   - The array sits in a module of its own.  Under lazy module loading (the
 *     CUDA default) the driver reserves its 32 MiB on a device during the
 *     first attn_bwd_noalloc call there, which also looks up the array's
 *     address (cudaGetSymbolAddress); the device then holds it until the
 *     process exits.  Processes that never call this entry do not hold it
 *     (unless CUDA_MODULE_LOADING=EAGER, which loads it at context creation).
 *     Make one first call per device before fixing a memory budget and before
 *     any stream capture (L = 0 with non-null, 16-byte aligned pointers does
 *     the set-up and no device work).
 *   - The cached address assumes the device's context is not reset
 *     (cudaDeviceReset) while the library is in use.
 *   - Every call shares the one array and clears it on the stream before use.
 *     Calls that can overlap on the GPU (different streams, no ordering) race
 *     on it and give wrong gradients; serialise them.
 *   - Nothing is allocated or freed by the call itself (no cudaMalloc, cudaFree
 *     or allocating library routine).
 */
attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               float* delta, int B, int H, int H_kv, int L, int d, float scale,
                               int causal,
                               void* stream);

/*
 * attn_poll_status - synchronise `stream`, then return and clear the first
 * error any kernel of this library recorded on the current device since the
 * last poll (ATTN_OK if none).
 */
attn_status_t attn_poll_status(void* stream);

/*
 * attn_bwd_time_main - measurement aid: the backward calls (attn_bwd,
 * attn_bwd_blocksparse, attn_bwd_noalloc) launch three kernels, the row
 * statistic D = rowsum(dO * O), the main kernel that recomputes the score
 * tiles and produces dK, dV and the dQ accumulator ("Exact Blocks, Rings, and
 * Sparsity", section 3), and the dQ conversion to bf16.  While `begin` and
 * `end` are set, every backward call records `begin` on its stream just
 * before the main kernel's launch and `end` just after it, so that the
 * elapsed time between them (cudaEventElapsedTime) is that kernel's own
 * duration.  `begin`, `end`: cudaEvent_t handles owned by the caller, created
 * on the device of the calls (and with timing enabled, for elapsed times).
 * Both NULL switches the recording off.  The setting is process-wide: set and
 * clear it from the thread that makes the calls.  Returns
 * ATTN_ERR_INVALID_ARG when exactly one of the two is NULL, else ATTN_OK.
 */
attn_status_t attn_bwd_time_main(void* begin, void* end);

/*
 * attn_probe_ex2_rate - measurement aid for the softmax's second ceiling:
 * the forward evaluates one exponential per pair ("FlashAttention: Fast and
 * Memory Efficient Exact Attention with IO Awareness", section 5.1, the
 * online softmax), so pairs/s cannot exceed the SMs' ex2 rate.  Launches
 * `blocks` blocks of 256 threads on `stream`; every thread evaluates
 * 8 * `iters` independent ex2.approx exponentials, blocks * 256 * 8 * iters
 * in all.  The caller times the launch.  `sink`: one device float,
 * 4-byte aligned, never written in practice (it keeps the work alive).
 * Returns ATTN_ERR_INVALID_ARG for a null sink or non-positive sizes, else
 * the launch status.
 */
attn_status_t attn_probe_ex2_rate(float* sink, int blocks, int iters, void* stream);

/*
 * attn_watchdog_selftest - launch one block that waits on a barrier nobody
 * arrives at, with a limit of `timeout_cycles` SM clock cycles; the wait gives
 * up, records ATTN_ERR_TIMEOUT and the block returns.  Lets a test observe the
 * watchdog path without hanging or faulting the GPU.  Returns the launch status.
 */
attn_status_t attn_watchdog_selftest(unsigned long long timeout_cycles, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSS_ATTN_H_ */
