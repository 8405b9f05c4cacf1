/*
 * dsa.h -- C ABI of the GB300 (sm_103a) sparse-attention decode/prefill chain:
 *          lightweight indexer -> Top-K selection -> gather-driven sparse attention.
 *
 * Method ("Day 0 Support for New LLM Architectures", Step 1 and Key Optimization 1): an indexer
 * scores every historical position of a query, the Top-K positions are selected, and a
 * sparse-attention kernel reads only those K rows of the low-rank (latent) KV cache and computes
 * exact softmax attention over them.  The score of position s for query t is
 *
 *     I[t, s] = sum_{h < H_idx} w[t, h] * ReLU( q_idx[t, h, :] . k_idx[s, :] ).
 *
 * Conventions shared by every entry point
 *  - Pointers named as device data must be device (or managed) memory visible to the current
 *    device.  The caller owns every buffer.  The library never allocates or frees device memory,
 *    never synchronises the stream, and enqueues all work on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream).
 *  - Arrays are row-major.  Strides are in BYTES unless stated otherwise.
 *  - Queries are grouped by cache: query t reads sequence  t / q_per_seq  of each cache
 *    (q_per_seq = 1 for batched decode, = T for one prefill chunk).
 *  - Visible positions of query t (n_t):  if q_pos0 < 0 (decode), n_t = n_valid[t] when n_valid
 *    is given (device int32 [T]) else L;  if q_pos0 >= 0 (causal chunk), query t sits at position
 *    q_pos0 + t % q_per_seq and n_t = q_pos0 + t % q_per_seq + 1.  n_t is clamped to [0, L].
 *  - Index rows hold positions within the query's own sequence; -1 marks an empty slot.
 *  - Validation happens before any launch; a rejected call launches nothing.  Launch failures
 *    return DSA_ERR_CUDA.  Device-side faults are never raised on purpose: kernels that meet an
 *    out-of-range index or a wait that exceeds its time limit record a code in a device error
 *    word, skip the offending access and finish; dsa_get_device_error() reads and clears it.
 *  - No C++ exception crosses this interface.  All entry points are thread-safe.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 3

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer or stride */
  DSA_ERR_UNSUPPORTED = 2, /* valid but not implemented (shape, dtype, device arch) */
  DSA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than dsa_workspace_size() */
  DSA_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute, symbol) */
  DSA_ERR_DEVICE = 5       /* a kernel recorded an error (see dsa_get_device_error) */
} dsa_status;

typedef enum dsa_dtype {
  DSA_BF16 = 0,       /* bfloat16 elements */
  DSA_FP8_E4M3 = 1,   /* E4M3 ("fn") codes with one fp32 scale per cache row (KV cache) */
  DSA_MXFP8_E4M3 = 2, /* E4M3 codes with one E8M0 exponent byte per 32 elements (indexer) */
  DSA_FP8_E4M3_T128 = 3 /* E4M3 codes with one fp32 scale per 128-element tile of a row (KV
                           cache, the 576/512 latent row: 5 scales per row, the last tile 64
                           wide); kv_scale holds ceil(D_qk / 128) floats per row */
} dsa_dtype;

/* Device error codes recorded by kernels (read with dsa_get_device_error). */
#define DSA_DEVERR_NONE 0
#define DSA_DEVERR_INDEX_RANGE 1  /* an index outside [-1, L) reached the attention gather */
#define DSA_DEVERR_WAIT_TIMEOUT 2 /* a bounded pipeline wait gave up */
#define DSA_DEVERR_TOPK_COUNTS 3  /* a row-split Top-K slot fell outside [0, K): the row's
                                     histogram disagreed with its scores; the write was skipped */

/* Human-readable name of a status code.  Never NULL. */
const char* dsa_status_string(int status);

/* DSA_ABI_VERSION of the loaded library. */
int dsa_abi_version(void);

/* Reads and clears the device error word of the current device.  Synchronises `stream` first
 * (this is the one call that blocks the host).  *code receives DSA_DEVERR_*. */
dsa_status dsa_get_device_error(int* code, void* stream);

/* Failure-path self-test (no counterpart in the method): launches one kernel whose single thread
 * waits, through the same bounded wait that every kernel of the chain uses, on a barrier that
 * nothing arrives on.  After the wait limit (about one second) the kernel records
 * DSA_DEVERR_WAIT_TIMEOUT in the device error word and returns normally, so the context stays
 * usable; dsa_get_device_error then reports (and clears) the code.  Returns DSA_OK once the kernel
 * is enqueued on `stream` (NULL = default stream). */
dsa_status dsa_selftest_wait_timeout(void* stream);

/* --------------------------------------------------------------------------------------------
 * dsa_index_score -- step 1: indexer relevance scores (per-position scoring followed by head
 * weighting, Day 0 Support for New LLM Architectures, Key Optimization 1; MXFP8 index path with
 * groups of 32 sharing one scale, Key Optimization 2).
 *
 *   scores[t * ld_scores + s] = sum_h w[t,h] * max(0, sum_j q_idx[t,h,j] * k_idx[seq(t), s, j])
 *
 * for 0 <= s < n_t (fp32, products of the stored values, fp32 accumulation).  Entries with
 * s >= n_t are left unspecified.
 *   q_idx     device [T, H_idx, d_idx]: bf16 (DSA_BF16) or E4M3 codes (DSA_MXFP8_E4M3)
 *   q_idx_sf  device [T, H_idx, d_idx/32] E8M0 bytes for DSA_MXFP8_E4M3, else NULL
 *   w         device fp32 [T, H_idx] head weights (any sign)
 *   k_idx     device: sequence q of the indexer-key cache starts at k_idx + q*k_seq_stride bytes
 *             and holds L rows of d_idx elements, rows packed (row pitch = d_idx * elem size)
 *   k_idx_sf  device, DSA_MXFP8_E4M3 only: sequence q at k_idx_sf + q*k_sf_seq_stride bytes,
 *             L rows of d_idx/32 bytes, packed; 4-byte aligned, k_sf_seq_stride a multiple
 *             of 4; else NULL
 *   scores    device fp32, row t at scores + t*ld_scores (ld_scores in ELEMENTS, >= L)
 * Supported: idx_dtype DSA_BF16 with d_idx in {64, 128}; DSA_MXFP8_E4M3 with d_idx = 128;
 * 1 <= H_idx <= 64.  q_idx, w, k_idx and scores 16-byte aligned; k_seq_stride a multiple of 16.
 * ------------------------------------------------------------------------------------------ */
dsa_status dsa_index_score(const void* q_idx, const uint8_t* q_idx_sf, const float* w,
                           const void* k_idx, const uint8_t* k_idx_sf, int64_t k_seq_stride,
                           int64_t k_sf_seq_stride, int T, int q_per_seq, int q_pos0,
                           const int32_t* n_valid, int L, int H_idx, int d_idx,
                           dsa_dtype idx_dtype, float* scores, int64_t ld_scores, void* stream);

/* --------------------------------------------------------------------------------------------
 * dsa_topk -- step 2: Top-K selection (keep the K best-scoring positions, Day 0 Support for New LLM
 * Architectures, Step 1; the Top-k selection operator of "Achieving Day-0 Readiness...",
 * section 2.1).
 *
 * For each query t: idx[t*K .. t*K+K) receives the min(K, n_t) positions s < n_t with the
 * largest scores[t*ld_scores + s], exact ties resolved toward the lower position, written in
 * ascending position order, followed by -1 in the remaining slots.  Scores are compared as
 * fp32 with -0 equal to +0; NaN scores are not supported.
 *   ws / ws_bytes  device workspace of at least dsa_topk_workspace_size(T, L, K) bytes,
 *                  zero-filled once before its first use (every completed call leaves it ready
 *                  for the next: the areas that must start at zero are zeroed again);
 *                  calls sharing a workspace must not run concurrently
 * Supported: 1 <= K <= 4096.
 * ------------------------------------------------------------------------------------------ */
dsa_status dsa_topk(const float* scores, int64_t ld_scores, int T, int q_per_seq, int q_pos0,
                    const int32_t* n_valid, int L, int K, int32_t* idx, void* ws,
                    size_t ws_bytes, void* stream);
size_t dsa_topk_workspace_size(int T, int L, int K);

/* --------------------------------------------------------------------------------------------
 * dsa_topk_noalloc -- dsa_topk for callers that cannot provide device memory.  The source pages
 * have no counterpart; this entry exists for callers such as a host framework that owns every
 * device allocation through its own pool, or a decode loop that must not allocate while it runs
 * (an allocation can synchronise the device and fragment memory).
 *
 * Same arguments, results and errors as dsa_topk, without ws / ws_bytes.  It allocates nothing:
 * its scratch is a fixed array inside the library, 16 queries x 38912 words (2.4 MB) on every
 * GPU that loads the library, held until the process exits.  T > 16 returns
 * DSA_ERR_UNSUPPORTED before any launch.
 *  - The first call on a device looks up the array's device address (once per device, with that
 *    device current); make that first call before any stream capture.  The address is kept for
 *    the life of the process: after cudaDeviceReset (or any teardown of the device's primary
 *    context) this entry must not be called again on that device.
 *  - Each call clears the part of the array it uses (an asynchronous memset on `stream`), then
 *    launches the Top-K kernel; the array keeps the last call's contents afterwards.
 *  - All calls share the one array: calls that overlap on the GPU (other streams, other threads)
 *    race and corrupt each other's results.  Serialise them on one stream.
 * ------------------------------------------------------------------------------------------ */
dsa_status dsa_topk_noalloc(const float* scores, int64_t ld_scores, int T, int q_per_seq,
                            int q_pos0, const int32_t* n_valid, int L, int K, int32_t* idx,
                            void* stream);

/* --------------------------------------------------------------------------------------------
 * dsa_sparse_attn -- step 3: gather the selected rows of the latent KV cache and compute exact
 * softmax attention over them (the sparse-attention kernel touches only the chosen cache entries
 * and computes attention over them without approximation, Day 0 Support for New LLM
 * Architectures, Step 1; gather by index then attention, "Achieving Day-0 Readiness...",
 * section 2.3; FP8 KV cache, Key Optimization 2).
 *
 * For query t, head h, with R = the valid entries (0 <= i < L) of idx[t*K .. t*K+K):
 *   logit[r] = sm_scale * sum_j q[t,h,j] * Kv[r, j]                 (j < D_qk)
 *   out[t,h,:] = sum_r softmax(logit)[r] * V[r, :D_v]               (bf16 result)
 *   lse[t,h]   = ln sum_r exp(logit[r])                             (fp32; -inf if R is empty)
 * where Kv[r] = kv row r of sequence seq(t) (times kv_scale[r] for DSA_FP8_E4M3, element j times
 * the scale of its tile j / 128 for DSA_FP8_E4M3_T128) and V[r] =
 * the first D_v columns of that same row when kv_v is NULL (latent cache), else row r of kv_v.
 * An out-of-range entry (< -1 or >= L) is skipped and recorded as DSA_DEVERR_INDEX_RANGE.
 *   q         device bf16 [T, H, D_qk]
 *   kv        device: row r of sequence q at kv + q*kv_seq_stride + r*kv_row_stride (bytes);
 *             bf16 or E4M3 codes per kv_dtype
 *   kv_v      device bf16 rows (row pitch v_row_stride, sequence pitch v_seq_stride) or NULL
 *   kv_scale  device fp32: DSA_FP8_E4M3: scale of row r of sequence q at kv_scale[q*L + r];
 *             DSA_FP8_E4M3_T128: the ceil(D_qk/128) tile scales of that row at
 *             kv_scale[(q*L + r) * ceil(D_qk/128) ...]; NULL for bf16
 *   idx       device int32 [T, K]
 *   out       device bf16 [T, H, D_v];  lse  device fp32 [T, H] or NULL
 *   ws        device workspace of at least dsa_sparse_attn_workspace_size(T, H, K, D_v)
 *             bytes, zero-filled once before its first use (the kernels leave it reusable)
 * Supported: kv_dtype DSA_BF16 or DSA_FP8_E4M3 with (D_qk, D_v) in {(576, 512), (64, 64)};
 * DSA_FP8_E4M3_T128 with (576, 512) and kv_v NULL; H <= 128; row strides multiples of 16
 * bytes; pointers 16-byte aligned.  E4M3 caches hold finite codes only (the quantisers below
 * saturate): a NaN code (0x7F / 0xFF) in a gathered row is not detected and gives unspecified
 * results (the 576/512 row widens it to a finite value).
 * ------------------------------------------------------------------------------------------ */
dsa_status dsa_sparse_attn(const void* q, const void* kv, const void* kv_v, const float* kv_scale,
                           int64_t kv_row_stride, int64_t kv_seq_stride, int64_t v_row_stride,
                           int64_t v_seq_stride, const int32_t* idx, int T, int q_per_seq, int L,
                           int K, int H, int D_qk, int D_v, float sm_scale, dsa_dtype kv_dtype,
                           void* out, float* lse, void* ws, size_t ws_bytes, void* stream);
size_t dsa_sparse_attn_workspace_size(int T, int H, int K, int D_v);

/* Which kernel computes the attention over the 576 / 512 latent row (process-wide; takes effect
 * for calls made after it returns, so do not change it while calls are in flight).
 *   DSA_ATTN_AUTO     the library's choice (warp-level mma.sync over gathered 64-row blocks, E4M3
 *                     rows widened exactly in registers); the default
 *   DSA_ATTN_TCGEN05  the tensor-memory kernel (128 rows per CTA in one swizzled bf16 tile, both
 *                     contractions on tcgen05.mma) for the entries that take it on their own
 *                     (dsa_sparse_attn, dsa_sparse_attn_partial); the fused dsa_decode / dsa_prefill
 *                     keep the library's choice
 * Other values return DSA_ERR_INVALID_ARG.  Results agree within the attention tolerance, not
 * bit for bit (the contractions add in different orders).  The workspace sizes
 * (dsa_sparse_attn_workspace_size, dsa_workspace_size) cover the kernel selected when they are
 * queried: query them after selecting. */
#define DSA_ATTN_AUTO 0
#define DSA_ATTN_TCGEN05 1
dsa_status dsa_set_attn_kernel(int kernel);

/* --------------------------------------------------------------------------------------------
 * Context split over slices: the pieces of a decode whose context is cut into G position ranges
 * (slices), each held by one device (the KV cache distributed by token with the communication
 * overlapped by compute, "Day-0 Support for Large Model Inference: From Operator Optimization to
 * Production Serving"; the index and attention steps of "Day 0 Support for New LLM
 * Architectures", Step 1, applied per slice).  Every position of the global Top-K is among the
 * Top-K of its own slice, so:
 *   1. each slice scores its positions (dsa_index_score on its rows) and emits its Top-K as
 *      (score, global position) pairs (dsa_topk_pairs);
 *   2. the G x K pairs of a query are put side by side (an all-gather across devices) and
 *      dsa_topk_merge selects the global K;
 *   3. each slice attends over the selected positions it holds (dsa_sparse_attn_partial), giving a
 *      normalised fp32 output and its log-sum-exp;
 *   4. dsa_attn_combine merges the G partial outputs (after a gather across devices).
 * The result equals the unsplit chain up to floating-point rounding of the attention; the index
 * set is the same (exact ties resolved toward the lower position in both).
 * ------------------------------------------------------------------------------------------ */

/* dsa_topk_pairs: dsa_topk over one slice (its scores, visible lengths and L are the slice's own),
 * writing for query t, slot k < K:  cand_pos[t*ld_cand + k] = the selected slice position plus
 * pos_offset (the slice's first position in the whole context), -1 in empty slots, and
 * cand_scores[t*ld_cand + k] = that position's score (0 in empty slots).  Positions come in
 * ascending order.  ld_cand >= K (so G slices can write side by side into one [T][G*K] buffer at
 * column offsets g*K).  ws / ws_bytes as for dsa_topk (dsa_topk_workspace_size(T, L, K)).
 * pos_offset >= 0 and pos_offset + L < 2^31. */
dsa_status dsa_topk_pairs(const float* scores, int64_t ld_scores, int T, int q_per_seq, int q_pos0,
                          const int32_t* n_valid, int L, int K, int pos_offset, int32_t* cand_pos,
                          float* cand_scores, int64_t ld_cand, void* ws, size_t ws_bytes, void* stream);

/* dsa_topk_merge: each query t has parts * per_part candidates; candidate j = g * per_part + k
 * (part g, entry k) sits at element offset g * part_stride + t * ld_cand + k of cand_scores (fp32)
 * and of cand_pos (int32).  So one [T][parts * per_part] buffer is ld_cand = parts * per_part,
 * part_stride = per_part, and parts gathered from devices as [parts][T][per_part] are
 * ld_cand = per_part, part_stride = T * per_part.  Among the candidates with cand_pos >= 0, the
 * min(K, count) with the largest scores, exact ties resolved toward the lower position, are
 * written to idx[t*K ..] in candidate order (j ascending), then -1.  (Parts in ascending slice
 * order, each with ascending positions as dsa_topk_pairs writes them, therefore give ascending
 * positions.)  Positions must be distinct within a query and the layout must not make two
 * candidates share an element (both layouts above satisfy this).  No workspace; one CTA per query.
 * Checked: ld_cand >= per_part when T > 1, part_stride >= per_part when parts > 1.
 * Supported: parts * per_part <= 16384, 1 <= K <= 4096. */
dsa_status dsa_topk_merge(const float* cand_scores, const int32_t* cand_pos, int T, int parts, int per_part,
                          int64_t ld_cand, int64_t part_stride, int K, int32_t* idx, void* stream);

/* dsa_sparse_attn_partial: dsa_sparse_attn for one slice whose cache holds context positions
 * [pos_lo, pos_lo + L): entries of idx in that range attend to cache row idx - pos_lo; every other
 * entry (-1, or a position held by another slice) is skipped without error.  Output, fp32:
 * o_part [T, H, D_v] = the softmax-weighted sum over this slice's attended rows (normalised over
 * them; 0 when there are none), lse_part [T, H] = their natural log-sum-exp (-inf when none).
 * Same arguments, layouts and support as dsa_sparse_attn otherwise; workspace
 * dsa_sparse_attn_workspace_size(T, H, K, D_v).  o_part 16-byte aligned, lse_part required. */
dsa_status dsa_sparse_attn_partial(const void* q, const void* kv, const void* kv_v, const float* kv_scale,
                                   int64_t kv_row_stride, int64_t kv_seq_stride, int64_t v_row_stride,
                                   int64_t v_seq_stride, const int32_t* idx, int T, int q_per_seq, int L,
                                   int K, int H, int D_qk, int D_v, float sm_scale, dsa_dtype kv_dtype,
                                   int pos_lo, float* o_part, float* lse_part, void* ws, size_t ws_bytes,
                                   void* stream);

/* dsa_attn_combine: merges G partial outputs.  Part g: o_parts + g*o_part_stride (fp32 [T, H, D_v])
 * and lse_parts + g*lse_part_stride (fp32 [T, H]); strides in elements.  With M = max_g lse_g:
 *   out[t,h,:] = sum_g e^(lse_g - M) o_g / sum_g e^(lse_g - M)   (bf16)
 *   lse[t,h]   = M + ln sum_g e^(lse_g - M)                       (fp32, or NULL)
 * Parts with lse = -inf contribute nothing; all -inf gives out = 0, lse = -inf.  D_v a multiple
 * of 4; o_parts (and o_part_stride * 4 bytes) and out 16-byte aligned. */
dsa_status dsa_attn_combine(const float* o_parts, const float* lse_parts, int G, int64_t o_part_stride,
                            int64_t lse_part_stride, int T, int H, int D_v, void* out, float* lse,
                            void* stream);

/* --------------------------------------------------------------------------------------------
 * dsa_quantize_mxfp8 / dsa_quantize_fp8_rows -- online quantisation that writes the caches the
 * chain reads ("Day 0 Support for New LLM Architectures", Key Optimization 2: the indexer stores
 * MXFP8, groups of 32 elements sharing one scale factor; the sparse-attention KV cache stores
 * FP8).  Input row r (bf16) goes to destination row dst_rows[r] of the outputs (dst_rows NULL:
 * row r; a negative entry drops the row), so appending new tokens to a cache laid out
 * [sequence][L][...] is a call with dst_rows[r] = sequence * L + position.
 *
 * dsa_quantize_mxfp8 (OCP Microscaling Formats v1.0): per group of 32 elements, amax = max |x|,
 * shared exponent e = floor(log2 amax) - 8 clamped to [-127, 127] (e = 0 for an all-zero
 * group); sf byte = e + 127; each code = E4M3(x / 2^e), round to nearest, ties to even,
 * saturating to +-448.
 *   x        device bf16, row r at x + r * x_row_stride ELEMENTS (x_row_stride >= d), 2-byte
 *            aligned; finite values
 *   codes    device E4M3 bytes, destination row q at codes + q * d
 *   sf       device E8M0 bytes, destination row q at sf + q * (d / 32)
 *   dst_rows device int64 [rows] or NULL
 * Supported: d a positive multiple of 32.
 *
 * dsa_quantize_fp8_rows: per row, s = amax / 448 (IEEE fp32 division; s = 1 for an all-zero
 * row); each code = E4M3(x / s) (IEEE fp32 division), rounded and saturated as above;
 * scales[q] = s for destination row q.
 *   codes    device E4M3 bytes, destination row q at codes + q * code_row_stride (>= width)
 *   scales   device fp32, destination row q at scales[q]
 * Both return DSA_ERR_INVALID_ARG for bad sizes or pointers before any launch; destination rows
 * must lie inside the caller's buffers (not checked).
 * ------------------------------------------------------------------------------------------ */
dsa_status dsa_quantize_mxfp8(const void* x, int64_t x_row_stride, int rows, int d, uint8_t* codes,
                              uint8_t* sf, const int64_t* dst_rows, void* stream);
dsa_status dsa_quantize_fp8_rows(const void* x, int64_t x_row_stride, int rows, int width,
                                 uint8_t* codes, int64_t code_row_stride, float* scales,
                                 const int64_t* dst_rows, void* stream);

/* dsa_quantize_fp8_tiles: dsa_quantize_fp8_rows applied to every `tile` consecutive elements of
 * a row (the last tile may be shorter; 1 <= tile <= 1024), one fp32 scale per tile: destination
 * row q's scales at scales + q * ceil(width / tile) (the page's per-token 128-element tiles for
 * DSA_FP8_E4M3_T128 caches, "Day 0 Support for New LLM Architectures", Key Optimization 2). */
dsa_status dsa_quantize_fp8_tiles(const void* x, int64_t x_row_stride, int rows, int width, int tile,
                                  uint8_t* codes, int64_t code_row_stride, float* scales,
                                  const int64_t* dst_rows, void* stream);

/* --------------------------------------------------------------------------------------------
 * Fused chain: dsa_decode / dsa_prefill run steps 1-3 back to back on `stream` (the indexer's
 * scoring, weighting and Top-K chain followed by the sparse gather kernel, Day 0 Support for New LLM
 * Architectures, Key Optimization 1), keeping the scores in the workspace.  dsa_decode expects
 * q_pos0 < 0; dsa_prefill expects q_pos0 >= 0 (a causal chunk, "Achieving Day-0 Readiness...",
 * section 2.3: prefill scores all queries in a batch) and processes the queries in slices so
 * the score scratch stays bounded.
 * ------------------------------------------------------------------------------------------ */
typedef struct dsa_args {
  /* shapes */
  int T, q_per_seq, q_pos0, L, K;
  int H_idx, d_idx;
  int H, D_qk, D_v;
  float sm_scale;
  dsa_dtype idx_dtype, kv_dtype;
  const int32_t* n_valid; /* device [T] or NULL (decode only) */
  /* indexer inputs (see dsa_index_score) */
  const void* q_idx;
  const uint8_t* q_idx_sf;
  const float* w;
  const void* k_idx;
  const uint8_t* k_idx_sf;
  int64_t k_seq_stride, k_sf_seq_stride;
  /* attention inputs (see dsa_sparse_attn) */
  const void* q;
  const void* kv;
  const void* kv_v;
  const float* kv_scale;
  int64_t kv_row_stride, kv_seq_stride, v_row_stride, v_seq_stride;
  /* outputs */
  void* out;          /* bf16 [T, H, D_v] */
  float* lse;         /* fp32 [T, H] or NULL */
  int32_t* idx_out;   /* int32 [T, K] or NULL (then kept in the workspace) */
  /* Paged caches (the pages' block-wise KV layout read through an index table, "Achieving
   * Day-0 Readiness...", section 2.2; the indexer reads the paged key cache in place, Day 0 Support for
   * New LLM Architectures, Key Optimization 1).  NULL block_table: every cache is contiguous per
   * sequence as described above.  Otherwise each cache is one pool of num_blocks * block_size
   * rows shared by all sequences: k_idx rows packed (row pitch d_idx * element size), k_idx_sf
   * rows of d_idx/32 bytes, kv / kv_v rows at kv_row_stride / v_row_stride, kv_scale one fp32
   * (DSA_FP8_E4M3_T128: ceil(D_qk/128) fp32)
   * per row; the *_seq_stride fields are ignored.  Position s of sequence q (= query t /
   * q_per_seq) lives in pool row block_table[q * max_blocks + s / block_size] * block_size +
   * s % block_size.  Entries for every position a query sees (s < n_t) must hold block ids in
   * [0, num_blocks); the others are never read. */
  const int32_t* block_table; /* device int32 [n_seq][max_blocks] or NULL */
  int block_size;             /* positions per block: a positive multiple of 64 */
  int max_blocks;             /* entries per sequence in block_table, >= ceil(L / block_size) */
  int num_blocks;             /* blocks in each pool; num_blocks * block_size < 2^31 */
} dsa_args;

/* Workspace bytes that dsa_decode (prefill = 0) or dsa_prefill (prefill = 1) needs for `a`.
 * The workspace is device memory owned by the caller.  It must be zero-filled once before its
 * first use (e.g. cudaMemsetAsync); every completed call leaves it ready for the next one.  Two
 * calls that share a workspace must not run concurrently. */
dsa_status dsa_workspace_size(const dsa_args* a, int prefill, size_t* bytes);

/* Number of kernels that one dsa_decode (prefill = 0) or dsa_prefill (prefill = 1) call with `a`
 * launches on its stream, written to *launches: per slice of queries the index score (when
 * L > 0), one Top-K kernel (or three for rows split over independent CTAs, four when the index
 * score did not supply the score histogram), the attention kernel and, when K is split over
 * CTAs, the combine kernel.  Validates `a` like dsa_workspace_size; launches nothing. */
dsa_status dsa_launch_count(const dsa_args* a, int prefill, int* launches);

dsa_status dsa_decode(const dsa_args* a, void* ws, size_t ws_bytes, void* stream);
dsa_status dsa_prefill(const dsa_args* a, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
