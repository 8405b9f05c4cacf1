// Internal declarations shared by the kernel translation units and the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "dsa_common.cuh"

namespace dsa {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch with cudaLaunchKernelEx; `pdl` lets the kernel start while the previous kernel in the
// stream finishes (the kernel then calls griddepcontrol.wait before reading its inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Paged caches: position s of sequence q lives in pool row
// table[q * max_blocks + s / block_size] * block_size + s % block_size (table null: contiguous).
struct PagedCache {
  const int32_t* table;
  int block_size, max_blocks, num_blocks;
};

__device__ __forceinline__ int64_t page_row(const PagedCache& pc, int64_t seq, int pos) {
  const int32_t b = __ldg(pc.table + seq * pc.max_blocks + pos / pc.block_size);
  return (int64_t)b * pc.block_size + pos % pc.block_size;
}

// ---------------------------------------------------------------------------------------------
// step 1: indexer scores

struct IndexScoreParams {
  const float* w;          // [T, H_idx]
  const uint8_t* q_sf;     // [T, H_idx, d/32] (MXFP8) or null
  const uint8_t* k_sf;     // sequence q at k_sf + q * k_sf_seq_stride (MXFP8) or null
  int64_t k_sf_seq_stride;
  const int32_t* n_valid;
  float* scores;
  int64_t ld_scores;
  int T, q_per_seq, q_pos0, L, H_idx;
  int t_off;               // global index of local query 0 (visibility and sequence use t + t_off)
  int tiles;               // ceil(L / 128) position tiles per query
  int* err;                // device error word
  uint32_t* hist;          // [T][4096] histograms of the top 12 key bits of the scores (added
                           // to; zero on entry), or null
  PagedCache pages;        // k_idx / k_sf pools (table null: contiguous per sequence)
  bool share_sms;          // fused chain: a short launch leaves half the resident slots free
};

constexpr int kHistBins = 4096;

// Launches the index-score kernel.  *hist_filled reports whether p.hist was filled (only the
// one-query-per-tile variants build it).
// Whether the index-score launch for these queries builds the 12-bit score histogram (the
// one-query-per-tile variants do; four-query prefill groups do not).
bool index_score_builds_hist(int T, int H_idx, int q_per_seq, bool mx);

cudaError_t launch_index_score(const void* q_idx, const void* k_idx, int64_t k_seq_stride,
                               int n_seq, int d_idx, bool mx, IndexScoreParams p,
                               cudaStream_t stream, bool pdl, bool* hist_filled);

// ---------------------------------------------------------------------------------------------
// step 2: Top-K

struct TopkParams {
  const float* scores;
  int64_t ld_scores;
  const int32_t* n_valid;
  int32_t* idx;
  int64_t idx_ld;          // elements between index rows (0: K)
  int T, q_per_seq, q_pos0, L, K;
  int t_off;               // global index of local query 0
  int* err;                // device error word
  uint32_t* hist;          // [T][4096] top-12-bit histograms from the index-score kernel, or
                           // null (then built here); zeroed after use
  uint32_t* work;          // per-query exchange areas (set by launch_topk from its workspace)
  int wide_chunk, wide_nch;  // row-split path: positions per CTA and CTAs per row (launch_topk)
  // Optional L2 prefetch of the selected rows of the attention cache (null kv: none), issued as
  // each selected position is written.
  const uint8_t* kv;
  int64_t kv_row_stride, kv_seq_stride;
  int kv_bytes;            // bytes of a row to prefetch (a multiple of 16)
  const uint8_t* kv_v;     // separate V rows, or null
  int64_t v_row_stride, v_seq_stride;
  int v_bytes;
  PagedCache pages;        // kv / kv_v pools for the prefetch (table null: contiguous)
};

// allow_wide: long rows may be split over independent CTAs (workspace from topk_ws_bytes);
// otherwise one cluster per query (workspace from topk_cluster_ws_bytes).
cudaError_t launch_topk(const TopkParams& p, void* ws, cudaStream_t stream, bool pdl,
                        bool allow_wide = true);
size_t topk_cluster_ws_bytes(int T, int L);
int topk_launches(int T, int L, bool hist_supplied);
size_t topk_ws_bytes(int T, int L, int K);

// Context split over slices: a slice's Top-K as (score, global position) pairs, and the merge of
// the pairs of all slices into the global Top-K.
struct PairsParams {
  const float* scores;     // the slice's scores [T][ld_scores]
  int64_t ld_scores;
  int32_t* cand_pos;       // [T][ld_cand]: local positions from the slice's Top-K -> global
  float* cand_scores;      // [T][ld_cand]
  int64_t ld_cand;
  int T, K, pos_offset;
};
struct MergeParams {
  const float* scores;     // candidate j = g * per_part + k of query t at g * part_stride + t * ld + k
  const int32_t* pos;      // same layout; < 0: no candidate
  int64_t ld, part_stride; // in elements
  int T, parts, per_part, K;
  int32_t* idx;            // [T][K]
};
// p.idx = cand_pos with p.idx_ld = ld_cand; the Top-K, then the pairs kernel (PDL)
cudaError_t launch_topk_pairs(const TopkParams& p, void* ws, const PairsParams& pp, cudaStream_t stream);
cudaError_t launch_topk_merge(const MergeParams& p, cudaStream_t stream, bool pdl);
int topk_merge_max_candidates();

// ---------------------------------------------------------------------------------------------
// step 3: sparse attention

struct SparseAttnParams {
  const __nv_bfloat16* q;  // [T, H, D_qk]
  const uint8_t* kv;
  const uint8_t* kv_v;
  const float* kv_scale;
  int64_t kv_row_stride, kv_seq_stride, v_row_stride, v_seq_stride;
  const int32_t* idx;      // [T, K]
  int T, q_per_seq, L, K, H;
  int t_off;               // global index of local query 0 (selects the sequence)
  float scale_log2;        // sm_scale * log2(e)
  __nv_bfloat16* out;      // [T, H, D_v]
  float* lse;              // [T, H] or null
  float* part_o;           // [T, H, splits, D_v] when splits > 1
  float* part_ml;          // [T, H, splits, 2]
  int splits;
  int rows_per_split;
  int* err;                // device error word
  // Set by the fused chain, whose index rows hold the min(K, n_t) selected positions first and
  // -1 after them: a split then stops at the query's last valid row (q_pos0 / n_valid give n_t).
  // It also selects the chain's choice of attention kernel.
  bool valid_prefix;
  int q_pos0;
  const int32_t* n_valid;
  PagedCache pages;        // kv / kv_v / kv_scale pools (table null: contiguous per sequence)
  // Context slice (slice_rows): the cache holds positions [pos_lo, pos_lo + L) of a longer
  // context; index entries outside that range belong to other slices and are skipped without an
  // error, the others address row idx - pos_lo.
  bool slice_rows;
  int pos_lo;
  float* out_f32;          // when set: fp32 [T, H, D_v] output instead of the bf16 `out`
};

// Combine of G context slices' partial outputs (o_g normalised fp32, lse_g natural log).
struct SliceCombineParams {
  const float* o_parts;    // part g at o_parts + g * o_stride: [T, H, D_v]
  const float* lse_parts;  // part g at lse_parts + g * lse_stride: [T, H]
  int64_t o_stride, lse_stride;  // in elements
  int G, T, H, D_v;
  __nv_bfloat16* out;      // [T, H, D_v]
  float* lse;              // [T, H] or null
};
cudaError_t launch_slice_combine(const SliceCombineParams& p, cudaStream_t stream, bool pdl);

int sparse_attn_splits(int T, int H, int K, bool chain);
bool set_attn_kernel(int kernel);  // false for an unknown kernel id
// kernels one attention step launches (the attention, plus the combine when K is split over CTAs);
// chain: inside the fused chain (whose index rows hold each query's valid positions first)
int sparse_attn_launches(int T, int H, int K, int D_qk, int D_v, bool fp8, bool sepv, bool tiled, bool chain);
size_t sparse_attn_ws_bytes(int T, int H, int K, int D_v);
// tiled: FP8 rows with one scale per 128-element tile (kv_scale [rows][ceil(D_qk / 128)])
cudaError_t launch_sparse_attn(SparseAttnParams p, int D_qk, int D_v, bool fp8, bool sepv,
                               void* ws, cudaStream_t stream, bool pdl, bool tiled);

// Argument checks and device facts shared with entry points defined outside dsa_api.cu.
dsa_status check_topk_args(const float* scores, int64_t ld_scores, int T, int q_per_seq, int q_pos0,
                           const int32_t* n_valid, int L, int K, const int32_t* idx);
dsa_status check_device_arch();
int* device_error_word();

// Driver entry point for tensor-map encoding (resolved once through the runtime).
CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank,
                           void* addr, const cuuint64_t* dims, const cuuint64_t* strides,
                           const cuuint32_t* box, CUtensorMapSwizzle swizzle);

}  // namespace dsa
