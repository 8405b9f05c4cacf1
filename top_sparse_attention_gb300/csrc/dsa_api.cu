// C ABI of the sparse-attention chain (see include/dsa.h): argument validation, workspace
// layout and launch sequencing on the caller's stream.  Nothing here allocates device memory or
// synchronises, except dsa_get_device_error, which reads the device error word.
#include <cudaTypedefs.h>

#include <mutex>

#include "dsa_internal.h"

namespace dsa {

__device__ int g_device_error = 0;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// Device address of g_device_error on the current device (resolved once per device).
int* device_error_ptr() {
  static std::mutex mu;
  static int* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) ptrs[dev] = reinterpret_cast<int*>(p);
  }
  return ptrs[dev];
}

// The kernels are built for sm_103a only; other devices are rejected before any launch.
dsa_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dsa_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DSA_OK;
  if (e == cudaErrorNotSupported) return DSA_ERR_UNSUPPORTED;
  return DSA_ERR_CUDA;
}

int64_t ld_for(int L) { return (int64_t)align_up((size_t)(L > 0 ? L : 1), 4); }

// ------------------------------------------------------------------------------------------
// validation of each step's arguments (returns DSA_OK or the reason)

dsa_status check_visibility(int T, int q_per_seq, int q_pos0, const int32_t* n_valid, int L) {
  if (T < 0 || L < 0 || q_per_seq < 1) return DSA_ERR_INVALID_ARG;
  if (T % q_per_seq != 0) return DSA_ERR_INVALID_ARG;
  if (q_pos0 >= 0 && n_valid) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status check_index_score(const void* q_idx, const uint8_t* q_idx_sf, const float* w,
                             const void* k_idx, const uint8_t* k_idx_sf, int64_t k_seq_stride,
                             int64_t k_sf_seq_stride, int T, int q_per_seq, int q_pos0,
                             const int32_t* n_valid, int L, int H_idx, int d_idx,
                             dsa_dtype idx_dtype, const float* scores, int64_t ld_scores) {
  dsa_status s = check_visibility(T, q_per_seq, q_pos0, n_valid, L);
  if (s != DSA_OK) return s;
  if (idx_dtype != DSA_BF16 && idx_dtype != DSA_MXFP8_E4M3) return DSA_ERR_UNSUPPORTED;
  if (H_idx < 1 || H_idx > 64) return H_idx < 1 ? DSA_ERR_INVALID_ARG : DSA_ERR_UNSUPPORTED;
  if (idx_dtype == DSA_BF16 && d_idx != 64 && d_idx != 128) return DSA_ERR_UNSUPPORTED;
  if (idx_dtype == DSA_MXFP8_E4M3 && d_idx != 128) return DSA_ERR_UNSUPPORTED;
  if (T == 0 || L == 0) return DSA_OK;
  if (!q_idx || !w || !k_idx || !scores) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(scores))
    return DSA_ERR_INVALID_ARG;
  if (ld_scores < L || ld_scores % 4 != 0) return DSA_ERR_INVALID_ARG;
  const int n_seq = T / q_per_seq;
  const int64_t row_bytes = (int64_t)d_idx * (idx_dtype == DSA_BF16 ? 2 : 1);
  if (n_seq > 1 && (k_seq_stride % 16 != 0 || k_seq_stride < (int64_t)L * row_bytes))
    return DSA_ERR_INVALID_ARG;
  if (idx_dtype == DSA_MXFP8_E4M3) {
    // the scale rows are read with 4-byte loads (4 groups of 32 per row)
    if (!q_idx_sf || !k_idx_sf || (reinterpret_cast<uintptr_t>(k_idx_sf) & 3u) != 0) return DSA_ERR_INVALID_ARG;
    if (n_seq > 1 && (k_sf_seq_stride % 4 != 0 || k_sf_seq_stride < (int64_t)L * (d_idx / 32)))
      return DSA_ERR_INVALID_ARG;
  }
  return DSA_OK;
}

dsa_status check_topk(const float* scores, int64_t ld_scores, int T, int q_per_seq, int q_pos0,
                      const int32_t* n_valid, int L, int K, const int32_t* idx) {
  dsa_status s = check_visibility(T, q_per_seq, q_pos0, n_valid, L);
  if (s != DSA_OK) return s;
  if (K < 1) return DSA_ERR_INVALID_ARG;
  if (K > 4096) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!idx) return DSA_ERR_INVALID_ARG;
  if (L > 0 && (!scores || ld_scores < L)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status check_sparse_attn(const void* q, const void* kv, const void* kv_v, const float* kv_scale,
                             int64_t kv_row_stride, int64_t kv_seq_stride, int64_t v_row_stride,
                             int64_t v_seq_stride, const int32_t* idx, int T, int q_per_seq, int L,
                             int K, int H, int D_qk, int D_v, dsa_dtype kv_dtype, const void* out) {
  if (T < 0 || L < 0 || q_per_seq < 1 || T % q_per_seq != 0 || K < 1 || H < 1)
    return DSA_ERR_INVALID_ARG;
  if (kv_dtype != DSA_BF16 && kv_dtype != DSA_FP8_E4M3 && kv_dtype != DSA_FP8_E4M3_T128)
    return DSA_ERR_UNSUPPORTED;
  const bool mla = D_qk == 576 && D_v == 512 && !kv_v;
  const bool small = D_qk == 64 && D_v == 64 && !(kv_v && kv_dtype != DSA_BF16);
  if (!mla && !small) return DSA_ERR_UNSUPPORTED;
  if (H > 128 || K > 4096) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!q || !kv || !idx || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  const int64_t elem = kv_dtype == DSA_BF16 ? 2 : 1;
  if (kv_row_stride % 16 != 0 || kv_row_stride < D_qk * elem) return DSA_ERR_INVALID_ARG;
  if (T / q_per_seq > 1 && (kv_seq_stride % 16 != 0 || kv_seq_stride < (int64_t)L * kv_row_stride))
    return DSA_ERR_INVALID_ARG;
  if (kv_dtype != DSA_BF16 && !kv_scale) return DSA_ERR_INVALID_ARG;
  if (kv_dtype == DSA_FP8_E4M3_T128 && !mla) return DSA_ERR_UNSUPPORTED;
  if (kv_v) {
    if (!aligned16(kv_v) || v_row_stride % 16 != 0 || v_row_stride < D_v * 2) return DSA_ERR_INVALID_ARG;
    if (T / q_per_seq > 1 && (v_seq_stride % 16 != 0 || v_seq_stride < (int64_t)L * v_row_stride))
      return DSA_ERR_INVALID_ARG;
  }
  return DSA_OK;
}

// ------------------------------------------------------------------------------------------
// launches of the three steps for queries [t_off, t_off + T)

PagedCache pages_of(const dsa_args& a) {
  PagedCache pc = {};
  if (a.block_table) {
    pc.table = a.block_table;
    pc.block_size = a.block_size;
    pc.max_blocks = a.max_blocks;
    pc.num_blocks = a.num_blocks;
  }
  return pc;
}

cudaError_t run_index_score(const dsa_args& a, int t_off, int T, float* scores, int64_t ld,
                            uint32_t* hist, bool* hist_filled, cudaStream_t st, bool pdl,
                            bool share_sms = false) {
  const int64_t row_bytes = (int64_t)a.d_idx * (a.idx_dtype == DSA_BF16 ? 2 : 1);
  IndexScoreParams p = {};
  p.w = a.w + (int64_t)t_off * a.H_idx;
  p.q_sf = a.q_idx_sf ? a.q_idx_sf + (int64_t)t_off * a.H_idx * (a.d_idx / 32) : nullptr;
  p.k_sf = a.k_idx_sf;
  p.k_sf_seq_stride = a.k_sf_seq_stride;
  p.n_valid = a.n_valid;
  p.scores = scores;
  p.ld_scores = ld;
  p.T = T;
  p.q_per_seq = a.q_per_seq;
  p.q_pos0 = a.q_pos0;
  p.L = a.L;
  p.H_idx = a.H_idx;
  p.t_off = t_off;
  p.tiles = (a.L + 127) / 128;
  p.err = device_error_ptr();
  p.hist = hist;
  p.pages = pages_of(a);
  p.share_sms = share_sms;
  const uint8_t* qi = reinterpret_cast<const uint8_t*>(a.q_idx) + (int64_t)t_off * a.H_idx * row_bytes;
  return launch_index_score(qi, a.k_idx, a.k_seq_stride, a.T / a.q_per_seq, a.d_idx,
                            a.idx_dtype == DSA_MXFP8_E4M3, p, st, pdl, hist_filled);
}

// 1: the chain's Top-K issues an L2 prefetch of every selected cache row as it writes the position.
// Off: since the Top-K lets the attention kernel launch at its output pass, the prefetch requests
// (one bulk prefetch per row) cost the Top-K more than they save the gather (B = 8, L = 32K, six
// batches in flight: bf16 18.1 -> 17.2 us per step, MXFP8 17.2 -> 16.8 us; one batch at a time
// 41.2 -> 40.4 us and 44.4 -> 43.3 us; L = 1M and varying lengths gained as well).
#ifndef DSA_TOPK_KV_PREFETCH
#define DSA_TOPK_KV_PREFETCH 0
#endif
cudaError_t run_topk(const dsa_args& a, int t_off, int T, const float* scores, int64_t ld,
                     int32_t* idx, uint32_t* hist, void* ws, cudaStream_t st, bool pdl) {
  TopkParams p = {};
  p.scores = scores;
  p.ld_scores = ld;
  p.n_valid = a.n_valid;
  p.idx = idx;
  p.T = T;
  p.q_per_seq = a.q_per_seq;
  p.q_pos0 = a.q_pos0;
  p.L = a.L;
  p.K = a.K;
  p.t_off = t_off;
  p.err = device_error_ptr();
  p.hist = hist;
  // the selected cache rows can be prefetched into L2 for the attention step (DSA_TOPK_KV_PREFETCH)
  p.kv = DSA_TOPK_KV_PREFETCH ? reinterpret_cast<const uint8_t*>(a.kv) : nullptr;
  p.kv_row_stride = a.kv_row_stride;
  p.kv_seq_stride = a.kv_seq_stride;
  p.kv_bytes = a.D_qk * (a.kv_dtype == DSA_BF16 ? 2 : 1);  // (E4M3 rows: one byte per element)
  p.kv_v = reinterpret_cast<const uint8_t*>(a.kv_v);
  p.v_row_stride = a.v_row_stride;
  p.v_seq_stride = a.v_seq_stride;
  p.v_bytes = a.D_v * 2;
  p.pages = pages_of(a);
  return launch_topk(p, ws, st, pdl);
}

// valid_prefix: idx rows hold each query's min(K, n_t) selected positions first and -1 after
// them (the chain's own Top-K output), so the attention may stop at the last valid row.
cudaError_t run_sparse_attn(const dsa_args& a, int t_off, int T, const int32_t* idx, void* ws,
                            cudaStream_t st, bool pdl, bool valid_prefix, int slice_pos_lo = -1,
                            float* out_f32 = nullptr) {
  SparseAttnParams p = {};
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q) + (int64_t)t_off * a.H * a.D_qk;
  p.kv = reinterpret_cast<const uint8_t*>(a.kv);
  p.kv_v = reinterpret_cast<const uint8_t*>(a.kv_v);
  p.kv_scale = a.kv_scale;
  p.kv_row_stride = a.kv_row_stride;
  p.kv_seq_stride = a.kv_seq_stride;
  p.v_row_stride = a.v_row_stride;
  p.v_seq_stride = a.v_seq_stride;
  p.idx = idx;
  p.T = T;
  p.q_per_seq = a.q_per_seq;
  p.L = a.L;
  p.K = a.K;
  p.H = a.H;
  p.t_off = t_off;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out) + (int64_t)t_off * a.H * a.D_v;
  p.lse = a.lse ? a.lse + (int64_t)t_off * a.H : nullptr;
  p.err = device_error_ptr();
  p.valid_prefix = valid_prefix;
  p.q_pos0 = a.q_pos0;
  p.n_valid = a.n_valid;
  p.pages = pages_of(a);
  p.slice_rows = slice_pos_lo >= 0;
  p.pos_lo = slice_pos_lo;
  p.out_f32 = out_f32;
  return launch_sparse_attn(p, a.D_qk, a.D_v, a.kv_dtype != DSA_BF16, a.kv_v != nullptr, ws, st, pdl,
                            a.kv_dtype == DSA_FP8_E4M3_T128);
}

// ------------------------------------------------------------------------------------------
// fused chain: workspace = [scores (Tc x ld fp32)] [idx (T x K int32) unless idx_out]
//                          [score histograms (Tc x 4096 u32)] [Top-K level histograms]
//                          [attention partials]; the histogram regions are zero between calls

constexpr size_t kPrefillScoreBudget = 256ull << 20;  // score scratch per prefill slice

int slice_queries(const dsa_args& a, int prefill) {
  if (!prefill) return a.T;
  const size_t row = (size_t)ld_for(a.L) * sizeof(float);
  int tc = (int)(kPrefillScoreBudget / row);
  tc = tc < 4 ? 4 : (tc / 4) * 4;
  return tc < a.T ? tc : a.T;
}

struct Layout {
  size_t scores, idx, hist, topk, attn, total;
  int tc;
};

Layout layout_of(const dsa_args& a, int prefill) {
  Layout l = {};
  l.tc = slice_queries(a, prefill);
  size_t off = 0;
  l.scores = off;
  off += align_up((size_t)l.tc * ld_for(a.L) * sizeof(float), 256);
  l.idx = off;
  if (!a.idx_out) off += align_up((size_t)a.T * a.K * sizeof(int32_t), 256);
  l.hist = off;
  off += align_up((size_t)l.tc * kHistBins * sizeof(uint32_t), 256);
  l.topk = off;
  off += align_up(topk_ws_bytes(l.tc, a.L, a.K), 256);
  l.attn = off;
  off += align_up(sparse_attn_ws_bytes(l.tc, a.H, a.K, a.D_v), 256);
  l.total = off;
  return l;
}

dsa_status check_args(const dsa_args* a, int prefill) {
  if (!a) return DSA_ERR_INVALID_ARG;
  if (a->block_table) {
    if (a->block_size <= 0 || a->block_size % 64 != 0 || a->num_blocks <= 0) return DSA_ERR_INVALID_ARG;
    if ((int64_t)a->max_blocks * a->block_size < a->L) return DSA_ERR_INVALID_ARG;
    if ((int64_t)a->num_blocks * a->block_size >= (1ll << 31)) return DSA_ERR_UNSUPPORTED;
  }
  if (prefill ? a->q_pos0 < 0 : a->q_pos0 >= 0) return DSA_ERR_INVALID_ARG;
  // pools have no per-sequence pitch: the checks below see the pitch of a contiguous layout
  const int64_t L = a->L;
  const int64_t k_seq = a->block_table ? (L * a->d_idx * (a->idx_dtype == DSA_BF16 ? 2 : 1) + 15) / 16 * 16
                                       : a->k_seq_stride;
  const int64_t k_sf_seq = a->block_table ? (L * (a->d_idx / 32) + 3) / 4 * 4 : a->k_sf_seq_stride;
  const int64_t kv_seq = a->block_table ? L * a->kv_row_stride : a->kv_seq_stride;
  const int64_t v_seq = a->block_table ? L * a->v_row_stride : a->v_seq_stride;
  dsa_status s = check_index_score(a->q_idx, a->q_idx_sf, a->w, a->k_idx, a->k_idx_sf,
                                   k_seq, k_sf_seq, a->T, a->q_per_seq,
                                   a->q_pos0, a->n_valid, a->L, a->H_idx, a->d_idx, a->idx_dtype,
                                   reinterpret_cast<const float*>(16), ld_for(a->L));
  if (s != DSA_OK) return s;
  s = check_topk(reinterpret_cast<const float*>(16), ld_for(a->L), a->T, a->q_per_seq, a->q_pos0,
                 a->n_valid, a->L, a->K, reinterpret_cast<const int32_t*>(16));
  if (s != DSA_OK) return s;
  return check_sparse_attn(a->q, a->kv, a->kv_v, a->kv_scale, a->kv_row_stride, kv_seq,
                           a->v_row_stride, v_seq, reinterpret_cast<const int32_t*>(16),
                           a->T, a->q_per_seq, a->L, a->K, a->H, a->D_qk, a->D_v, a->kv_dtype,
                           a->out);
}

dsa_status run_chain(const dsa_args* a, void* ws, size_t ws_bytes, void* stream, int prefill) {
  dsa_status s = check_args(a, prefill);
  if (s != DSA_OK) return s;
  if (a->T == 0) return DSA_OK;
  const Layout l = layout_of(*a, prefill);
  if (!ws || ws_bytes < l.total || !aligned16(ws)) return DSA_ERR_WORKSPACE;
  if ((s = check_device()) != DSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  float* scores = reinterpret_cast<float*>(base + l.scores);
  int32_t* idx = a->idx_out ? a->idx_out : reinterpret_cast<int32_t*>(base + l.idx);
  const int64_t ld = ld_for(a->L);
  for (int t0 = 0; t0 < a->T; t0 += l.tc) {
    const int tn = (a->T - t0) < l.tc ? (a->T - t0) : l.tc;
    int32_t* idx_slice = idx + (int64_t)t0 * a->K;
    uint32_t* hist = reinterpret_cast<uint32_t*>(base + l.hist);
    cudaError_t e = cudaSuccess;
    bool filled = false;
    // every launch may overlap its predecessor's tail (programmatic dependent launch); each
    // kernel waits for its predecessor before reading anything that predecessor could write
    if (a->L > 0) e = run_index_score(*a, t0, tn, scores, ld, hist, &filled, st, true, /*share_sms=*/true);
    if (e == cudaSuccess)
      e = run_topk(*a, t0, tn, scores, ld, idx_slice, filled ? hist : nullptr, base + l.topk, st, true);
    if (e == cudaSuccess)
      e = run_sparse_attn(*a, t0, tn, idx_slice, base + l.attn, st, true, /*valid_prefix=*/true);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return DSA_OK;
}

// Failure-path self-test: one thread waits, through the same bounded wait every kernel of the
// chain uses, on an mbarrier that nothing arrives on.  The wait gives up after its limit, records
// DSA_DEVERR_WAIT_TIMEOUT and the kernel returns normally.
__global__ void selftest_wait_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, err);
  }
}

}  // namespace

dsa_status check_topk_args(const float* scores, int64_t ld_scores, int T, int q_per_seq, int q_pos0,
                           const int32_t* n_valid, int L, int K, const int32_t* idx) {
  return check_topk(scores, ld_scores, T, q_per_seq, q_pos0, n_valid, L, K, idx);
}

dsa_status check_device_arch() { return check_device(); }

int* device_error_word() { return device_error_ptr(); }

CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank, void* addr,
                           const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                           CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return CUDA_ERROR_NOT_FOUND;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return g_encode(map, dtype, rank, addr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: invalid argument";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: shape, dtype or device not supported";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace missing or too small";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: a CUDA runtime call failed";
    case DSA_ERR_DEVICE: return "DSA_ERR_DEVICE: a kernel recorded an error";
    default: return "unknown dsa_status";
  }
}

int dsa_abi_version(void) { return DSA_ABI_VERSION; }

dsa_status dsa_get_device_error(int* code, void* stream) {
  if (!code) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return DSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  *code = v;
  return DSA_OK;
}

dsa_status dsa_selftest_wait_timeout(void* stream) {
  dsa_status s = check_device();
  if (s != DSA_OK) return s;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(device_error_ptr());
  return from_cuda(cudaGetLastError());
}

dsa_status dsa_index_score(const void* q_idx, const uint8_t* q_idx_sf, const float* w,
                           const void* k_idx, const uint8_t* k_idx_sf, int64_t k_seq_stride,
                           int64_t k_sf_seq_stride, int T, int q_per_seq, int q_pos0,
                           const int32_t* n_valid, int L, int H_idx, int d_idx,
                           dsa_dtype idx_dtype, float* scores, int64_t ld_scores, void* stream) {
  dsa_status s = check_index_score(q_idx, q_idx_sf, w, k_idx, k_idx_sf, k_seq_stride, k_sf_seq_stride,
                                   T, q_per_seq, q_pos0, n_valid, L, H_idx, d_idx, idx_dtype, scores,
                                   ld_scores);
  if (s != DSA_OK || T == 0 || L == 0) return s;
  if ((s = check_device()) != DSA_OK) return s;
  dsa_args a = {};
  a.T = T;
  a.q_per_seq = q_per_seq;
  a.q_pos0 = q_pos0;
  a.L = L;
  a.H_idx = H_idx;
  a.d_idx = d_idx;
  a.idx_dtype = idx_dtype;
  a.n_valid = n_valid;
  a.q_idx = q_idx;
  a.q_idx_sf = q_idx_sf;
  a.w = w;
  a.k_idx = k_idx;
  a.k_idx_sf = k_idx_sf;
  a.k_seq_stride = k_seq_stride;
  a.k_sf_seq_stride = k_sf_seq_stride;
  return from_cuda(run_index_score(a, 0, T, scores, ld_scores, nullptr, nullptr,
                                   reinterpret_cast<cudaStream_t>(stream), false));
}

size_t dsa_topk_workspace_size(int T, int L, int K) { return topk_ws_bytes(T, L, K); }

dsa_status dsa_topk(const float* scores, int64_t ld_scores, int T, int q_per_seq, int q_pos0,
                    const int32_t* n_valid, int L, int K, int32_t* idx, void* ws, size_t ws_bytes,
                    void* stream) {
  dsa_status s = check_topk(scores, ld_scores, T, q_per_seq, q_pos0, n_valid, L, K, idx);
  if (s != DSA_OK || T == 0) return s;
  if (!ws || ws_bytes < topk_ws_bytes(T, L, K) || !aligned16(ws)) return DSA_ERR_WORKSPACE;
  if ((s = check_device()) != DSA_OK) return s;
  dsa_args a = {};
  a.T = T;
  a.q_per_seq = q_per_seq;
  a.q_pos0 = q_pos0;
  a.n_valid = n_valid;
  a.L = L;
  a.K = K;
  return from_cuda(run_topk(a, 0, T, scores, ld_scores, idx, nullptr, ws, reinterpret_cast<cudaStream_t>(stream), false));
}

dsa_status dsa_topk_pairs(const float* scores, int64_t ld_scores, int T, int q_per_seq, int q_pos0,
                          const int32_t* n_valid, int L, int K, int pos_offset, int32_t* cand_pos,
                          float* cand_scores, int64_t ld_cand, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = check_topk(scores, ld_scores, T, q_per_seq, q_pos0, n_valid, L, K, cand_pos);
  if (s != DSA_OK || T == 0) return s;
  if (!cand_scores || ld_cand < K || pos_offset < 0 || (int64_t)pos_offset + L > INT32_MAX)
    return DSA_ERR_INVALID_ARG;
  if (!ws || ws_bytes < topk_ws_bytes(T, L, K) || !aligned16(ws)) return DSA_ERR_WORKSPACE;
  if ((s = check_device()) != DSA_OK) return s;
  TopkParams p = {};
  p.scores = scores;
  p.ld_scores = ld_scores;
  p.n_valid = n_valid;
  p.idx = cand_pos;
  p.idx_ld = ld_cand;
  p.T = T;
  p.q_per_seq = q_per_seq;
  p.q_pos0 = q_pos0;
  p.L = L;
  p.K = K;
  p.err = device_error_ptr();
  PairsParams pp = {};
  pp.scores = scores;
  pp.ld_scores = ld_scores;
  pp.cand_pos = cand_pos;
  pp.cand_scores = cand_scores;
  pp.ld_cand = ld_cand;
  pp.T = T;
  pp.K = K;
  pp.pos_offset = pos_offset;
  return from_cuda(launch_topk_pairs(p, ws, pp, reinterpret_cast<cudaStream_t>(stream)));
}

dsa_status dsa_topk_merge(const float* cand_scores, const int32_t* cand_pos, int T, int parts, int per_part,
                          int64_t ld_cand, int64_t part_stride, int K, int32_t* idx, void* stream) {
  if (T < 0 || parts < 1 || per_part < 0 || K < 1) return DSA_ERR_INVALID_ARG;
  if (K > 4096 || (int64_t)parts * per_part > topk_merge_max_candidates()) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!idx) return DSA_ERR_INVALID_ARG;
  if (per_part > 0) {
    if (!cand_scores || !cand_pos) return DSA_ERR_INVALID_ARG;
    if ((T > 1 && ld_cand < per_part) || (parts > 1 && part_stride < per_part)) return DSA_ERR_INVALID_ARG;
  }
  dsa_status s = check_device();
  if (s != DSA_OK) return s;
  MergeParams p = {};
  p.scores = cand_scores;
  p.pos = cand_pos;
  p.ld = ld_cand;
  p.part_stride = part_stride;
  p.T = T;
  p.parts = parts;
  p.per_part = per_part;
  p.K = K;
  p.idx = idx;
  return from_cuda(launch_topk_merge(p, reinterpret_cast<cudaStream_t>(stream), false));
}

dsa_status dsa_sparse_attn_partial(const void* q, const void* kv, const void* kv_v, const float* kv_scale,
                                   int64_t kv_row_stride, int64_t kv_seq_stride, int64_t v_row_stride,
                                   int64_t v_seq_stride, const int32_t* idx, int T, int q_per_seq, int L,
                                   int K, int H, int D_qk, int D_v, float sm_scale, dsa_dtype kv_dtype,
                                   int pos_lo, float* o_part, float* lse_part, void* ws, size_t ws_bytes,
                                   void* stream) {
  dsa_status s = check_sparse_attn(q, kv, kv_v, kv_scale, kv_row_stride, kv_seq_stride, v_row_stride,
                                   v_seq_stride, idx, T, q_per_seq, L, K, H, D_qk, D_v, kv_dtype, o_part);
  if (s != DSA_OK || T == 0) return s;
  if (pos_lo < 0 || !lse_part) return DSA_ERR_INVALID_ARG;
  const size_t need = sparse_attn_ws_bytes(T, H, K, D_v);
  if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return DSA_ERR_WORKSPACE;
  if ((s = check_device()) != DSA_OK) return s;
  dsa_args a = {};
  a.T = T;
  a.q_per_seq = q_per_seq;
  a.L = L;
  a.K = K;
  a.H = H;
  a.D_qk = D_qk;
  a.D_v = D_v;
  a.sm_scale = sm_scale;
  a.kv_dtype = kv_dtype;
  a.q = q;
  a.kv = kv;
  a.kv_v = kv_v;
  a.kv_scale = kv_scale;
  a.kv_row_stride = kv_row_stride;
  a.kv_seq_stride = kv_seq_stride;
  a.v_row_stride = v_row_stride;
  a.v_seq_stride = v_seq_stride;
  a.out = o_part;
  a.lse = lse_part;
  return from_cuda(run_sparse_attn(a, 0, T, idx, ws, reinterpret_cast<cudaStream_t>(stream), false,
                                   /*valid_prefix=*/false, pos_lo, o_part));
}

dsa_status dsa_attn_combine(const float* o_parts, const float* lse_parts, int G, int64_t o_part_stride,
                            int64_t lse_part_stride, int T, int H, int D_v, void* out, float* lse,
                            void* stream) {
  if (G < 1 || T < 0 || H < 1 || D_v < 4 || D_v % 4 != 0) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  if (!o_parts || !lse_parts || !out || !aligned16(o_parts) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)T * H;
  if (G > 1 && (o_part_stride < rows * D_v || o_part_stride % 4 != 0 || lse_part_stride < rows))
    return DSA_ERR_INVALID_ARG;
  dsa_status s = check_device();
  if (s != DSA_OK) return s;
  SliceCombineParams p = {};
  p.o_parts = o_parts;
  p.lse_parts = lse_parts;
  p.o_stride = o_part_stride;
  p.lse_stride = lse_part_stride;
  p.G = G;
  p.T = T;
  p.H = H;
  p.D_v = D_v;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  return from_cuda(launch_slice_combine(p, reinterpret_cast<cudaStream_t>(stream), false));
}

dsa_status dsa_set_attn_kernel(int kernel) { return set_attn_kernel(kernel) ? DSA_OK : DSA_ERR_INVALID_ARG; }

size_t dsa_sparse_attn_workspace_size(int T, int H, int K, int D_v) {
  if (T <= 0 || H <= 0 || K <= 0 || D_v <= 0) return 0;
  return sparse_attn_ws_bytes(T, H, K, D_v);
}

dsa_status dsa_sparse_attn(const void* q, const void* kv, const void* kv_v, const float* kv_scale,
                           int64_t kv_row_stride, int64_t kv_seq_stride, int64_t v_row_stride,
                           int64_t v_seq_stride, const int32_t* idx, int T, int q_per_seq, int L,
                           int K, int H, int D_qk, int D_v, float sm_scale, dsa_dtype kv_dtype,
                           void* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = check_sparse_attn(q, kv, kv_v, kv_scale, kv_row_stride, kv_seq_stride, v_row_stride,
                                   v_seq_stride, idx, T, q_per_seq, L, K, H, D_qk, D_v, kv_dtype, out);
  if (s != DSA_OK || T == 0) return s;
  const size_t need = sparse_attn_ws_bytes(T, H, K, D_v);
  if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return DSA_ERR_WORKSPACE;
  if ((s = check_device()) != DSA_OK) return s;
  dsa_args a = {};
  a.T = T;
  a.q_per_seq = q_per_seq;
  a.L = L;
  a.K = K;
  a.H = H;
  a.D_qk = D_qk;
  a.D_v = D_v;
  a.sm_scale = sm_scale;
  a.kv_dtype = kv_dtype;
  a.q = q;
  a.kv = kv;
  a.kv_v = kv_v;
  a.kv_scale = kv_scale;
  a.kv_row_stride = kv_row_stride;
  a.kv_seq_stride = kv_seq_stride;
  a.v_row_stride = v_row_stride;
  a.v_seq_stride = v_seq_stride;
  a.out = out;
  a.lse = lse;
  return from_cuda(run_sparse_attn(a, 0, T, idx, ws, reinterpret_cast<cudaStream_t>(stream), false,
                                   /*valid_prefix=*/false));
}

dsa_status dsa_workspace_size(const dsa_args* a, int prefill, size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARG;
  dsa_status s = check_args(a, prefill);
  if (s != DSA_OK) return s;
  *bytes = layout_of(*a, prefill).total;
  return DSA_OK;
}

dsa_status dsa_launch_count(const dsa_args* a, int prefill, int* launches) {
  if (!launches) return DSA_ERR_INVALID_ARG;
  const dsa_status s = check_args(a, prefill);
  if (s != DSA_OK) return s;
  const int tc = slice_queries(*a, prefill);
  int n = 0;
  for (int t0 = 0; t0 < a->T; t0 += tc) {
    const int tn = (a->T - t0) < tc ? (a->T - t0) : tc;
    const bool filled =
        a->L > 0 && index_score_builds_hist(tn, a->H_idx, a->q_per_seq, a->idx_dtype == DSA_MXFP8_E4M3);
    n += (a->L > 0 ? 1 : 0) + topk_launches(tn, a->L, filled) +
         sparse_attn_launches(tn, a->H, a->K, a->D_qk, a->D_v, a->kv_dtype != DSA_BF16, a->kv_v != nullptr,
                              a->kv_dtype == DSA_FP8_E4M3_T128, /*chain=*/true);
  }
  *launches = n;
  return DSA_OK;
}

dsa_status dsa_decode(const dsa_args* a, void* ws, size_t ws_bytes, void* stream) {
  return run_chain(a, ws, ws_bytes, stream, 0);
}

dsa_status dsa_prefill(const dsa_args* a, void* ws, size_t ws_bytes, void* stream) {
  return run_chain(a, ws, ws_bytes, stream, 1);
}

}  // extern "C"
