// Step 2 of the chain: Top-K selection ("select the Top-K positions", Day 0 Support for New LLM
// Architectures, Step 1; the Top-k selection operator run after batched scoring, "Achieving
// Day-0 Readiness...", section 2.1).
//
// Radix select on order-preserving 32-bit keys of the fp32 scores, never sorting: three digit
// passes (11, 11, 10 bits) each build a shared-memory histogram of the keys that still match
// the chosen prefix (warp-aggregated with __match_any_sync), and a block-wide suffix scan of the
// histogram picks the digit that holds the K-th largest key.  The final pass keeps every key
// above the threshold prefix and the first `kr` keys equal to it in position order, so exact
// ties go to the lower position, and writes the K positions in ascending order with two
// block-wide prefix scans (no sort, no atomics on the output).
//
// One CTA of 1024 threads per query.  Up to kCachedKeys keys are loaded into shared memory up
// front (padded by one word per 32 so that per-thread contiguous ranges read without
// bank conflicts); longer rows are re-read from global memory (L2) in every pass.
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kBins = 2048;
constexpr int kCachedKeys = 40960;
constexpr int kSmemBytes = (kBins + 64) * 4 + (kCachedKeys + kCachedKeys / 32) * 4;

__device__ __forceinline__ int pad(int i) { return i + (i >> 5); }

// Inclusive prefix sum over the block in thread order.  `ws` holds >= 33 words.
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) ws[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = ws[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    ws[lane] = s;  // inclusive totals per warp
  }
  __syncthreads();
  const uint32_t r = v + (warp > 0 ? ws[warp - 1] : 0u);
  __syncthreads();
  return r;
}

// Inclusive suffix sum over the block (thread i receives the sum over threads >= i).
__device__ __forceinline__ uint32_t block_incl_suffix(uint32_t v, uint32_t* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_down_sync(0xffffffffu, v, o);
    if (lane + o < 32) v += n;
  }
  if (lane == 0) ws[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = ws[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_down_sync(0xffffffffu, s, o);
      if (lane + o < 32) s += n;
    }
    ws[lane] = s;
  }
  __syncthreads();
  const uint32_t r = v + (warp < 31 ? ws[warp + 1] : 0u);
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;             // kBins
  uint32_t* ws = hist + kBins;     // 64 words of scan scratch / broadcast
  uint32_t* keys = ws + 64;        // padded key cache

  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  pdl_wait();
  const int n = visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid);
  const float* sc = p.scores + (int64_t)t * p.ld_scores;
  int32_t* out = p.idx + (int64_t)t * p.K;

  if (n <= p.K) {
    for (int i = tid; i < p.K; i += kThreads) out[i] = i < n ? i : -1;
    pdl_launch_dependents();
    return;
  }
  const bool cached = n <= kCachedKeys;
  if (cached) {
    // load every key first (independent loads, no barriers in between), then count from smem
#pragma unroll 8
    for (int i = tid; i < n; i += kThreads) keys[pad(i)] = float_key(sc[i]);
    __syncthreads();
  }

  uint32_t prefix = 0;  // chosen high digits so far
  int pbits = 0;        // how many high bits are fixed
  uint32_t kr = (uint32_t)p.K;  // how many keys still to take among those matching the prefix
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int width = widths[pass];
    const int shift = 32 - pbits - width;
    const uint32_t dmask = (1u << width) - 1u;
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kThreads) {
      const int i = i0 + tid;
      uint32_t digit = 0xFFFFFFFFu;
      if (i < n) {
        const uint32_t key = cached ? keys[pad(i)] : float_key(sc[i]);
        if (pbits == 0 || (key >> (32 - pbits)) == prefix) digit = (key >> shift) & dmask;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (digit != 0xFFFFFFFFu && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
    }
    __syncthreads();
    // digit d* with  count(digits > d*) < kr <= count(digits >= d*)
    const uint32_t c0 = hist[2 * tid], c1 = hist[2 * tid + 1];
    const uint32_t suffix = block_incl_suffix(c0 + c1, ws);  // keys in bins >= 2*tid
    const uint32_t above1 = suffix - c0 - c1;                // keys in bins > 2*tid + 1
    const uint32_t above0 = above1 + c1;                     // keys in bins > 2*tid
    if (above1 < kr && above1 + c1 >= kr) {
      ws[40] = 2 * tid + 1;
      ws[41] = above1;
    }
    if (above0 < kr && above0 + c0 >= kr) {
      ws[40] = 2 * tid;
      ws[41] = above0;
    }
    __syncthreads();
    const uint32_t d = ws[40];
    kr -= ws[41];
    prefix = (prefix << width) | d;
    pbits += width;
    const uint32_t in_bin = hist[d];
    __syncthreads();
    if (in_bin == kr) break;  // every key with this prefix is taken
  }

  // Final pass: thread tid owns positions [tid*E, tid*E + E) in order.
  const int E = (n + kThreads - 1) / kThreads;
  const int lo = min(n, tid * E), hi = min(n, lo + E);
  const int sh = 32 - pbits;
  auto top = [&](int i) -> uint32_t {
    const uint32_t key = cached ? keys[pad(i)] : float_key(sc[i]);
    return sh >= 32 ? 0u : (key >> sh);
  };
  uint32_t n_gt = 0, n_eq = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t k = top(i);
    n_gt += k > prefix;
    n_eq += k == prefix;
  }
  const uint32_t eq_before = block_incl_scan(n_eq, ws) - n_eq;
  const uint32_t eq_take = eq_before >= kr ? 0u : min(n_eq, kr - eq_before);
  const uint32_t mine = n_gt + eq_take;
  uint32_t pos = block_incl_scan(mine, ws) - mine;
  uint32_t eq_left = eq_take;
  for (int i = lo; i < hi; ++i) {
    const uint32_t k = top(i);
    bool take = k > prefix;
    if (k == prefix && eq_left > 0) {
      take = true;
      --eq_left;
    }
    if (take && pos < (uint32_t)p.K) out[pos++] = i;
  }
  pdl_launch_dependents();
}

}  // namespace

size_t topk_ws_bytes(int, int, int) { return 0; }

cudaError_t launch_topk(const TopkParams& p, void*, cudaStream_t stream, bool pdl) {
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  if (p.T <= 0) return cudaSuccess;
  return launch_kernel(topk_kernel, dim3(p.T), dim3(kThreads), kSmemBytes, stream, pdl, p);
}

}  // namespace dsa
