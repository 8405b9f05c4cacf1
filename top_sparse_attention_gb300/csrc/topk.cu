// Step 2 of the chain: Top-K selection ("select the Top-K positions", Day 0 Support for New LLM
// Architectures, Step 1; the Top-k selection operator run after batched scoring, "Achieving
// Day-0 Readiness...", section 2.1).
//
// Radix select on order-preserving 32-bit keys of the fp32 scores, never sorting.  One
// thread-block cluster of C CTAs (C = 1..16) handles one query; CTA r owns a contiguous slice of
// the query's positions and keeps its keys in shared memory when they fit.
//  * Level 0: a histogram of the top 12 key bits.  In the fused chain it arrives ready-made from
//    the index-score kernel's epilogue; otherwise every CTA adds its non-zero bins into a global
//    per-query histogram (L2 atomics) before a cluster barrier.  Every CTA then reads it and
//    finds, with a block-wide suffix scan, the bin b0 holding the K-th largest key (all CTAs get
//    the same answer, so nothing is broadcast).
//  * Few candidates (the keys of bin b0; the usual case): each CTA lists its candidates in
//    position order, one cluster barrier later every CTA copies all lists through distributed
//    shared memory and resolves the exact threshold key T on its own (two 10-bit digit passes
//    over the candidates), again identically in every CTA.
//  * Many candidates: two more digit levels (12 and 8 bits) run like level 0, with global
//    histograms and a cluster barrier each.
//  * Output in ascending position order: keys above T, then the first ties by position (exact
//    ties go to the lower position).  Per-CTA counts come from the candidate lists (or, on the
//    many-candidate path, through distributed shared memory); a block-wide scan places each
//    thread's positions.  Global histograms are zeroed again before the kernel ends.
// Cluster barriers are hardware barriers: there is no spin loop.
#include <mutex>

#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCachedKeys = 16384;  // largest cached slice
constexpr int kCand = 4096;         // candidates resolved through distributed shared memory
constexpr int kWorkWords = 2 * kHistBins + 256;  // per query: level-0, level-1, level-2 bins

// Shared memory (in 32-bit words): histogram | scratch (96) | counts (4) | own candidate keys,
// positions (min(slice, kCand) each) | all candidate keys, positions (kCand each) | keys
struct TopkSmem {
  int own, keys, words;
  __host__ __device__ TopkSmem(int slice, bool cached) {
    own = slice < kCand ? slice : kCand;
    keys = cached ? slice + slice / 32 : 0;
    words = kHistBins + 96 + 4 + 2 * own + 2 * kCand + keys;
  }
};

__device__ __forceinline__ int pad(int i) { return i + (i >> 5); }

// Block-wide inclusive prefix sum in thread order.
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t* sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) sc[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < kWarps ? sc[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    if (lane < kWarps) sc[lane] = s;
  }
  __syncthreads();
  const uint32_t r = v + (warp > 0 ? sc[warp - 1] : 0u);
  __syncthreads();
  return r;
}

// Block-wide inclusive suffix sum (thread i receives the sum over threads >= i).
__device__ __forceinline__ uint32_t block_incl_suffix(uint32_t v, uint32_t* sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_down_sync(0xffffffffu, v, o);
    if (lane + o < 32) v += n;
  }
  if (lane == 0) sc[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < kWarps ? sc[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_down_sync(0xffffffffu, s, o);
      if (lane + o < 32) s += n;
    }
    if (lane < kWarps) sc[lane] = s;
  }
  __syncthreads();
  const uint32_t r = v + (warp < kWarps - 1 ? sc[warp + 1] : 0u);
  __syncthreads();
  return r;
}

// In the global histogram g of `bins` bins, the bin d holding the kr-th largest element:
// count(bins > d) < kr <= count(bins >= d).  Returns d; `above` = count(bins > d),
// `in_bin` = g[d].
__device__ __forceinline__ uint32_t find_digit(const uint32_t* g, int bins, uint32_t kr, uint32_t* sc,
                                               uint32_t& above, uint32_t& in_bin) {
  const int per = bins >= kThreads ? bins / kThreads : 1;
  const int b0 = threadIdx.x * per;
  uint32_t c[8];
  uint32_t mine = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    c[k] = (k < per && b0 + k < bins) ? __ldcg(g + b0 + k) : 0u;
    mine += c[k];
  }
  uint32_t a = block_incl_suffix(mine, sc) - mine;  // count in bins >= b0 + per
#pragma unroll
  for (int k = 7; k >= 0; --k) {
    if (k < per && b0 + k < bins) {
      if (a < kr && a + c[k] >= kr) {
        sc[64] = (uint32_t)(b0 + k);
        sc[65] = a;
        sc[66] = c[k];
      }
      a += c[k];
    }
  }
  __syncthreads();
  const uint32_t d = sc[64];
  above = sc[65];
  in_bin = sc[66];
  __syncthreads();
  return d;
}

__global__ void __launch_bounds__(kThreads) topk_cluster_kernel(const TopkParams p) {
  extern __shared__ uint32_t sm[];
  pdl_launch_dependents();
  const int t = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int C = (int)cluster_size();
  const int r = (int)cluster_rank();
  pdl_wait();
  const int n = visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid);
  const float* scr = p.scores + (int64_t)t * p.ld_scores;
  int32_t* out = p.idx + (int64_t)t * p.K;
  uint32_t* work = p.work + (int64_t)t * kWorkWords;
  uint32_t* g0 = p.hist ? p.hist + (int64_t)t * kHistBins : work;  // level-0 histogram
  uint32_t* g1 = work + kHistBins;
  uint32_t* g2 = work + 2 * kHistBins;

  if (n <= p.K) {  // the whole cluster leaves here together (n is the same for all its CTAs)
    if (r == 0 && p.hist)
      for (int b = tid; b < kHistBins; b += kThreads) g0[b] = 0;  // leave it zeroed
    for (int i = r * kThreads + tid; i < p.K; i += C * kThreads) out[i] = i < n ? i : -1;
    return;
  }
  const int slice = (((n + C - 1) / C) + 31) & ~31;
  const int lo = min(n, r * slice), hi = min(n, lo + slice), cnt = hi - lo;
  // the shared-memory layout follows the longest row of the launch (the host sizes it the same
  // way), so every CTA of every cluster uses the same offsets
  const int slice_max = (((p.L + C - 1) / C) + 31) & ~31;
  const bool cached = slice_max <= kCachedKeys;
  const TopkSmem L(slice_max, cached);
  uint32_t* hist = sm;              // this CTA's histogram
  uint32_t* sc = hist + kHistBins;  // scan scratch and broadcast words
  uint32_t* counts = sc + 96;       // [0] keys above the threshold / candidates, [1] ties
  uint32_t* own_key = counts + 4;
  uint32_t* own_pos = own_key + L.own;
  uint32_t* all_key = own_pos + L.own;
  uint32_t* all_pos = all_key + kCand;
  uint32_t* keys = all_pos + kCand;
  if (cached) {
#pragma unroll 4
    for (int i = tid; i < cnt; i += kThreads) keys[pad(i)] = float_key(scr[lo + i]);
  }
  auto key_at = [&](int i) -> uint32_t { return cached ? keys[pad(i)] : float_key(scr[lo + i]); };

  // adds this CTA's keys that match `prefix` (pbits high bits) into `hist`, digit = the next
  // `width` bits, then flushes the non-zero bins into the global histogram g
  auto count_level = [&](uint32_t prefix, int pbits, int width, uint32_t* g) {
    const int bins = 1 << width;
    const int shift = 32 - pbits - width;
    for (int b = tid; b < bins; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < cnt; i0 += kThreads) {
      const int i = i0 + tid;
      uint32_t d = 0xFFFFFFFFu;
      if (i < cnt) {
        const uint32_t key = key_at(i);
        if (pbits == 0 || (key >> (32 - pbits)) == prefix) d = (key >> shift) & (uint32_t)(bins - 1);
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (d != 0xFFFFFFFFu && lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
    }
    __syncthreads();
    for (int b = tid; b < bins; b += kThreads)
      if (hist[b]) atomicAdd(&g[b], hist[b]);
    __threadfence();  // the global counts are visible before the cluster barrier completes
  };

  uint32_t prefix = 0;  // chosen high digits so far
  int pbits = 0;        // how many high bits are fixed
  uint32_t kr = (uint32_t)p.K;
  uint32_t above, in_bin;
  // level 0: top 12 bits (complete on entry when it comes from the index-score kernel)
  if (!p.hist) {
    count_level(0, 0, 12, g0);
    cluster_sync();
  } else {
    __syncthreads();
  }
  uint32_t d = find_digit(g0, kHistBins, kr, sc, above, in_bin);
  kr -= above;
  prefix = d;
  pbits = 12;
  const int E = (cnt + kThreads - 1) / kThreads;  // per-thread contiguous ranges, in order
  const int a = min(cnt, tid * E), z = min(cnt, a + E);

  if (in_bin <= (uint32_t)kCand && in_bin != kr) {
    // ---- few candidates: list them, exchange the lists, resolve T in every CTA
    uint32_t n_gt = 0, n_c = 0;
    for (int i = a; i < z; ++i) {
      const uint32_t b = key_at(i) >> 20;
      n_gt += b > d;
      n_c += b == d;
    }
    const uint32_t c_incl = block_incl_scan(n_c, sc);
    const uint32_t gt_incl = block_incl_scan(n_gt, sc);
    uint32_t at = c_incl - n_c;
    for (int i = a; i < z; ++i) {
      const uint32_t key = key_at(i);
      if ((key >> 20) == d) {
        own_key[at] = key;
        own_pos[at] = (uint32_t)(lo + i);
        ++at;
      }
    }
    if (tid == kThreads - 1) {
      counts[0] = c_incl;   // candidates of this CTA
      counts[1] = gt_incl;  // keys in higher bins
    }
    cluster_sync();  // lists and counts complete
    // warp 0: lane q reads CTA q's counts; exclusive prefixes give each list's place
    if (tid < 32) {
      const uint32_t cq = tid < C ? dsmem_ld_u32(dsmem_addr(&counts[0], (uint32_t)tid)) : 0u;
      const uint32_t gq = tid < C ? dsmem_ld_u32(dsmem_addr(&counts[1], (uint32_t)tid)) : 0u;
      uint32_t ci = cq, gi = gq;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t a = __shfl_up_sync(0xffffffffu, ci, o), b = __shfl_up_sync(0xffffffffu, gi, o);
        if (tid >= o) {
          ci += a;
          gi += b;
        }
      }
      sc[32 + tid] = ci - cq;  // candidates before CTA tid
      if (tid == r) sc[80] = gi - gq;  // keys in higher bins before this CTA
      if (tid == 31) sc[81] = ci;      // all candidates
    }
    __syncthreads();
    const uint32_t total = sc[81], my_start = sc[32 + r], gt_before = sc[80];
    // copy every CTA's list (rank order = position order): thread tid fetches entries
    // tid, tid + 512, ... of the concatenated lists, all remote loads first, then the stores
    {
      constexpr int PER = kCand / kThreads;
      uint32_t kk[PER], pp[PER];
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const uint32_t j = (uint32_t)(tid + e * kThreads);
        kk[e] = pp[e] = 0;
        if (j < total) {
          int q = 0;
          while (q + 1 < C && sc[32 + q + 1] <= j) ++q;  // the CTA whose list holds entry j
          const uint32_t local = j - sc[32 + q];
          kk[e] = dsmem_ld_u32(dsmem_addr(own_key, (uint32_t)q) + 4 * local);
          pp[e] = dsmem_ld_u32(dsmem_addr(own_pos, (uint32_t)q) + 4 * local);
        }
      }
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const uint32_t j = (uint32_t)(tid + e * kThreads);
        if (j < total) {
          all_key[j] = kk[e];
          all_pos[j] = pp[e];
        }
      }
    }
    __syncthreads();
    // two 10-bit passes over the candidates' low 20 bits
    uint32_t pre = d;
    int pb = 12;
    for (int pass = 0; pass < 2; ++pass) {
      for (int b = tid; b < 1024; b += kThreads) hist[b] = 0;
      __syncthreads();
      const int shift = 32 - pb - 10;
      // few candidates spread over 1024 bins: plain shared-memory atomics rarely collide
      for (int j = tid; j < (int)total; j += kThreads) {
        const uint32_t key = all_key[j];
        if ((key >> (32 - pb)) == pre) atomicAdd(&hist[(key >> shift) & 1023u], 1u);
      }
      __syncthreads();
      uint32_t ab, ib;
      uint32_t* ls = sc;  // find_digit reads a global histogram; here the bins are in shared memory
      const int per = 2;  // 1024 bins / 512 threads
      uint32_t c0 = hist[2 * tid], c1 = hist[2 * tid + 1];
      uint32_t above1 = block_incl_suffix(c0 + c1, ls) - c0 - c1;
      if (above1 < kr && above1 + c1 >= kr) { ls[64] = 2 * tid + 1; ls[65] = above1; }
      const uint32_t above0 = above1 + c1;
      if (above0 < kr && above0 + c0 >= kr) { ls[64] = 2 * tid; ls[65] = above0; }
      __syncthreads();
      const uint32_t dd = ls[64];
      ab = ls[65];
      (void)per;
      (void)ib;
      __syncthreads();
      kr -= ab;
      pre = (pre << 10) | dd;
      pb += 10;
    }
    const uint32_t T = pre;  // full threshold key; take every key > T and the first kr keys == T
    // selected candidates and ties before this CTA's part of the list
    uint32_t sel_b = 0, tie_b = 0;
    for (uint32_t j = tid; j < my_start; j += kThreads) {
      sel_b += all_key[j] > T;
      tie_b += all_key[j] == T;
    }
    sel_b = block_incl_scan(sel_b, sc);  // the last thread holds the block total
    tie_b = block_incl_scan(tie_b, sc);
    if (tid == kThreads - 1) {
      sc[84] = sel_b;
      sc[85] = tie_b;
    }
    __syncthreads();
    const uint32_t ties_before_cta = sc[85];
    const uint32_t tie_take_before = min(ties_before_cta, kr);
    const uint32_t out_before_cta = gt_before + sc[84] + tie_take_before;
    uint32_t n_sel = 0, n_tie = 0;
    for (int i = a; i < z; ++i) {
      const uint32_t key = key_at(i);
      n_sel += key > T;
      n_tie += key == T;
    }
    const uint32_t tie_incl = block_incl_scan(n_tie, sc);
    const uint32_t tb = ties_before_cta + tie_incl - n_tie;  // ties before this thread's range
    const uint32_t tie_take = tb >= kr ? 0u : min(n_tie, kr - tb);
    const uint32_t take = n_sel + tie_take;
    uint32_t pos = out_before_cta + block_incl_scan(take, sc) - take;
    uint32_t tie_left = tie_take;
    for (int i = a; i < z; ++i) {
      const uint32_t key = key_at(i);
      bool keep = key > T;
      if (key == T && tie_left > 0) {
        keep = true;
        --tie_left;
      }
      if (keep && pos < (uint32_t)p.K) out[pos++] = lo + i;
    }
    cluster_sync();  // every CTA has read the lists
    if (r == 0)
      for (int b = tid; b < kHistBins; b += kThreads) g0[b] = 0;
    return;
  }

  // ---- many candidates: levels 1 and 2 (next 12, then last 8 bits) over all keys
  const int widths[2] = {12, 8};
  uint32_t* gl[2] = {g1, g2};
  for (int lv = 0; lv < 2 && in_bin != kr; ++lv) {
    count_level(prefix, pbits, widths[lv], gl[lv]);
    cluster_sync();
    d = find_digit(gl[lv], 1 << widths[lv], kr, sc, above, in_bin);
    kr -= above;
    prefix = (prefix << widths[lv]) | d;
    pbits += widths[lv];
  }
  // selected: top bits > prefix, plus the first kr keys (by position) whose top bits == prefix
  const int sh = 32 - pbits;
  uint32_t n_gt = 0, n_eq = 0;
  for (int i = a; i < z; ++i) {
    const uint32_t k = key_at(i) >> sh;
    n_gt += k > prefix;
    n_eq += k == prefix;
  }
  const uint32_t eq_incl = block_incl_scan(n_eq, sc);
  const uint32_t gt_incl = block_incl_scan(n_gt, sc);
  if (tid == kThreads - 1) {
    counts[0] = gt_incl;
    counts[1] = eq_incl;
  }
  cluster_sync();  // per-CTA counts visible to the cluster
  if (tid == 0) {
    uint32_t eq_before = 0, out_before = 0;
    for (int q = 0; q < r; ++q) {
      const uint32_t gt_q = dsmem_ld_u32(dsmem_addr(&counts[0], (uint32_t)q));
      const uint32_t eq_q = dsmem_ld_u32(dsmem_addr(&counts[1], (uint32_t)q));
      const uint32_t take_q = eq_before >= kr ? 0u : min(eq_q, kr - eq_before);
      out_before += gt_q + take_q;
      eq_before += eq_q;
    }
    sc[80] = eq_before;
    sc[81] = out_before;
  }
  __syncthreads();
  const uint32_t eq_before = sc[80] + eq_incl - n_eq;
  const uint32_t eq_take = eq_before >= kr ? 0u : min(n_eq, kr - eq_before);
  const uint32_t take = n_gt + eq_take;
  uint32_t pos = sc[81] + block_incl_scan(take, sc) - take;
  uint32_t eq_left = eq_take;
  for (int i = a; i < z; ++i) {
    const uint32_t k = key_at(i) >> sh;
    bool keep = k > prefix;
    if (k == prefix && eq_left > 0) {
      keep = true;
      --eq_left;
    }
    if (keep && pos < (uint32_t)p.K) out[pos++] = lo + i;
  }
  cluster_sync();  // every CTA has read the counts and the global histograms
  if (r == 0) {
    for (int b = tid; b < kHistBins; b += kThreads) {
      g0[b] = 0;
      g1[b] = 0;
    }
    for (int b = tid; b < 256; b += kThreads) g2[b] = 0;
  }
}

// About 2048 keys per CTA, at most 16 CTAs per cluster.
int cluster_ctas(int n_max) {
  int c = 1;
  while (c < 16 && (int64_t)c * 2048 < n_max) c <<= 1;
  return c;
}

}  // namespace

size_t topk_ws_bytes(int T, int, int) { return align_up((size_t)T * kWorkWords * sizeof(uint32_t), 256); }

cudaError_t launch_topk(const TopkParams& p, void* ws, cudaStream_t stream, bool pdl) {
  if (p.T <= 0) return cudaSuccess;
  if (!ws) return cudaErrorInvalidValue;
  TopkParams q = p;
  q.work = reinterpret_cast<uint32_t*>(ws);
  auto kern = topk_cluster_kernel;
  const int C = cluster_ctas(p.L);
  const int slice = (((p.L + C - 1) / C) + 31) & ~31;  // the largest slice of any query
  const size_t smem = (size_t)TopkSmem(slice, slice <= kCachedKeys).words * 4;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, p.T);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, q);
}

// ---------------------------------------------------------------------------------------------
// Top-K without a caller workspace.
//
// Some callers cannot hand the library device memory: a host framework that owns every device
// allocation through its own pool and forbids raw cudaMalloc, or a decode loop that must not
// allocate while it runs (an allocation can synchronise the device and fragment memory).  For
// them dsa_topk_noalloc keeps the Top-K level histograms in the file-scope array below, sized for
// kNoAllocMaxQueries queries.  Every GPU that loads the library holds these bytes until the
// process exits.

constexpr int kNoAllocMaxQueries = 64;
static __device__ __align__(256) uint32_t g_topk_scratch[kNoAllocMaxQueries * kWorkWords];

namespace {

// The array's device address on the current device.  In host code `g_topk_scratch` names a
// host-side stand-in, not device memory, so the address is looked up (once per device, with that
// device current) and passed to the kernel.
cudaError_t scratch_address(uint32_t** out) {
  static std::mutex mu;
  static uint32_t* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_topk_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = reinterpret_cast<uint32_t*>(ptr);
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_topk_noalloc(const float* scores, int64_t ld_scores, int T, int q_per_seq,
                                       int q_pos0, const int32_t* n_valid, int L, int K, int32_t* idx,
                                       void* stream) {
  using namespace dsa;
  dsa_status s = check_topk_args(scores, ld_scores, T, q_per_seq, q_pos0, n_valid, L, K, idx);
  if (s != DSA_OK || T == 0) return s;
  if (T > kNoAllocMaxQueries) return DSA_ERR_UNSUPPORTED;
  if ((s = check_device_arch()) != DSA_OK) return s;
  uint32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the histograms must start at zero; the array keeps whatever the previous call left
  if (cudaMemsetAsync(scratch, 0, (size_t)T * kWorkWords * sizeof(uint32_t), st) != cudaSuccess)
    return DSA_ERR_CUDA;
  TopkParams p = {};
  p.scores = scores;
  p.ld_scores = ld_scores;
  p.n_valid = n_valid;
  p.idx = idx;
  p.T = T;
  p.q_per_seq = q_per_seq;
  p.q_pos0 = q_pos0;
  p.L = L;
  p.K = K;
  p.err = device_error_word();
  return launch_topk(p, scratch, st, false) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
