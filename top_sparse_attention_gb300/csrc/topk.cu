// Step 2 of the chain: Top-K selection (keep the K best-scoring positions, Day 0 Support for New LLM
// Architectures, Step 1; the Top-k selection operator run after batched scoring, "Achieving
// Day-0 Readiness...", section 2.1).
//
// Radix select on order-preserving 32-bit keys of the fp32 scores, never sorting.  One
// thread-block cluster of C CTAs (C = 1..16, about 8192 positions per CTA) handles one query; CTA
// r owns a contiguous slice of the query's positions and keeps its keys in shared memory when the
// slice fits.  Threads read keys four at a time (16-byte loads, chunk-major, thread order within a
// chunk equals position order).  Bulk data crosses CTAs through a per-query area of the workspace
// (L2); single counts go through distributed shared memory; the cluster's hardware barrier orders
// both (no spin loop).
//  * Level 0, the top 12 key bits.  In the fused chain the histogram arrives ready-made from the
//    index-score epilogue; otherwise each CTA counts its keys in shared memory and adds the
//    non-zero bins into the workspace histogram before a barrier.  Every CTA reads it and finds,
//    with a block-wide suffix scan, the same bin b0 holding the K-th largest key.
//  * Pass A: each CTA lists its candidates (keys in bin b0, with positions), counts its keys
//    above b0 and copies the list to its own region of the workspace.  One barrier; the counts
//    then come from the other CTAs' shared memory.
//  * Few candidates (at most 1024 in any CTA, the usual case): every CTA reads every list (thread
//    i holds entry i of each) and resolves the last 20 bits of the threshold key T with two
//    10-bit levels on its own; the lists also give the keys above T and equal to T before its
//    slice.
//    Many candidates: the two levels and the per-CTA counts go through the cluster, one barrier
//    each.
//  * Output, ascending positions: the slot of a kept key is (keys > T before it) + min(keys == T
//    before it, ties to take), so exact ties go to the lower positions; each CTA writes its keys
//    straight to the index row.
// The workspace histograms are zeroed again before the kernel ends.  When given the attention
// cache (TopkParams::kv; the fused chain's build switch DSA_TOPK_KV_PREFETCH, off by default) the
// kernel also prefetches every selected row into L2 as its position is written.
#include <mutex>

#include "dsa_internal.h"

namespace dsa {
namespace {

#ifndef DSA_TOPK_THREADS
#define DSA_TOPK_THREADS 1024
#endif
constexpr int kThreads = DSA_TOPK_THREADS;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 4 * kThreads;  // keys per block-wide step
constexpr int kCachedKeys = 16384;    // largest slice kept in shared memory
// Keys per CTA when sizing a cluster.  A CTA's time is mostly its barriers and scans, so a
// cluster of fewer, fuller CTAs costs less SM time; with independent batches in flight the
// freed SMs run other batches' kernels (decode B = 8, L = 32K: 4-CTA clusters gave 8 % more
// queries/s than 8-CTA ones, at 4 % more latency for one batch alone).
#ifndef DSA_TOPK_KEYS_PER_CTA
#define DSA_TOPK_KEYS_PER_CTA 8192
#endif
constexpr int kKeysPerCta = DSA_TOPK_KEYS_PER_CTA;
// When the cluster kernel signals the attention kernel (griddepcontrol.launch_dependents): 0 at its
// start, 1 once the threshold is known (before the output pass), 2 at its exit.  1 keeps the
// attention CTAs (174 KB of shared memory each) off the SMs while the selection runs.
#ifndef DSA_PDL_LATE_TOPK
#define DSA_PDL_LATE_TOPK 1
#endif
constexpr int kManyQueries = 64;        // launches with at least this many queries ...
constexpr int kManyKeysPerCta = 65536;  // ... use clusters of about this many keys per CTA
constexpr int kCand = 4096;           // own candidate list capacity (shared memory)
constexpr int kRegion = kThreads;     // workspace list entries per CTA (one per thread)
constexpr int kMaxK = 4096;
constexpr int kLevelBins = 1024;      // levels 1 and 2: 10-bit digits
constexpr uint32_t kNoBin = 0xFFFFFFFFu;
constexpr int kBins0 = kHistBins / kThreads;   // level-0 bins per thread
constexpr int kBins1 = kLevelBins / kThreads;  // level-1/2 bins per thread
static_assert(kBins1 >= 1 && kWarps <= 32, "block shape");
// scratch words in sc: [0, 2 * kWarps + 2) scans; named slots from kScOff
constexpr int kScOff = 128;   // [kScOff + q] list entries before CTA q, q = 0..16
constexpr int kScMax = 160;   // longest list
constexpr int kScAbove = 161; // keys above b0 in the CTAs before this one
constexpr int kScGt = 162, kScEq = 163;  // many-candidate path: counts before this CTA
constexpr int kScCand = 200, kScAboveOwn = 201;  // this CTA's candidate and above-b0 counters

// Per-query workspace, in 32-bit words: level-0 histogram (when the chain does not supply one) |
// level-1 histogram | level-2 histogram | C lists of kRegion (key, position) entries.
constexpr int kWsGh0 = 0;
constexpr int kWsGh1 = kWsGh0 + kHistBins;
constexpr int kWsGh2 = kWsGh1 + kLevelBins;
constexpr int kWsList = kWsGh2 + kLevelBins;
__host__ __device__ inline int64_t ws_words(int C) { return kWsList + 2 * (int64_t)C * kRegion; }

// Shared-memory layout in 32-bit words.  The host sizes it from the longest row of the launch.
struct TopkSmem {
  int h0, h1, h2, sc, pub, own, keys, own_cap, words;
  bool cached;
  __host__ __device__ explicit TopkSmem(int slice_max) {
    cached = slice_max <= kCachedKeys;
    own_cap = slice_max < kCand ? slice_max : kCand;
    h0 = 0;                        // level-0 counts of this CTA (kHistBins)
    h1 = h0 + kHistBins;           // level-1 counts
    h2 = h1 + kLevelBins;          // level-2 counts
    sc = h2 + kLevelBins;          // 256 words of scan scratch and broadcasts
    pub = sc + 256;                // 8 words read by the other CTAs of the cluster
    own = pub + 8;                 // this CTA's candidates (key, position), own_cap entries
    keys = own + 2 * own_cap;      // cached keys (16-byte aligned: every offset is a multiple of 4)
    words = keys + (cached ? slice_max : 0);
  }
};

__host__ __device__ inline int slice_of(int n, int C) { return (((n + C - 1) / C) + 31) & ~31; }

// Adds 1 to hist[d] for every lane with d != kNoBin; a warp whose lanes all carry the same digit
// adds 32 with one atomic, so equal keys do not serialise on one shared-memory address.  Every
// lane of the warp must call it.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t d) {
  const uint32_t d0 = __shfl_sync(0xffffffffu, d, 0);
  if (__all_sync(0xffffffffu, d == d0)) {
    if ((threadIdx.x & 31) == 0 && d0 != kNoBin) atomicAdd(&hist[d0], 32u);
  } else if (d != kNoBin) {
    atomicAdd(&hist[d], 1u);
  }
}

// Block-wide exclusive prefix sum of 64-bit values in thread order; *total receives the block
// sum.  Callers pack several counts into disjoint bit fields.  sc: 2 * kWarps + 2 words.
__device__ __forceinline__ uint64_t block_excl_scan(uint64_t v, uint32_t* sc, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  uint64_t* s64 = reinterpret_cast<uint64_t*>(sc);
  if (lane == 31) s64[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint64_t w = lane < kWarps ? s64[lane] : 0ull;
    uint64_t s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kWarps) s64[lane] = s - w;
    if (lane == 31) s64[kWarps] = s;
  }
  __syncthreads();
  const uint64_t r = x - v + s64[warp];
  *total = s64[kWarps];
  __syncthreads();
  return r;
}

// Thread i holds the counts c[0..PER) of bins i*PER .. i*PER+PER-1 (ascending digits).  Finds the
// digit d with count(> d) < kr <= count(>= d); returns d and sets *above = count(> d).
template <int PER>
__device__ __forceinline__ uint32_t find_digit(const uint32_t (&c)[PER], uint32_t kr, uint32_t* sc,
                                               uint32_t* above) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t mine = 0;
#pragma unroll
  for (int k = 0; k < PER; ++k) mine += c[k];
  uint32_t x = mine;  // inclusive suffix sum over the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) sc[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = lane < kWarps ? sc[lane] : 0u;
    uint32_t s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, s, o);
      if (lane + o < 32) s += y;
    }
    if (lane < kWarps) sc[lane] = s - w;  // count in higher warps
  }
  __syncthreads();
  uint32_t a = x - mine + sc[warp];  // count in higher threads' bins
#pragma unroll
  for (int k = PER - 1; k >= 0; --k) {
    if (a < kr && a + c[k] >= kr) {  // exactly one bin of the block satisfies this
      sc[kWarps] = (uint32_t)(threadIdx.x * PER + k);
      sc[kWarps + 1] = a;
    }
    a += c[k];
  }
  __syncthreads();
  const uint32_t d = sc[kWarps];
  *above = sc[kWarps + 1];
  __syncthreads();
  return d;
}

// Global histogram read as PER consecutive bins per thread.
template <int PER>
__device__ __forceinline__ void load_bins(const uint32_t* g, uint32_t (&c)[PER]) {
  if constexpr (PER % 4 == 0) {
#pragma unroll
    for (int v = 0; v < PER / 4; ++v) {
      const uint4 a = __ldcg(reinterpret_cast<const uint4*>(g) + (PER / 4) * threadIdx.x + v);
      c[4 * v] = a.x, c[4 * v + 1] = a.y, c[4 * v + 2] = a.z, c[4 * v + 3] = a.w;
    }
  } else if constexpr (PER == 2) {
    const uint2 a = __ldcg(reinterpret_cast<const uint2*>(g) + threadIdx.x);
    c[0] = a.x, c[1] = a.y;
  } else {
    static_assert(PER == 1, "bins per thread");
    c[0] = __ldcg(g + threadIdx.x);
  }
}

// Adds a shared-memory histogram's non-zero bins into a global one: one 64-bit atomic add per pair
// of bins with a non-zero count (the low word never carries: a row has fewer than 2^32 positions),
// or one 32-bit add per bin when the global histogram is not 8-byte aligned.
__device__ __forceinline__ void flush_bins(const uint32_t* h, uint32_t* g, int bins) {
  if ((reinterpret_cast<uintptr_t>(g) & 7u) == 0 && bins % 2 == 0) {
    const uint2* h2 = reinterpret_cast<const uint2*>(h);
    unsigned long long* g2 = reinterpret_cast<unsigned long long*>(g);
    for (int pr = threadIdx.x; pr < bins / 2; pr += kThreads) {
      const uint2 v = h2[pr];
      if (v.x | v.y) atomicAdd(g2 + pr, (unsigned long long)v.y << 32 | v.x);
    }
    return;
  }
  for (int b = threadIdx.x; b < bins; b += kThreads) {
    const uint32_t v = h[b];
    if (v) atomicAdd(&g[b], v);
  }
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads) topk_cluster_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t sm[];
  if (DSA_PDL_LATE_TOPK == 0) pdl_launch_dependents();
  const int t = blockIdx.y;
  const int tid = threadIdx.x;
  const int C = (int)cluster_size();
  const int r = (int)cluster_rank();
  pdl_wait();
  const int n = visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid);
  const float* scr = p.scores + (int64_t)t * p.ld_scores;
  int32_t* out = p.idx + (int64_t)t * p.idx_ld;
  uint32_t* ws = p.work + (int64_t)t * ws_words(C);
  uint32_t* gh0 = p.hist ? p.hist + (int64_t)t * kHistBins : ws + kWsGh0;
  uint32_t* gh1 = ws + kWsGh1;
  uint32_t* gh2 = ws + kWsGh2;
  uint2* glist = reinterpret_cast<uint2*>(ws + kWsList);

  // L2 prefetch of a selected row of the attention cache (chain only)
  const int64_t seq = (t + p.t_off) / p.q_per_seq;
  const bool paged = p.pages.table != nullptr;
  const uint8_t* pf_kv = p.kv ? p.kv + (paged ? 0 : seq * p.kv_seq_stride) : nullptr;
  const uint8_t* pf_v = p.kv_v ? p.kv_v + (paged ? 0 : seq * p.v_seq_stride) : nullptr;
  auto prefetch_row = [&](uint32_t pos) {
    const int64_t row = paged ? page_row(p.pages, seq, (int)pos) : (int64_t)pos;
    prefetch_l2(pf_kv + row * p.kv_row_stride, (uint32_t)p.kv_bytes);
    if (pf_v) prefetch_l2(pf_v + row * p.v_row_stride, (uint32_t)p.v_bytes);
  };

  if (n <= p.K) {  // the whole cluster leaves here together (n is the same for all its CTAs)
    if (r == 0 && p.hist)
      for (int b = tid; b < kHistBins; b += kThreads) gh0[b] = 0;  // leave it zeroed
    for (int i = r * kThreads + tid; i < p.K; i += C * kThreads) {
      out[i] = i < n ? i : -1;
      if (pf_kv && i < n) prefetch_row((uint32_t)i);
    }
    return;
  }
  const TopkSmem S(slice_of(p.L, C));
  const int slice = slice_of(n, C);
  const int lo = min(n, r * slice), cnt = min(n, lo + slice) - lo;
  uint32_t* h0 = sm + S.h0;
  uint32_t* h1 = sm + S.h1;
  uint32_t* h2 = sm + S.h2;
  uint32_t* sc = sm + S.sc;
  uint32_t* pub = sm + S.pub;
  uint2* own = reinterpret_cast<uint2*>(sm + S.own);
  uint32_t* keys = sm + S.keys;
  const float* src = scr + lo;
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;

  // keys at local positions i .. i+3 (i a multiple of 4); positions >= cnt read as 0 and every
  // caller excludes them with its own bound check
  auto load_global = [&](int i, uint32_t (&k)[4]) {
    if (vec && i + 3 < cnt) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + i));
      k[0] = float_key(v.x), k[1] = float_key(v.y), k[2] = float_key(v.z), k[3] = float_key(v.w);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) k[j] = i + j < cnt ? float_key(__ldcg(src + i + j)) : 0u;
    }
  };
  auto load4 = [&](int i, uint32_t (&k)[4]) {
    if (i >= cnt) {
      k[0] = k[1] = k[2] = k[3] = 0u;
    } else if (S.cached) {
      const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
      k[0] = v.x, k[1] = v.y, k[2] = v.z, k[3] = v.w;
    } else {
      load_global(i, k);
    }
  };

  // ---- loads: the level-0 counts (when ready-made) and this slice's keys, all in flight at once
  uint32_t c0[kBins0];
  if (p.hist) load_bins<kBins0>(gh0, c0);
  if (S.cached) {
    constexpr int kFill = kCachedKeys / kChunk;
    uint32_t k[kFill][4];
#pragma unroll
    for (int f = 0; f < kFill; ++f)
      if (f * kChunk < cnt) load_global(f * kChunk + 4 * tid, k[f]);
#pragma unroll
    for (int f = 0; f < kFill; ++f) {
      const int i = f * kChunk + 4 * tid;
      if (i < cnt) *reinterpret_cast<uint4*>(keys + i) = make_uint4(k[f][0], k[f][1], k[f][2], k[f][3]);
    }
  }
#pragma unroll
  for (int k = 0; k < kBins1; ++k) h1[kBins1 * tid + k] = h2[kBins1 * tid + k] = 0;
  if (tid == 0) sc[kScCand] = sc[kScAboveOwn] = 0;

  // ---- level 0: top 12 bits
  if (!p.hist) {
    for (int b = tid; b < kHistBins / 4; b += kThreads) reinterpret_cast<uint4*>(h0)[b] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    for (int base = 0; base < cnt; base += kChunk) {
      const int i = base + 4 * tid;
      uint32_t k[4];
      load4(i, k);
#pragma unroll
      for (int j = 0; j < 4; ++j) hist_add(h0, i + j < cnt ? k[j] >> 20 : kNoBin);
    }
    __syncthreads();
    flush_bins(h0, gh0, kHistBins);
    cluster_sync();  // every CTA's counts are in gh0 (the barrier's release orders the atomics)
    load_bins<kBins0>(gh0, c0);
  } else {
    __syncthreads();  // cached keys and cleared histograms visible
  }
  uint32_t above;
  uint32_t kr = (uint32_t)p.K;
  const uint32_t b0 = find_digit<kBins0>(c0, kr, sc, &above);
  kr -= above;

  // ---- pass A: this CTA's candidates (bin b0) and its count of keys above b0.  A thread takes its
  // keys of up to two chunks per step (the list order does not matter to the steps after it)
  {
    uint32_t n_above = 0;
    const int lane = tid & 31;
    for (int base = 0; base < cnt; base += 2 * kChunk) {
      const int i = base + 4 * tid;
      uint32_t k[8];
      {
        uint32_t a[4], b[4];
        load4(i, a);
        load4(i + kChunk, b);
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = a[j], k[4 + j] = b[j];
      }
      uint32_t cm = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int pos = i + (j < 4 ? j : kChunk + j - 4);
        const bool ok = pos < cnt;
        const uint32_t d = k[j] >> 20;
        n_above += ok && d > b0;
        cm |= (uint32_t)(ok && d == b0) << j;
      }
      // one shared-memory atomic per warp places the warp's candidates
      const uint32_t nc = __popc(cm);
      uint32_t x = nc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      uint32_t at = 0;
      if (lane == 31 && x) at = atomicAdd(&sc[kScCand], x);
      at = __shfl_sync(0xffffffffu, at, 31) + x - nc;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if ((cm >> j) & 1u) {
          const int pos = i + (j < 4 ? j : kChunk + j - 4);
          if (at < (uint32_t)S.own_cap) own[at] = make_uint2(k[j], (uint32_t)(lo + pos));
          ++at;
        }
    }
    n_above = __reduce_add_sync(0xffffffffu, n_above);
    if ((tid & 31) == 0 && n_above) atomicAdd(&sc[kScAboveOwn], n_above);
  }
  __syncthreads();
  const uint32_t own_cand = sc[kScCand];
  if (tid == 0) {
    pub[0] = own_cand;
    pub[1] = sc[kScAboveOwn];
  }
  {
    const uint32_t m = min(own_cand, (uint32_t)kRegion);
    uint2* region = glist + (int64_t)r * kRegion;
    for (uint32_t j = tid; j < m; j += kThreads) region[j] = own[j];
  }
  cluster_sync();  // lists and counts of every CTA are published

  // ---- every CTA's counts (distributed shared memory): list offsets, keys above b0 before
  if (tid < 32) {
    const uint2 v = tid < C ? dsmem_ld_u2(dsmem_addr(pub, (uint32_t)tid)) : make_uint2(0u, 0u);
    (void)__reduce_or_sync(0xffffffffu, v.x);  // every lane's count has arrived before the scan
    uint32_t x = v.x, mx = v.x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (tid >= o) x += y;
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const uint32_t ab = __reduce_add_sync(0xffffffffu, tid < r ? v.y : 0u);
    if (tid <= 16) sc[kScOff + tid] = x - v.x;  // entries before CTA tid (entry C = total)
    if (tid == 0) {
      sc[kScMax] = mx;
      sc[kScAbove] = ab;
    }
  }
  __syncthreads();
  const bool few = sc[kScMax] <= (uint32_t)kRegion;
  uint32_t gt_before = sc[kScAbove], eq_before = 0;
  uint32_t T;
  uint64_t bf = 0;  // (list keys > T << 48) | (list keys == T << 32) before this slice, per thread

  if (few) {
    cluster_arrive();  // this CTA's reads of the others' shared memory are done
    // ---- few candidates: every CTA's list, levels 1 and 2 resolved here
    // entry tid of every CTA's list (a list holds at most kRegion = kThreads entries):
    // coalesced loads, no search for the owner.  Threads past the longest list hold nothing.
    const bool holds = (uint32_t)tid < sc[kScMax];
    uint32_t vm = 0;  // bit q: this thread holds entry tid of CTA q's list
    uint2 e[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (q >= C || !holds) break;
      if ((uint32_t)tid < sc[kScOff + q + 1] - sc[kScOff + q]) {
        vm |= 1u << q;
        e[q] = __ldcg(glist + (int64_t)q * kRegion + tid);
      }
    }
    // few candidates spread over 1024 bins: plain shared-memory atomics rarely collide
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (!(vm >> q)) break;
      if ((vm >> q) & 1u) atomicAdd(&h1[(e[q].x >> 10) & (kLevelBins - 1)], 1u);
    }
    __syncthreads();
    uint32_t c1[kBins1];
#pragma unroll
    for (int k = 0; k < kBins1; ++k) c1[k] = h1[kBins1 * tid + k];
    const uint32_t d1 = find_digit<kBins1>(c1, kr, sc, &above);
    kr -= above;
    const uint32_t p22 = (b0 << 10) | d1;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (!(vm >> q)) break;
      if (((vm >> q) & 1u) && (e[q].x >> 10) == p22) atomicAdd(&h2[e[q].x & (kLevelBins - 1)], 1u);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBins1; ++k) c1[k] = h2[kBins1 * tid + k];
    const uint32_t d2 = find_digit<kBins1>(c1, kr, sc, &above);
    kr -= above;
    T = (p22 << 10) | d2;
    uint32_t g_ = 0, q_ = 0;
    const uint32_t before_mask = vm & ((1u << r) - 1u);  // lists of the CTAs before this one
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (!(before_mask >> q)) break;
      const bool m = (before_mask >> q) & 1u;
      g_ += m && e[q].x > T;
      q_ += m && e[q].x == T;
    }
    bf = ((uint64_t)g_ << 48) | ((uint64_t)q_ << 32);
  } else {
    // ---- many candidates: levels 1 and 2 and the per-CTA counts go through the cluster
    const bool listed = own_cand <= (uint32_t)S.own_cap;
    uint32_t prefix = b0;
    int pbits = 12;
#pragma unroll 1
    for (int lv = 0; lv < 2; ++lv) {
      uint32_t* h = lv == 0 ? h1 : h2;
      uint32_t* gh = lv == 0 ? gh1 : gh2;
      const int shift = 32 - pbits - 10;
      if (listed) {
        for (uint32_t j0 = 0; j0 < own_cand; j0 += kThreads) {
          const uint32_t j = j0 + tid;
          const bool m = j < own_cand && (own[j].x >> (32 - pbits)) == prefix;
          hist_add(h, m ? (own[j].x >> shift) & (kLevelBins - 1) : kNoBin);
        }
      } else {
        for (int base = 0; base < cnt; base += kChunk) {
          const int i = base + 4 * tid;
          uint32_t k[4];
          load4(i, k);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const bool m = i + j < cnt && (k[j] >> (32 - pbits)) == prefix;
            hist_add(h, m ? (k[j] >> shift) & (kLevelBins - 1) : kNoBin);
          }
        }
      }
      __syncthreads();
      flush_bins(h, gh, kLevelBins);
      cluster_sync();  // every CTA's level counts are in gh
      uint32_t c1[kBins1];
      load_bins<kBins1>(gh, c1);
      const uint32_t d = find_digit<kBins1>(c1, kr, sc, &above);
      kr -= above;
      prefix = (prefix << 10) | d;
      pbits += 10;
    }
    T = prefix;
    uint32_t g_ = 0, q_ = 0;  // this CTA's candidates above T, keys equal to T
    if (listed) {
      for (uint32_t j = tid; j < own_cand; j += kThreads) {
        const uint32_t key = own[j].x;
        g_ += key > T;
        q_ += key == T;
      }
    } else {
      for (int base = 0; base < cnt; base += kChunk) {
        const int i = base + 4 * tid;
        uint32_t k[4];
        load4(i, k);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          g_ += i + j < cnt && (k[j] >> 20) == b0 && k[j] > T;
          q_ += i + j < cnt && k[j] == T;
        }
      }
    }
    uint64_t tot;
    block_excl_scan(((uint64_t)g_ << 32) | q_, sc, &tot);
    if (tid == 0) {
      pub[2] = pub[1] + (uint32_t)(tot >> 32);  // keys above T
      pub[3] = (uint32_t)tot;                   // keys equal to T
    }
    cluster_sync();  // per-CTA counts visible
    if (tid < 32) {
      const uint2 v = tid < r ? dsmem_ld_u2(dsmem_addr(pub + 2, (uint32_t)tid)) : make_uint2(0u, 0u);
      const uint32_t x = __reduce_add_sync(0xffffffffu, v.x), y = __reduce_add_sync(0xffffffffu, v.y);
      if (tid == 0) {
        sc[kScGt] = x;
        sc[kScEq] = y;
      }
    }
    __syncthreads();
    cluster_arrive();  // this CTA's reads of the others' shared memory are done
    gt_before = sc[kScGt];
    eq_before = sc[kScEq];
  }

  if (DSA_PDL_LATE_TOPK == 1) pdl_launch_dependents();
  // ---- output, ascending positions: slot = (keys > T before) + min(keys == T before, kr).
  // One 64-bit scan per chunk: low half = (ties << 16 | keys above T) prefix in the chunk, high
  // half = the list counts before this slice (first chunk only; summed over the block).
  uint32_t gt_in = 0, eq_in = 0;  // keys above T / ties of this slice before the chunk
  for (int base = 0; base < cnt; base += kChunk) {
    const int i = base + 4 * tid;
    uint32_t k[4];
    load4(i, k);
    uint32_t ng = 0, ne = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      ng += i + j < cnt && k[j] > T;
      ne += i + j < cnt && k[j] == T;
    }
    uint64_t tot;
    const uint64_t ex = block_excl_scan((uint64_t)(ng | (ne << 16)) | (base == 0 ? bf : 0ull), sc, &tot);
    if (base == 0) {
      gt_before += (uint32_t)(tot >> 48);
      eq_before += (uint32_t)(tot >> 32) & 0xFFFFu;
    }
    uint32_t gb = gt_before + gt_in + ((uint32_t)ex & 0xFFFFu);
    uint32_t eb = eq_before + eq_in + (((uint32_t)ex >> 16) & 0xFFFFu);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool ok = i + j < cnt;
      const bool is_gt = ok && k[j] > T, is_eq = ok && k[j] == T;
      if (is_gt || (is_eq && eb < kr)) {
        const uint32_t slot = gb + min(eb, kr);
        if (slot < (uint32_t)p.K) out[slot] = lo + i + j;
        if (pf_kv) prefetch_row((uint32_t)(lo + i + j));
      }
      gb += is_gt;
      eb += is_eq;
    }
    gt_in += (uint32_t)tot & 0xFFFFu;
    eq_in += ((uint32_t)tot >> 16) & 0xFFFFu;
  }
  cluster_wait();  // every CTA is past its reads of the workspace histograms and of this CTA
  // leave the workspace histograms zeroed, split over the cluster's CTAs
  for (int i = r * kThreads + tid; i < kHistBins / 4; i += C * kThreads)
    reinterpret_cast<uint4*>(gh0)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (!few)
    for (int i = r * kThreads + tid; i < 2 * kLevelBins / 4; i += C * kThreads)
      reinterpret_cast<uint4*>(gh1)[i] = make_uint4(0u, 0u, 0u, 0u);  // gh1 and gh2 are adjacent
}

// ---------------------------------------------------------------------------------------------
// Row-split Top-K for long rows.
//
// A cluster holds at most 16 CTAs, so one query over a million positions would keep 16 SMs busy
// and re-read most of its keys from L2 on every pass.  Here a row is cut into chunks, one CTA
// each, and the CTAs of a row exchange counts through the workspace between kernels, so no CTA
// ever waits on another:
//  * scan (one CTA per chunk): every CTA finds the level-0 bin b0 from the row's 12-bit histogram,
//    counts its keys above b0, appends its candidates (keys in b0, with positions) to its own
//    list and adds their next 10 bits into the row's level-1 histogram;
//  * resolve (one CTA per row): the level-1 digit, a level-2 histogram of the matching candidates
//    (one warp per chunk list), the threshold key T and the ties to take, then each chunk's
//    candidates above and equal to T and their exclusive prefixes over the chunks; the row's
//    histograms are zeroed again;
//  * emit (one CTA per chunk): the chunk's keys are read once more and every kept position goes
//    to slot (keys > T before it) + min(keys == T before it, ties to take), as in the cluster path.
// Without a histogram from the index-score kernel a first kernel builds it from the chunks.

// Per-query workspace of the row-split path, in 32-bit words: level-0 histogram (when none is
// supplied) | level-1 histogram | 8 row words | 4 words per chunk | one (key, position) list of
// `chunk` entries per chunk.
constexpr int kWsWGh0 = 0;
constexpr int kWsWGh1 = kWsWGh0 + kHistBins;
constexpr int kWsWRow = kWsWGh1 + kLevelBins;  // [0] T, [1] ties to take
constexpr int kWsWChunk = kWsWRow + 8;         // per chunk: above b0, candidates, > T before, == T before
constexpr int kWideMaxChunks = kThreads;       // the resolve kernel scans one chunk per thread
__host__ __device__ inline int64_t wide_words(int nch, int chunk) {
  return kWsWChunk + 4 * (int64_t)nch + 2 * (int64_t)nch * chunk;
}

struct WideRow {
  uint32_t* gh0;
  uint32_t* gh1;
  uint32_t* row;
  uint32_t* chunk;
  uint2* lists;
};

__device__ __forceinline__ WideRow wide_row(const TopkParams& p, int t) {
  uint32_t* ws = p.work + (int64_t)t * wide_words(p.wide_nch, p.wide_chunk);
  WideRow w;
  w.gh0 = p.hist ? p.hist + (int64_t)t * kHistBins : ws + kWsWGh0;
  w.gh1 = ws + kWsWGh1;
  w.row = ws + kWsWRow;
  w.chunk = ws + kWsWChunk;
  w.lists = reinterpret_cast<uint2*>(ws + kWsWChunk + 4 * (int64_t)p.wide_nch);
  return w;
}

// Keys of one chunk: positions [lo, lo + cnt) of row t.
struct ChunkKeys {
  const float* src;
  int lo, cnt;
  bool vec;
  __device__ ChunkKeys(const TopkParams& p, int t, int c, int n) {
    lo = min(n, c * p.wide_chunk);
    cnt = min(n, lo + p.wide_chunk) - lo;
    src = p.scores + (int64_t)t * p.ld_scores + lo;
    vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  }
  // keys at local positions i .. i+3; positions >= cnt read as 0 (callers bound-check)
  __device__ __forceinline__ void load(int i, uint32_t (&k)[4]) const {
    if (vec && i + 3 < cnt) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + i));
      k[0] = float_key(v.x), k[1] = float_key(v.y), k[2] = float_key(v.z), k[3] = float_key(v.w);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) k[j] = i + j < cnt ? float_key(__ldcg(src + i + j)) : 0u;
    }
  }
};

__global__ void __launch_bounds__(kThreads) topk_wide_hist_kernel(const TopkParams p) {
  __shared__ uint32_t h0[kHistBins];
  pdl_launch_dependents();
  const int c = blockIdx.x, t = blockIdx.y, tid = threadIdx.x;
  for (int b = tid; b < kHistBins; b += kThreads) h0[b] = 0;
  pdl_wait();
  const int n = visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid);
  if (n <= p.K) return;  // every position is kept; nothing to count
  const ChunkKeys ck(p, t, c, n);
  __syncthreads();
  for (int base = 0; base < ck.cnt; base += kChunk) {
    const int i = base + 4 * tid;
    uint32_t k[4];
    ck.load(i, k);
#pragma unroll
    for (int j = 0; j < 4; ++j) hist_add(h0, i + j < ck.cnt ? k[j] >> 20 : kNoBin);
  }
  __syncthreads();
  flush_bins(h0, wide_row(p, t).gh0, kHistBins);
}

__global__ void __launch_bounds__(kThreads) topk_wide_scan_kernel(const TopkParams p) {
  __shared__ uint32_t h1[kLevelBins];
  __shared__ uint32_t sc[256];
  pdl_launch_dependents();
  const int c = blockIdx.x, t = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
#pragma unroll
  for (int k = 0; k < kBins1; ++k) h1[kBins1 * tid + k] = 0;
  if (tid == 0) sc[kScCand] = sc[kScAboveOwn] = 0;
  pdl_wait();
  const int n = visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid);
  if (n <= p.K) return;
  const WideRow w = wide_row(p, t);
  const ChunkKeys ck(p, t, c, n);
  uint32_t c0[kBins0];
  load_bins<kBins0>(w.gh0, c0);
  uint32_t above;
  const uint32_t b0 = find_digit<kBins0>(c0, (uint32_t)p.K, sc, &above);  // also orders the zeroing
  uint2* list = w.lists + (int64_t)c * p.wide_chunk;
  uint32_t n_above = 0;
  for (int base = 0; base < ck.cnt; base += kChunk) {
    const int i = base + 4 * tid;
    uint32_t k[4];
    ck.load(i, k);
    uint32_t cm = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool ok = i + j < ck.cnt;
      const uint32_t d = k[j] >> 20;
      n_above += ok && d > b0;
      cm |= (uint32_t)(ok && d == b0) << j;
    }
    // candidates go to this chunk's list (one shared-memory atomic per warp places them)
    const uint32_t nc = __popc(cm);
    uint32_t incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
    if (tot) {
      uint32_t wbase = 0;
      if (lane == 31) wbase = atomicAdd(&sc[kScCand], tot);
      uint32_t o = __shfl_sync(0xffffffffu, wbase, 31) + incl - nc;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if ((cm >> j) & 1u) {
          list[o++] = make_uint2(k[j], (uint32_t)(ck.lo + i + j));
          atomicAdd(&h1[(k[j] >> 10) & (kLevelBins - 1)], 1u);
        }
    }
  }
  n_above = __reduce_add_sync(0xffffffffu, n_above);
  if (lane == 0 && n_above) atomicAdd(&sc[kScAboveOwn], n_above);
  __syncthreads();
  flush_bins(h1, w.gh1, kLevelBins);
  if (tid == 0) {
    w.chunk[4 * c] = sc[kScAboveOwn];
    w.chunk[4 * c + 1] = sc[kScCand];
  }
}

// Adds 1 to arr[idx] for every lane with pred; a warp whose predicated lanes share one index adds
// them with a single atomic (equal keys and long same-chunk runs do not serialise on one
// address).  Every lane of the warp must call it.
__device__ __forceinline__ void warp_count(uint32_t* arr, uint32_t idx, bool pred) {
  const uint32_t m = __ballot_sync(0xffffffffu, pred);
  if (!m) return;
  const int first = __ffs(m) - 1;
  const uint32_t i0 = __shfl_sync(0xffffffffu, idx, first);
  if (__all_sync(0xffffffffu, !pred || idx == i0)) {
    if ((threadIdx.x & 31) == first) atomicAdd(&arr[i0], (uint32_t)__popc(m));
  } else if (pred) {
    atomicAdd(&arr[idx], 1u);
  }
}

constexpr int kStash = 2048;  // candidates that share the first 22 bits of T, kept in shared memory

__global__ void __launch_bounds__(kThreads) topk_wide_resolve_kernel(const TopkParams p) {
  __shared__ uint32_t h2[kLevelBins];
  __shared__ uint32_t sc[256];
  __shared__ uint32_t off_c[kWideMaxChunks + 1];  // first flattened candidate of each chunk
  __shared__ uint32_t gt_c[kWideMaxChunks];       // per chunk: candidates above T
  __shared__ uint32_t eq_c[kWideMaxChunks];       // per chunk: keys equal to T
  __shared__ uint2 stash[kStash];                 // (chunk, key) of the candidates in T's 22-bit bin
  pdl_launch_dependents();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = p.wide_nch;
#pragma unroll
  for (int k = 0; k < kBins1; ++k) h2[kBins1 * tid + k] = 0;
  for (int c = tid; c < kWideMaxChunks; c += kThreads) gt_c[c] = eq_c[c] = 0;
  if (tid == 0) sc[kScCand] = 0;
  pdl_wait();
  const int n = visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid);
  const WideRow w = wide_row(p, t);
  if (n <= p.K) {  // the ready-made histogram is left zeroed; the emit kernel keeps everything
    if (p.hist)
      for (int b = tid; b < kHistBins / 4; b += kThreads)
        reinterpret_cast<uint4*>(w.gh0)[b] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  // all loads of the row's small data at once: histograms and this thread's chunk counts
  uint32_t c0[kBins0], c1[kBins1];
  load_bins<kBins0>(w.gh0, c0);
  load_bins<kBins1>(w.gh1, c1);
  const uint32_t above_b0 = tid < nch ? __ldcg(w.chunk + 4 * tid) : 0u;
  const uint32_t cand = tid < nch ? __ldcg(w.chunk + 4 * tid + 1) : 0u;
  uint32_t above, kr = (uint32_t)p.K;
  const uint32_t b0 = find_digit<kBins0>(c0, kr, sc, &above);
  kr -= above;
  const uint32_t d1 = find_digit<kBins1>(c1, kr, sc, &above);
  kr -= above;
  const uint32_t p22 = (b0 << 10) | d1;  // the first 22 bits of T
  // every thread has read both histograms (find_digit ends with a barrier): leave them zeroed
  for (int b = tid; b < kHistBins / 4; b += kThreads)
    reinterpret_cast<uint4*>(w.gh0)[b] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int k = 0; k < kBins1; ++k) w.gh1[kBins1 * tid + k] = 0;
  uint64_t total;
  const uint64_t ex = block_excl_scan(cand, sc, &total);
  if (tid < nch) off_c[tid] = (uint32_t)ex;
  if (tid == 0) off_c[nch] = (uint32_t)total;
  __syncthreads();
  const uint32_t n_cand = (uint32_t)total;

  // candidate i of the flattened lists: its chunk (binary search over off_c) and its key
  auto cand_key = [&](uint32_t i, uint32_t* c_out) -> uint32_t {
    int lo = 0, hi = nch - 1;  // largest c with off_c[c] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off_c[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    *c_out = (uint32_t)lo;
    return __ldcg(&w.lists[(int64_t)lo * p.wide_chunk + (i - off_c[lo])].x);
  };

  // level 2 over the candidates in T's 22-bit bin; candidates above that bin count for their
  // chunk now; the bin's candidates are stashed for the per-chunk counts
  for (uint32_t base = (uint32_t)warp * 32; base < n_cand; base += kThreads) {
    const uint32_t i = base + lane;
    uint32_t c = 0, key = 0;
    if (i < n_cand) key = cand_key(i, &c);
    const bool in_bin = i < n_cand && (key >> 10) == p22;
    warp_count(gt_c, c, i < n_cand && (key >> 10) > p22);
    hist_add(h2, in_bin ? (key & (kLevelBins - 1)) : kNoBin);
    const uint32_t m = __ballot_sync(0xffffffffu, in_bin);
    if (m) {
      uint32_t at = 0;
      if (lane == 0) at = atomicAdd(&sc[kScCand], (uint32_t)__popc(m));
      at = __shfl_sync(0xffffffffu, at, 0) + __popc(m & ((1u << lane) - 1u));
      if (in_bin && at < kStash) stash[at] = make_uint2(c, key);
    }
  }
  __syncthreads();
  const uint32_t n_bin = sc[kScCand];
#pragma unroll
  for (int k = 0; k < kBins1; ++k) c1[k] = h2[kBins1 * tid + k];
  const uint32_t d2 = find_digit<kBins1>(c1, kr, sc, &above);
  kr -= above;  // ties to take
  const uint32_t T = (p22 << 10) | d2;

  // per chunk: bin candidates above T and keys equal to T (from the stash, or the lists again
  // when the bin held more than the stash)
  if (n_bin <= (uint32_t)kStash) {
    for (uint32_t base = (uint32_t)warp * 32; base < n_bin; base += kThreads) {
      const uint32_t i = base + lane;
      const uint2 e = i < n_bin ? stash[i] : make_uint2(0u, 0u);
      warp_count(gt_c, e.x, i < n_bin && e.y > T);
      warp_count(eq_c, e.x, i < n_bin && e.y == T);
    }
  } else {
    for (uint32_t base = (uint32_t)warp * 32; base < n_cand; base += kThreads) {
      const uint32_t i = base + lane;
      uint32_t c = 0, key = 0;
      if (i < n_cand) key = cand_key(i, &c);
      const bool in_bin = i < n_cand && (key >> 10) == p22;
      warp_count(gt_c, c, in_bin && key > T);
      warp_count(eq_c, c, in_bin && key == T);
    }
  }
  __syncthreads();
  // exclusive prefixes over the chunks (one chunk per thread; both sums stay below 2^32)
  const uint64_t v = tid < nch ? ((uint64_t)eq_c[tid] << 32) | (gt_c[tid] + above_b0) : 0ull;
  const uint64_t exc = block_excl_scan(v, sc, &total);
  if (tid < nch) {
    w.chunk[4 * tid + 2] = (uint32_t)exc;
    w.chunk[4 * tid + 3] = (uint32_t)(exc >> 32);
  }
  if (tid == 0) {
    w.row[0] = T;
    w.row[1] = kr;
  }
}

__global__ void __launch_bounds__(kThreads) topk_wide_emit_kernel(const TopkParams p) {
  __shared__ uint32_t sc[256];
  pdl_launch_dependents();
  const int c = blockIdx.x, t = blockIdx.y, tid = threadIdx.x;
  pdl_wait();
  const int n = visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid);
  int32_t* out = p.idx + (int64_t)t * p.idx_ld;
  const int64_t seq = (t + p.t_off) / p.q_per_seq;
  const bool paged = p.pages.table != nullptr;
  const uint8_t* pf_kv = p.kv ? p.kv + (paged ? 0 : seq * p.kv_seq_stride) : nullptr;
  const uint8_t* pf_v = p.kv_v ? p.kv_v + (paged ? 0 : seq * p.v_seq_stride) : nullptr;
  auto prefetch_row = [&](uint32_t pos) {
    if (!pf_kv) return;
    const int64_t row = paged ? page_row(p.pages, seq, (int)pos) : (int64_t)pos;
    prefetch_l2(pf_kv + row * p.kv_row_stride, (uint32_t)p.kv_bytes);
    if (pf_v) prefetch_l2(pf_v + row * p.v_row_stride, (uint32_t)p.v_bytes);
  };
  const ChunkKeys ck(p, t, c, n);
  if (n <= p.K) {  // every visible position, in order, then -1
    for (int i = tid; i < ck.cnt; i += kThreads) {
      out[ck.lo + i] = ck.lo + i;
      prefetch_row((uint32_t)(ck.lo + i));
    }
    if (c == 0)
      for (int i = n + tid; i < p.K; i += kThreads) out[i] = -1;
    return;
  }
  const WideRow w = wide_row(p, t);
  const uint32_t T = __ldcg(w.row), take = __ldcg(w.row + 1);
  uint32_t gt_before = __ldcg(w.chunk + 4 * c + 2), eq_before = __ldcg(w.chunk + 4 * c + 3);
  for (int base = 0; base < ck.cnt; base += kChunk) {
    const int i = base + 4 * tid;
    uint32_t k[4];
    ck.load(i, k);
    uint32_t g = 0, q = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool ok = i + j < ck.cnt;
      g += ok && k[j] > T;
      q += ok && k[j] == T;
    }
    uint64_t tot;
    const uint64_t ex = block_excl_scan(((uint64_t)q << 32) | g, sc, &tot);
    uint32_t ga = gt_before + (uint32_t)ex, qa = eq_before + (uint32_t)(ex >> 32);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (i + j >= ck.cnt) break;
      const uint32_t pos = (uint32_t)(ck.lo + i + j);
      uint32_t slot = kNoBin;
      if (k[j] > T) {
        slot = ga + min(qa, take);
        ++ga;
      } else if (k[j] == T) {
        if (qa < take) slot = ga + qa;
        ++qa;
      }
      if (slot != kNoBin) {
        if (slot < (uint32_t)p.K) {  // always, when the counts of the row agree
          out[slot] = (int32_t)pos;
          prefetch_row(pos);
        } else {
          record_error(p.err, DSA_DEVERR_TOPK_COUNTS);
        }
      }
    }
    gt_before += (uint32_t)tot;
    eq_before += (uint32_t)(tot >> 32);
  }
}

// About kKeysPerCta keys per CTA, at most 16 CTAs per cluster; at most 8 when more clusters are
// needed than 16-CTA clusters can run at once.
int cluster_ctas(int n_max, int T, size_t smem16) {
  int c = 1;
  while (c < 16 && (int64_t)c * kKeysPerCta < n_max) c <<= 1;
  // Many queries in one launch (a prefill slice): the SMs are full of clusters either way, and a
  // CTA's fixed work (block scans over the histogram levels) dominates, so fewer, fuller CTAs per
  // query cost less: at most one per kManyKeysPerCta positions.  Prefill chunk of 4096 queries at
  // L = 128K: Top-K 4.91 -> 3.56 ms, step 13.6 -> 11.7 ms (clusters of 8 / 4 / 2 / 1 CTAs gave
  // 4.91 / 3.63 / 3.56 / 3.48 ms for the Top-K and 13.6 / 12.2 / 11.7 / 12.1 ms for the step).
  if (T >= kManyQueries) {
    int m = 1;
    while (m < c && (int64_t)m * kManyKeysPerCta < n_max) m <<= 1;
    return m;
  }
  if (c == 16) {
    static std::mutex mu;
    static size_t cached_smem = 0;
    static int cached_active = 0;
    int active = 0;
    {
      std::lock_guard<std::mutex> lock(mu);
      if (cached_smem == smem16) active = cached_active;
    }
    if (active == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16, 1);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem16;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 16;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&active, topk_cluster_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        active = 1;
      }
      std::lock_guard<std::mutex> lock(mu);
      cached_smem = smem16;
      cached_active = active;
    }
    if (T > active) c = 8;
  }
  return c;
}

}  // namespace

// Largest cluster a row of n_max positions can use (the launch may use fewer).
int cluster_ctas_max(int n_max) {
  int c = 1;
  while (c < 16 && (int64_t)c * kKeysPerCta < n_max) c <<= 1;
  return c;
}

size_t topk_cluster_ws_bytes(int T, int L) {
  return align_up((size_t)T * ws_words(cluster_ctas_max(L)) * sizeof(uint32_t), 256);
}

namespace {

// Row-split plan: rows longer than a 16-CTA cluster can keep in shared memory are cut into
// chunks of a multiple of kChunk positions, sized so that all rows together take about
// DSA_TOPK_WIDE_CTAS CTAs (a fixed figure, so that workspace sizing needs no device query).  Each
// CTA of the scan and emit kernels holds a whole SM (1024 threads x 64 registers), so fewer, longer
// chunks leave more SMs to other batches' kernels: one query at L = 1M, six batches in flight,
// 128 / 86 / 64 / 32 chunks gave 30.2 / 29.65 / 29.55 / 30.6 us per step, one batch at a time
// 59.3 / 59.4 / 60.4 / 67.4 us.
#ifndef DSA_TOPK_WIDE_CTAS
#define DSA_TOPK_WIDE_CTAS 100
#endif
struct WidePlan {
  bool use;
  int chunk, nch;
};

WidePlan wide_plan(int T, int L) {
  WidePlan w = {false, 0, 0};
  // (decode-sized batches only: the candidate lists take 8 bytes per position of every row)
  if (T <= 0 || T > 32 || (int64_t)L <= 16ll * kCachedKeys) return w;
  const int64_t target = T >= DSA_TOPK_WIDE_CTAS ? 1 : DSA_TOPK_WIDE_CTAS / T;  // chunks per row
  int64_t chunk = ((L + target - 1) / target + kChunk - 1) / kChunk * kChunk;
  while ((L + chunk - 1) / chunk > kWideMaxChunks) chunk += kChunk;
  w.use = true;
  w.chunk = (int)chunk;
  w.nch = (int)((L + chunk - 1) / chunk);
  return w;
}

template <typename Kern>
cudaError_t launch_plain(Kern kern, dim3 grid, const TopkParams& p, cudaStream_t stream, bool pdl) {
  return launch_kernel(kern, grid, dim3(kThreads), 0, stream, pdl, p);
}

cudaError_t launch_wide(TopkParams q, const WidePlan& w, cudaStream_t stream, bool pdl) {
  q.wide_chunk = w.chunk;
  q.wide_nch = w.nch;
  const dim3 chunks(w.nch, q.T);
  cudaError_t e = cudaSuccess;
  if (!q.hist) {
    e = launch_plain(topk_wide_hist_kernel, chunks, q, stream, pdl);
    pdl = true;
  }
  if (e == cudaSuccess) e = launch_plain(topk_wide_scan_kernel, chunks, q, stream, pdl);
  if (e == cudaSuccess) e = launch_plain(topk_wide_resolve_kernel, dim3(q.T), q, stream, true);
  if (e == cudaSuccess) e = launch_plain(topk_wide_emit_kernel, chunks, q, stream, true);
  return e;
}

}  // namespace

int topk_launches(int T, int L, bool hist_supplied) {
  if (T <= 0) return 0;
  return wide_plan(T, L).use ? (hist_supplied ? 3 : 4) : 1;
}

size_t topk_ws_bytes(int T, int L, int) {
  const size_t cl = topk_cluster_ws_bytes(T, L);
  const WidePlan w = wide_plan(T, L);
  if (!w.use) return cl;
  const size_t wide = align_up((size_t)T * wide_words(w.nch, w.chunk) * sizeof(uint32_t), 256);
  return wide > cl ? wide : cl;
}

cudaError_t launch_topk(const TopkParams& p, void* ws, cudaStream_t stream, bool pdl,
                        bool allow_wide) {
  if (p.T <= 0) return cudaSuccess;
  if (!ws) return cudaErrorInvalidValue;
  if (p.K > kMaxK) return cudaErrorNotSupported;
  TopkParams q = p;
  q.work = reinterpret_cast<uint32_t*>(ws);
  if (q.idx_ld <= 0) q.idx_ld = q.K;
  const WidePlan w = wide_plan(p.T, p.L);
  if (allow_wide && w.use) return launch_wide(q, w, stream, pdl);
  auto kern = topk_cluster_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  const size_t smem16 = (size_t)TopkSmem(slice_of(p.L, 16)).words * 4;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem16);
  if (e != cudaSuccess) return e;
  const int C = cluster_ctas(p.L, p.T, smem16);
  const size_t smem = (size_t)TopkSmem(slice_of(p.L, C)).words * 4;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
// Context split over G slices (a query's positions cut into G ranges, e.g. one per GPU).  Every
// position of the global Top-K is among the Top-K of its own slice, so the global selection is the
// Top-K of the union of the slices' selections, taken in the same order (score descending, exact
// ties toward the lower position).  Each slice turns its selection into (score, position) pairs
// (topk_pairs_kernel), the pairs of all slices are put side by side, and topk_merge_kernel selects
// K of them.

namespace {

constexpr int kMergePer = 16;                    // candidates per thread
constexpr int kMergeMax = kThreads * kMergePer;  // candidates per query

// After the slice's Top-K wrote local positions into cand_pos: the score of each selected position
// into cand_scores, and the position moved by the slice's first position (-1 entries stay -1).
__global__ void __launch_bounds__(256) topk_pairs_kernel(const PairsParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= p.K) return;
  int32_t* cp = p.cand_pos + (int64_t)t * p.ld_cand + j;
  const int32_t pos = *cp;
  float s = 0.f;
  if (pos >= 0) {
    s = p.scores[(int64_t)t * p.ld_scores + pos];
    *cp = pos + p.pos_offset;
  }
  p.cand_scores[(int64_t)t * p.ld_cand + j] = s;
}

// The key T and the count `take` with (entries above T) + take = kr, over the entries of this
// thread marked in `mask` (all threads together hold at least kr of them).  Radix levels of 12, 10
// and 10 bits with shared-memory histograms.
__device__ uint32_t merge_threshold(const uint32_t (&k)[kMergePer], uint32_t mask, uint32_t kr,
                                    uint32_t* hist, uint32_t* sc, uint32_t* take) {
  for (int b = threadIdx.x; b < kHistBins; b += kThreads) hist[b] = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kMergePer; ++i)
    if ((mask >> i) & 1u) atomicAdd(&hist[k[i] >> 20], 1u);
  __syncthreads();
  uint32_t c0[kBins0];
#pragma unroll
  for (int j = 0; j < kBins0; ++j) c0[j] = hist[kBins0 * threadIdx.x + j];
  uint32_t above;
  uint32_t prefix = find_digit<kBins0>(c0, kr, sc, &above);  // ends with a barrier: hist is free
  kr -= above;
#pragma unroll 1
  for (int lv = 0; lv < 2; ++lv) {
    const int shift = 10 - 10 * lv;  // the digit: bits 19..10, then 9..0
    for (int b = threadIdx.x; b < kLevelBins; b += kThreads) hist[b] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kMergePer; ++i)
      if (((mask >> i) & 1u) && (k[i] >> (shift + 10)) == prefix)
        atomicAdd(&hist[(k[i] >> shift) & (kLevelBins - 1)], 1u);
    __syncthreads();
    uint32_t c1[kBins1];
#pragma unroll
    for (int j = 0; j < kBins1; ++j) c1[j] = hist[kBins1 * threadIdx.x + j];
    const uint32_t d = find_digit<kBins1>(c1, kr, sc, &above);
    kr -= above;
    prefix = (prefix << 10) | d;
  }
  *take = kr;
  return prefix;
}

// One CTA per query; thread i holds candidates [i * per, i * per + per) of the query's list.
__global__ void __launch_bounds__(kThreads, 1) topk_merge_kernel(const MergeParams p) {
  __shared__ uint32_t hist[kHistBins];
  __shared__ uint32_t sc[256];
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x, tid = threadIdx.x;
  const int n_cand = p.parts * p.per_part;
  int32_t* out = p.idx + (int64_t)t * p.K;
  const int per = (n_cand + kThreads - 1) / kThreads;
  const int lo = tid * per;
  // element offset of candidate j of this query
  auto at = [&](int j) -> int64_t {
    const int g = j / p.per_part;
    return (int64_t)g * p.part_stride + (int64_t)t * p.ld + (j - g * p.per_part);
  };
  const float* s = p.scores;
  const int32_t* ps = p.pos;
  uint32_t k[kMergePer];
  uint32_t valid = 0;
#pragma unroll
  for (int i = 0; i < kMergePer; ++i) {
    k[i] = 0u;
    const int j = lo + i;
    if (i < per && j < n_cand && __ldg(ps + at(j)) >= 0) {
      k[i] = float_key(__ldg(s + at(j)));
      valid |= 1u << i;
    }
  }
  uint64_t tot;
  block_excl_scan((uint64_t)__popc(valid), sc, &tot);
  uint32_t sel = valid;
  if (tot > (uint64_t)p.K) {
    uint32_t take;
    const uint32_t T = merge_threshold(k, valid, (uint32_t)p.K, hist, sc, &take);
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int i = 0; i < kMergePer; ++i) {
      const bool v = (valid >> i) & 1u;
      gt |= (uint32_t)(v && k[i] > T) << i;
      eq |= (uint32_t)(v && k[i] == T) << i;
    }
    block_excl_scan((uint64_t)__popc(eq), sc, &tot);
    sel = gt;
    if ((uint64_t)take == tot) {
      sel |= eq;
    } else {
      // the `take` lowest positions among the entries equal to T: the take largest of ~position
#pragma unroll
      for (int i = 0; i < kMergePer; ++i) k[i] = ((eq >> i) & 1u) ? ~(uint32_t)__ldg(ps + at(lo + i)) : 0u;
      uint32_t take2;
      const uint32_t P = merge_threshold(k, eq, take, hist, sc, &take2);
#pragma unroll
      for (int i = 0; i < kMergePer; ++i) sel |= (uint32_t)(((eq >> i) & 1u) && k[i] >= P) << i;
    }
  }
  // kept candidates in list order, then -1
  const uint32_t ex = (uint32_t)block_excl_scan((uint64_t)__popc(sel), sc, &tot);
  uint32_t slot = ex;
#pragma unroll
  for (int i = 0; i < kMergePer; ++i)
    if ((sel >> i) & 1u) {
      if (slot < (uint32_t)p.K) out[slot] = __ldg(ps + at(lo + i));  // (duplicate positions: extra dropped)
      ++slot;
    }
  for (int j = (int)min(tot, (uint64_t)p.K) + tid; j < p.K; j += kThreads) out[j] = -1;
}

}  // namespace

int topk_merge_max_candidates() { return kMergeMax; }

cudaError_t launch_topk_pairs(const TopkParams& p, void* ws, const PairsParams& pp, cudaStream_t stream) {
  cudaError_t e = launch_topk(p, ws, stream, false);
  if (e != cudaSuccess || p.T <= 0) return e;
  return launch_kernel(topk_pairs_kernel, dim3((pp.K + 255) / 256, pp.T), dim3(256), 0, stream, true, pp);
}

cudaError_t launch_topk_merge(const MergeParams& p, cudaStream_t stream, bool pdl) {
  if (p.T <= 0) return cudaSuccess;
  if ((int64_t)p.parts * p.per_part > kMergeMax || p.K > kMaxK) return cudaErrorNotSupported;
  return launch_kernel(topk_merge_kernel, dim3(p.T), dim3(kThreads), 0, stream, pdl, p);
}

// ---------------------------------------------------------------------------------------------
// Top-K without a caller workspace.
//
// Some callers cannot hand the library device memory: a host framework that owns every device
// allocation through its own pool and forbids raw cudaMalloc, or a decode loop that must not
// allocate while it runs (an allocation can synchronise the device and fragment memory).  For
// them dsa_topk_noalloc keeps the Top-K exchange areas (histograms, counts, candidate lists) in
// the file-scope array below, sized for kNoAllocMaxQueries queries.  Every GPU that loads the
// library holds these bytes until the process exits.

constexpr int kNoAllocMaxQueries = 16;
constexpr int64_t kNoAllocWords = kNoAllocMaxQueries * (kWsList + 2 * 16 * kRegion);
static __device__ __align__(256) uint32_t g_topk_scratch[kNoAllocWords];

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
  if (cudaMemsetAsync(scratch, 0, topk_cluster_ws_bytes(T, L), st) != cudaSuccess)
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
  return launch_topk(p, scratch, st, false, /*allow_wide=*/false) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
