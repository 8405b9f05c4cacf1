// Step 1 of the chain: indexer relevance scores,
//   I[t, s] = sum_h w[t, h] * ReLU(q_idx[t, h, :] . k_idx[s, :])
// (scoring each position, then weighting the heads: Day 0 Support for New LLM Architectures,
// Key Optimization 1; MXFP8 index path with groups of 32 sharing a scale, Key Optimization 2).
//
// The contraction runs on the 5th-generation tensor cores: a tile of 128 cache positions is the
// M = 128 side of tcgen05.mma (A = k_idx rows, K-major, streamed by TMA with 128-byte swizzle),
// the G queries x H_idx heads of one query group are the N side (B = q_idx rows, staged once per
// group), and the fp32 accumulator lives in tensor memory.  Each epilogue thread owns one TMEM
// lane = one position and all of its head columns, so ReLU, the head weights and (for MXFP8) the
// per-group E8M0 scales are applied in registers with no cross-thread reduction.
//
// Warp roles: warp 0 = producer (TMA for A and B), warp 1 = TMEM owner and MMA issuer, the rest
// epilogue.  One-query tiles have two epilogue groups of four warps that take alternate tiles,
// so two tiles' epilogues (TMEM loads, stores, histogram) overlap; the four-query prefill tiles
// (N = 256) use four groups that split each tile by query.  A ring of shared-memory stages
// decouples loads from MMAs; four TMEM accumulators let the epilogue trail the MMAs.
// The grid is persistent: CTA c processes a contiguous range of (query group, tile) units.
//
// For the Top-K step, the epilogue also builds a histogram of the top 12 bits of each score's
// order-preserving key (shared memory, flushed to a per-query global histogram with atomics on
// non-zero bins), so selection starts with its first digit pass done.
//
// MXFP8: the tensor cores apply the scales.  One block-scaled kind::mxf8f6f4 MMA covers K = 32 =
// one scale group, and reads each key row's and each head's E8M0 exponent for that group from
// tensor memory, so a tile accumulates  sum_g 2^(ea_g + eb_g - 254) D_g  into one accumulator and
// the epilogue is the bf16 one.  The epilogue warps write the scale words into tensor memory
// (one slot per accumulator, a full pipeline depth ahead of the tile they read).
#include <string.h>

#include <utility>

#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kTileM = 128;
// When a CTA signals the next kernel of the chain (griddepcontrol.launch_dependents): 1 when its
// tiles are done, 0 right after its setup.  Signalling late keeps the dependent's CTAs from taking
// SMs long before they can start (decode B = 8, L = 32K, one batch at a time: the three kernels
// signalling late took the step from 43.5 to 41.8 us for bf16 and from 49.6 to 46.3 us for MXFP8;
// six batches in flight: unchanged within 1 %).
// Inside the fused chain a long one-query launch takes this many quarters of the two-CTA slots, so
// that the next batch's scoring starts while this one streams (its ramp, about 3 us to the first
// tile, overlaps): L = 1M, six batches in flight, 4 / 3 / 2 quarters gave 29.8 / 28.5 / 27.7 us
// per step, one batch at a time 59.1 / 65.7 / 72.2 us.
#ifndef DSA_IDX_LONG_SLOTS_Q
#define DSA_IDX_LONG_SLOTS_Q 3
#endif
#ifndef DSA_PDL_LATE_IDX
#define DSA_PDL_LATE_IDX 1
#endif
constexpr int kSmemBudget = 225 * 1024;  // per SM

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

template <bool MX, int D, int G, int NPAD>
struct Cfg {
  static constexpr int ELEM = MX ? 1 : 2;
  static constexpr int ROW_BYTES = D * ELEM;
  static constexpr int BOXES = ROW_BYTES / 128;  // 128-byte swizzle atoms per row
  static constexpr int BOX_COLS = 128 / ELEM;
  static constexpr int KSTEPS = ROW_BYTES / 32;  // MMAs per tile (32 bytes of K each)
  static constexpr int N = G * NPAD;              // MMA N
  static constexpr int A_BYTES = kTileM * ROW_BYTES;
  static constexpr int B_BYTES = N * ROW_BYTES;
  static constexpr int B_BUFS = (G == 1 && !MX) ? 1 : ((2 * B_BYTES <= 64 * 1024) ? 2 : 1);
  static constexpr int GROUPS = MX ? D / 32 : 1;  // scale groups per row (MMAs per tile)
  // One-query tiles run two CTAs per SM: each CTA's pipeline spends much of its time in the
  // handshakes between stage ring, accumulators and epilogue, and a second CTA fills those gaps
  // (MXFP8, B = 1, L = 1M: 36.8 -> 25.4 us; bf16, B = 8, L = 32K: 15.1 -> 13.8 us, with two
  // 32 KB stages and one query buffer per CTA).  Four-query prefill tiles keep one CTA per SM.
  static constexpr int CTAS_PER_SM = G == 1 ? 2 : 1;
  static constexpr int ACC_COLS = N;
  // accumulators in flight between the MMA warp and the epilogue: as many as fit in 512 columns,
  // up to 4 (two were not enough to hide MMA completion + epilogue latency per tile)
  static constexpr int ACC_BUFS = CTAS_PER_SM == 2 ? 2 : (512 / ACC_COLS >= 4 ? 4 : 2);
  // MXFP8 scale slots after the accumulators, 16 columns each: A scales (4 copies of the row's
  // scale word, so that quarter q finds it in column q) and, 8 columns in, B scales (one
  // column per 32 heads, repeated in every lane quarter)
  static constexpr int SF_BASE = ACC_BUFS * ACC_COLS;
  static constexpr int SF_COLS = MX ? 16 * ACC_BUFS : 0;
  static constexpr int TMEM_COLS = pow2_at_least(SF_BASE + SF_COLS);
  static constexpr int HIST_BYTES = G == 1 ? kHistBins * 4 : 0;  // fused score histogram
  // epilogue groups of four warps (each group covers all 128 rows of a tile): SPLITS groups
  // split a tile's columns by query, TG sets of them take alternate tiles
  static constexpr int SPLITS = G;
  static constexpr int TG = (G == 1 && CTAS_PER_SM == 1) ? 2 : 1;
  static constexpr int EPI = 4 * SPLITS * TG;  // epilogue warps
  static constexpr int THREADS = 64 + 32 * EPI;
  static constexpr int COLS = N / SPLITS;     // accumulator columns per epilogue warp (= NPAD)
  static constexpr int AUX_BYTES = 1024 + 4096 + G * NPAD * 4 + HIST_BYTES;
  static constexpr int STAGES_FIT = (kSmemBudget / CTAS_PER_SM - B_BUFS * B_BYTES - AUX_BYTES - 1024) / A_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int OFF_B = STAGES * A_BYTES;
  static constexpr int OFF_BAR = OFF_B + B_BUFS * B_BYTES;
  static constexpr int OFF_W = OFF_BAR + 1024;
  static constexpr int OFF_HIST = OFF_W + G * NPAD * 4;
  static constexpr int SMEM = OFF_HIST + HIST_BYTES + 1024;  // + alignment slack
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "MMA N out of range");
  static_assert(TMEM_COLS * CTAS_PER_SM <= 512, "accumulators exceed tensor memory");
  static_assert(SMEM * CTAS_PER_SM <= 228 * 1024, "shared memory exceeds the SM");
  static_assert(!MX || (G == 1 && (N == 32 || N == 64) && GROUPS <= 4), "MXFP8 tile shape");
  static_assert(STAGES >= 2, "not enough shared memory for the pipeline");
  static_assert(ROW_BYTES % 128 == 0, "rows must fill whole swizzle atoms");
  static_assert(ACC_BUFS % TG == 0, "alternate tiles need an even number of accumulators");
  static_assert(COLS >= 8, "at least one 8-column TMEM load per warp");
};

// named barrier of the epilogue warps (id 1; 0 is __syncthreads)
template <int THREADS>
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory"); }

// Walks this CTA's share of the visible (query group, tile) units, in order.  A unit is visible
// when its tile holds a position that some query of the group sees (a prefix of the group's
// tiles).  The visible units are numbered group by group and CTA b of B takes numbers
// [V*b/B, V*(b+1)/B) of the V in total, so the CTAs get equal work whatever the queries' lengths
// (a batch of sequences of different lengths, or the causal rows of a prefill chunk).  Group facts
// (visible lengths, cache sequence) are computed on entering a group; a step costs no division.
template <int G>
struct UnitWalk {
  int left;  // units of this CTA still to visit
  int g, tile, vt, n_max, seq;
  int n[G];  // visible length of each query of the group (0 past the last query)

  __device__ __forceinline__ static int visible_tiles(const IndexScoreParams& p, int g) {
    int m = 0;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int t = g * G + j;
      if (t < p.T) m = max(m, visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid));
    }
    return min(p.tiles, (m + kTileM - 1) / kTileM);
  }
  __device__ __forceinline__ void enter_group(const IndexScoreParams& p) {
    n_max = 0;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int t = g * G + j;
      n[j] = t < p.T ? visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid) : 0;
      n_max = max(n_max, n[j]);
    }
    vt = min(p.tiles, (n_max + kTileM - 1) / kTileM);
    seq = (g * G + p.t_off) / p.q_per_seq;
  }
  // starts at visible unit `first` of group g0 (acc = visible units before g0), `count` units
  __device__ __forceinline__ UnitWalk(const IndexScoreParams& p, const int* share) {
    g = share[0];
    left = share[2];
    enter_group(p);
    tile = share[1] - 1;  // one step before this CTA's first unit
  }
  // advances to the next unit; false when this CTA's share is done
  __device__ __forceinline__ bool next(const IndexScoreParams& p) {
    if (left <= 0) return false;
    --left;
    if (++tile >= vt) {
      do {  // a later group with a visible tile exists while units are left
        ++g;
        enter_group(p);
      } while (vt == 0);
      tile = 0;
    }
    return true;
  }
  __device__ __forceinline__ int t0() const { return g * G; }
};

// This CTA's share of the visible units, found by one warp: lane l sums the visible tiles of a
// contiguous block of groups, a warp scan gives the total V and each block's start, and the lane
// whose block holds unit V*b/B walks it to the exact group.  share = {group, first visible tile
// in it, units to visit}.
template <int G>
__device__ __forceinline__ void unit_share(const IndexScoreParams& p, int* share) {
  const int lane = threadIdx.x & 31;
  const int n_groups = (p.T + G - 1) / G;
  if (p.q_pos0 < 0 && p.n_valid == nullptr) {
    // every query sees all L positions: every group has the same `tiles` visible units, so the
    // share is a closed form (32-bit arithmetic when V * gridDim.x fits)
    if (lane == 0) {
      const uint32_t vt = (uint32_t)p.tiles, B = gridDim.x, b = blockIdx.x;
      const uint64_t V = (uint64_t)n_groups * vt;
      uint32_t b0, b1;
      if (V * B < (1ull << 32)) {
        b0 = (uint32_t)V * b / B;
        b1 = (uint32_t)V * (b + 1) / B;
      } else {
        b0 = (uint32_t)(V * b / B);
        b1 = (uint32_t)(V * (b + 1) / B);
      }
      const uint32_t g = vt ? b0 / vt : 0;
      share[0] = (int)min(g, (uint32_t)max(n_groups - 1, 0));
      share[1] = (int)(b0 - g * vt);
      share[2] = (int)(b1 - b0);
    }
    return;
  }
  const int g_lo = (int)((int64_t)n_groups * lane / 32), g_hi = (int)((int64_t)n_groups * (lane + 1) / 32);
  int64_t mine = 0;
  for (int g = g_lo; g < g_hi; ++g) mine += UnitWalk<G>::visible_tiles(p, g);
  int64_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int64_t V = __shfl_sync(0xffffffffu, incl, 31);
  const int64_t b0 = V * blockIdx.x / gridDim.x, b1 = V * (blockIdx.x + 1) / gridDim.x;
  const int64_t before = incl - mine;  // visible units before this lane's block
  // the lane whose block holds unit b0 (the last lane when b0 == V)
  const bool holds = (b0 >= before && b0 < incl) || (lane == 31 && b0 >= incl);
  const uint32_t m = __ballot_sync(0xffffffffu, holds);
  if (lane == __ffs(m) - 1) {
    int g = g_lo;
    int64_t acc = before;
    for (; g < g_hi - 1; ++g) {
      const int v = UnitWalk<G>::visible_tiles(p, g);
      if (acc + v > b0) break;
      acc += v;
    }
    if (g_hi <= g_lo) g = min(g_lo, n_groups - 1);  // an empty block (more lanes than groups)
    share[0] = g;
    share[1] = (int)(b0 - acc);
    share[2] = (int)(b1 - b0);
  }
}

template <bool MX, int D, int G, int NPAD>
__global__ void __launch_bounds__(Cfg<MX, D, G, NPAD>::THREADS, Cfg<MX, D, G, NPAD>::CTAS_PER_SM)
index_score_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const uint8_t* __restrict__ q_idx, const int q_by_tma, const IndexScoreParams p) {
  using C = Cfg<MX, D, G, NPAD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* a_s = smem;
  uint8_t* b_s = smem + C::OFF_B;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* bfull = empty + C::STAGES;
  uint64_t* bempty = bfull + 2;
  uint64_t* tfull = bempty + 2;
  uint64_t* tempty = tfull + 4;
  uint64_t* sf_full = tempty + 4;  // MXFP8 scale slot written (one arrival per epilogue warp)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + 4);
  int* share = reinterpret_cast<int*>(tmem_slot + 1);  // [3]: this CTA's units (unit_share)
  float* w_s = reinterpret_cast<float*>(smem + C::OFF_W);    // [G][NPAD]
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + C::OFF_HIST);  // G == 1 only
  const bool build_hist = G == 1 && p.hist != nullptr;

  const int warp = warp_id();
  const int lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < C::ACC_BUFS; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4 * C::SPLITS);  // one arrival per warp that reads the tile
      mbar_init(&sf_full[i], 4);              // one arrival per warp of the writing group
    }
    fence_mbar_init();
    prefetch_tmap(&tm_k);
    if (q_by_tma) prefetch_tmap(&tm_q);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    pdl_wait();  // the per-query lengths may come from the previous kernel in the stream
    unit_share<G>(p, share);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // let the next kernel in the stream launch now: its CTAs take SMs as this grid's CTAs retire
  // and wait (griddepcontrol.wait) for this grid's results before reading them
  if (!DSA_PDL_LATE_IDX) pdl_launch_dependents();
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const uint64_t evict_first = l2_evict_first_policy();  // key tiles are read once
    int it = 0, qn = -1, cur_t0 = -1;
    bool ok = true;
    UnitWalk<G> w(p, share);
    // paged caches: a tile is two 64-row halves, each inside one block; lane i holds the pool
    // rows of the halves of the i-th of the next 32 units (looked up 32 units at a time, one
    // memory round trip), or kNoRow for a half past the group's longest visible row
    constexpr uint32_t kNoRow = 0xFFFFFFFFu;
    const bool paged = p.pages.table != nullptr;
    UnitWalk<G> look(p, share);
    uint32_t pr0 = kNoRow, pr1 = kNoRow;
    int nb = 32;
    while (ok && w.next(p)) {
      uint32_t row0 = 0, row1 = kNoRow;
      if (paged) {
        if (nb == 32) {
          UnitWalk<G> c = look;
          bool have = true;
          for (int q = 0; q <= lane && have; ++q) have = c.next(p);
          pr0 = pr1 = kNoRow;
          if (have) {
            const int pos = c.tile * kTileM;
            pr0 = (uint32_t)page_row(p.pages, c.seq, pos);
            if (pos + 64 < c.n_max) pr1 = (uint32_t)page_row(p.pages, c.seq, pos + 64);
          }
          for (int q = 0; q < 32; ++q) look.next(p);  // every lane moves the same 32 units on
          nb = 0;
        }
        row0 = __shfl_sync(0xffffffffu, pr0, nb);
        row1 = __shfl_sync(0xffffffffu, pr1, nb);
        ++nb;
      }
      if (w.t0() != cur_t0) {
        cur_t0 = w.t0();
        ++qn;
        const int bb = qn % C::B_BUFS;
        if (qn >= C::B_BUFS) ok = mbar_wait(&bempty[bb], ((qn - C::B_BUFS) / C::B_BUFS) & 1, p.err);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        uint8_t* bdst = b_s + bb * C::B_BYTES;
        if (q_by_tma) {
          // B tile = q_idx rows t0*H_idx .. t0*H_idx + N - 1 (G*NPAD rows; rows past the last query
          // arrive zero-filled; rows of a following query meet zero head weights)
          if (lane == 0) {
            mbar_arrive_expect_tx(&bfull[bb], C::B_BYTES);
#pragma unroll
            for (int b = 0; b < C::BOXES; ++b)
              tma_load_2d(bdst + b * (C::N * 128), &tm_q, &bfull[bb], b * C::BOX_COLS, w.t0() * p.H_idx);
          }
          __syncwarp();
        } else {
          // few query rows: rows j*NPAD + h <- q_idx row (t0 + j) * H_idx + h, zero past H_idx / T,
          // written in the 128-byte swizzled K-major layout the MMA descriptor expects
          constexpr int CH = C::ROW_BYTES / 16;
          for (int i = lane; i < C::N * CH; i += 32) {
            const int r = i / CH, c = i % CH;
            const int j = r / NPAD, h = r % NPAD;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < p.H_idx && w.t0() + j < p.T)
              v = *reinterpret_cast<const uint4*>(q_idx + ((int64_t)(w.t0() + j) * p.H_idx + h) * C::ROW_BYTES + c * 16);
            const int box = c >> 3, cc = c & 7;
            *reinterpret_cast<uint4*>(bdst + box * (C::N * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bfull[bb]);
        }
      }
      const int s = it % C::STAGES;
      if (it >= C::STAGES) ok = mbar_wait(&empty[s], ((it / C::STAGES) - 1) & 1, p.err);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        if (!paged) {
          mbar_arrive_expect_tx(&full[s], C::A_BYTES);
#pragma unroll
          for (int b = 0; b < C::BOXES; ++b)
            tma_load_3d_hint(a_s + s * C::A_BYTES + b * (kTileM * 128), &tm_k, &full[s], b * C::BOX_COLS,
                             w.tile * kTileM, w.seq, evict_first);
        } else {
          // a half past the visible rows is not loaded: its MMA rows hold stale data and are
          // never scored (every accumulator row depends on its own A row only)
          const int halves = row1 == kNoRow ? 1 : 2;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(halves * C::A_BYTES / 2));
#pragma unroll
          for (int b = 0; b < C::BOXES; ++b) {
            uint8_t* dst = a_s + s * C::A_BYTES + b * (kTileM * 128);
            tma_load_2d_hint(dst, &tm_k, &full[s], b * C::BOX_COLS, (int)row0, evict_first);
            if (halves == 2) tma_load_2d_hint(dst + 64 * 128, &tm_k, &full[s], b * C::BOX_COLS, (int)row1, evict_first);
          }
        }
      }
      if constexpr (MX) {
        // the tile's key-scale words (4 bytes per row; 32 rows per lane, inside one cache block)
        // into L2 now: the epilogue loads them a stage ring later, and an L2 hit keeps that
        // load off its per-tile path
        const int pos = w.tile * kTileM + 32 * lane;
        if (lane < kTileM / 32 && pos < w.n_max) {
          const uint8_t* a = paged ? p.k_sf + page_row(p.pages, w.seq, pos) * 4
                                   : p.k_sf + (int64_t)w.seq * p.k_sf_seq_stride + (int64_t)pos * 4;
          const int last = min(32, w.n_max - pos) * 4 - 4;
          prefetch_line_l2(a);
          prefetch_line_l2(a + last);
        }
      }
      __syncwarp();
      ++it;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = make_idesc(1, 1, kTileM, C::N);
    int it = 0, qn = -1, cur_t0 = -1, ai = 0;
    bool ok = true;
    UnitWalk<G> w(p, share);
    while (ok && w.next(p)) {
      if (w.t0() != cur_t0) {
        if (qn >= 0 && lane == 0) tc_commit(&bempty[qn % C::B_BUFS]);
        cur_t0 = w.t0();
        ++qn;
        ok = __all_sync(0xffffffffu, mbar_wait(&bfull[qn % C::B_BUFS], (qn / C::B_BUFS) & 1, p.err));
        if (!ok) break;
      }
      const int s = it % C::STAGES;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (it / C::STAGES) & 1, p.err));
      const int ab = ai % C::ACC_BUFS;
      if (ok && ai >= C::ACC_BUFS)
        ok = __all_sync(0xffffffffu, mbar_wait(&tempty[ab], ((ai - C::ACC_BUFS) / C::ACC_BUFS) & 1, p.err));
      if (MX && ok) ok = __all_sync(0xffffffffu, mbar_wait(&sf_full[ab], (ai / C::ACC_BUFS) & 1, p.err));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a_base = smem_u32(a_s + s * C::A_BYTES);
        const uint32_t b_base = smem_u32(b_s + (qn % C::B_BUFS) * C::B_BYTES);
        const uint32_t d0 = tmem + ab * C::ACC_COLS;
        const uint32_t sf = tmem + C::SF_BASE + 16 * ab;  // this tile's scale slot (MXFP8)
#pragma unroll
        for (int k = 0; k < C::KSTEPS; ++k) {
          const int box = k >> 2, off = (k & 3) * 32;
          const uint64_t ad = smem_desc_sw128(a_base + box * (kTileM * 128) + off);
          const uint64_t bd = smem_desc_sw128(b_base + box * (C::N * 128) + off);
          if (MX)  // K step k = scale group k: byte k of the scale words
            mma_mxf8(d0, ad, bd, make_idesc_mx(kTileM, C::N, k, k), sf, sf + 8, k > 0 ? 1u : 0u);
          else
            mma_f16(d0, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        tc_commit(&empty[s]);
        tc_commit(&tfull[ab]);
      }
      __syncwarp();
      ++it;
      ++ai;
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    constexpr int ET = 32 * C::EPI;  // epilogue threads
    const int q4 = warp & 3;         // the TMEM lane quarter this warp may access
    const int grp = (warp - 2) >> 2;
    const int half = grp % C::SPLITS;  // which query of the tile this warp scores
    const int tg = grp / C::SPLITS;    // which of the alternate tiles this warp takes
    const int row = q4 * 32 + lane;
    const int et = threadIdx.x - 64;
    int ai = 0, cur_t0 = -1;
    bool ok = true;
    // flushes the shared histogram of query t into the global one and clears it: 16-byte reads
    // (all of a thread's in flight at once), then one 64-bit atomic add per pair of bins with a
    // non-zero count (the low word of a pair never carries: a row has fewer than 2^32 positions)
    auto flush_hist = [&](int t) {
      static_assert(kHistBins % (4 * ET) == 0, "whole 16-byte groups of bins per thread");
      constexpr int NV = kHistBins / (4 * ET);
      uint4* h4 = reinterpret_cast<uint4*>(hist_s);
      unsigned long long* g2 = reinterpret_cast<unsigned long long*>(p.hist + (int64_t)t * kHistBins);
      uint4 v[NV];
#pragma unroll
      for (int k = 0; k < NV; ++k) v[k] = h4[et + k * ET];
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int pair = 2 * (et + k * ET);  // bins 2 pair .. 2 pair + 3
        if (v[k].x | v[k].y) atomicAdd(g2 + pair, (unsigned long long)v[k].y << 32 | v[k].x);
        if (v[k].z | v[k].w) atomicAdd(g2 + pair + 1, (unsigned long long)v[k].w << 32 | v[k].z);
        h4[et + k * ET] = make_uint4(0u, 0u, 0u, 0u);
      }
    };
    if (build_hist)
      for (int b = et; b < kHistBins; b += ET) hist_s[b] = 0;
    // MXFP8 scale writer.  The n-th visible unit's scale words go to slot n % ACC_BUFS, a full
    // pipeline depth ahead of the accumulator the epilogue reads, written by the group that takes
    // that unit (n % TG); a unit's key-scale word is loaded when the group's previous unit is
    // written, so the global load overlaps a tile's epilogue.  Each lane writes its lane of the
    // warp's quarter: its row's four group exponents (byte g = group g) into the four A columns,
    // and those of heads (lane) and (32 + lane) of the unit's query into the two B columns.
    UnitWalk<G> sfw(p, share);
    bool sf_more = false;
    int sf_n = 0, sf_t = -1;
    uint32_t sf_a = 0, sf_b0 = 0, sf_b1 = 0;
    auto sf_load_a = [&]() -> uint32_t {
      const int pos = sfw.tile * kTileM + row;
      if (pos >= sfw.n_max) return 0x7F7F7F7Fu;  // a row that is not scored: any finite scale
      if (p.pages.table)
        return __ldg(reinterpret_cast<const uint32_t*>(p.k_sf + page_row(p.pages, sfw.seq, pos) * 4));
      return __ldg(reinterpret_cast<const uint32_t*>(p.k_sf + (int64_t)sfw.seq * p.k_sf_seq_stride + (int64_t)pos * 4));
    };
    auto q_word = [&](int t, int h) -> uint32_t {
      if (h >= p.H_idx || t >= p.T) return 0x7F7F7F7Fu;  // padding heads meet zero weights
      const uint8_t* q = p.q_sf + ((int64_t)t * p.H_idx + h) * 4;
      return (uint32_t)q[0] | (uint32_t)q[1] << 8 | (uint32_t)q[2] << 16 | (uint32_t)q[3] << 24;
    };
    auto sf_step = [&]() {  // cursor to the next visible unit
      sf_more = sfw.next(p);
      ++sf_n;
    };
    auto sf_write = [&]() {
      const int slot = sf_n % C::ACC_BUFS;
      if (sfw.t0() != sf_t) {
        sf_t = sfw.t0();
        sf_b0 = q_word(sf_t, lane);
        sf_b1 = q_word(sf_t, 32 + lane);
      }
      const uint32_t addr = tmem + ((uint32_t)(q4 * 32) << 16) + C::SF_BASE + 16 * slot;
      tmem_st_x4(addr, sf_a, sf_a, sf_a, sf_a);
      tmem_st_x2(addr + 8, sf_b0, sf_b1);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_full[slot]);
      for (int k = 0; k < C::TG && sf_more; ++k) sf_step();  // this group's next unit
      if (sf_more) sf_a = sf_load_a();
    };
    if constexpr (MX) {
      sf_more = sfw.next(p);
      for (int k = 0; k < tg && sf_more; ++k) sf_step();
      if (sf_more) sf_a = sf_load_a();
      while (sf_more && sf_n < C::ACC_BUFS) sf_write();
    }
    // after a timed-out wait the epilogue warps keep walking the units (so that every named
    // barrier below is reached by every epilogue thread) but skip the waits and the tile work
    UnitWalk<G> w(p, share);
    while (w.next(p)) {
      if (w.t0() != cur_t0) {
        epi_bar<ET>();
        if (build_hist && cur_t0 >= 0) {
          flush_hist(cur_t0);
          epi_bar<ET>();
        }
        cur_t0 = w.t0();
        for (int i = et; i < G * NPAD; i += ET) {
          const int j = i / NPAD, h = i % NPAD;
          const bool valid = h < p.H_idx && w.t0() + j < p.T;
          w_s[i] = valid ? p.w[(int64_t)(w.t0() + j) * p.H_idx + h] : 0.f;
        }
        epi_bar<ET>();
      }
      if (ai % C::TG != tg) {  // the other group's tile
        ++ai;
        continue;
      }
      const int pos = w.tile * kTileM + row;
      const int ab = ai % C::ACC_BUFS;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&tfull[ab], (ai / C::ACC_BUFS) & 1, p.err));
      float score = 0.f;  // this warp's query: the group's query `half`
      if (ok) {
        tc_fence_after();
        // this slot's MMAs are complete: its scale slot takes the unit ACC_BUFS ahead
        if (MX && sf_more) sf_write();
        const uint32_t tb = tmem + ((uint32_t)(q4 * 32) << 16) + ab * C::ACC_COLS;
        constexpr int CW = C::COLS < 32 ? C::COLS : 32;  // columns per TMEM load
#pragma unroll
        for (int c = 0; c < C::COLS / CW; ++c) {
          const int col = half * C::COLS + c * CW;  // first accumulator column of this load
          float v[CW];
          tmem_ld_sync(tb + col, v);
          // columns in pairs: packed fp32x2 multiply-adds (same rounding as scalar fp32)
          float2 sc2 = make_float2(0.f, 0.f);
          const float4* wv = reinterpret_cast<const float4*>(w_s + col);
#pragma unroll
          for (int i = 0; i < CW / 4; ++i) {
            const float4 w4 = wv[i];
            sc2 = ffma2(make_float2(w4.x, w4.y), make_float2(fmaxf(v[4 * i], 0.f), fmaxf(v[4 * i + 1], 0.f)), sc2);
            sc2 = ffma2(make_float2(w4.z, w4.w), make_float2(fmaxf(v[4 * i + 2], 0.f), fmaxf(v[4 * i + 3], 0.f)), sc2);
          }
          score += sc2.x + sc2.y;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[ab]);
        const bool vis = pos < w.n[half];  // zero past the last query
        if (vis) p.scores[(int64_t)(w.t0() + half) * p.ld_scores + pos] = score;
        // shared-memory atomics: lanes on the same bin serialise in the atomic unit, which costs
        // far less than grouping them first with a warp match
        if (build_hist && vis) atomicAdd(&hist_s[float_key(score) >> 20], 1u);
      }
      ++ai;
    }
    if (build_hist && cur_t0 >= 0) {
      epi_bar<ET>();
      flush_hist(cur_t0);
    }
  }

  if (DSA_PDL_LATE_IDX) pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <bool MX, int D, int G, int NPAD>
cudaError_t launch_cfg(const void* q_idx, const void* k_idx, int64_t k_seq_stride, int n_seq,
                       const IndexScoreParams& p, cudaStream_t stream, bool pdl) {
  using C = Cfg<MX, D, G, NPAD>;
  CUtensorMap tm;
  CUresult r;
  if (!p.pages.table) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.L, (cuuint64_t)n_seq};
    const cuuint64_t seq_stride = n_seq > 1 ? (cuuint64_t)k_seq_stride : (cuuint64_t)p.L * C::ROW_BYTES;
    const cuuint64_t strides[2] = {(cuuint64_t)C::ROW_BYTES, seq_stride};
    const cuuint32_t box[3] = {(cuuint32_t)C::BOX_COLS, (cuuint32_t)kTileM, 1};
    r = encode_tensor_map(&tm, MX ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void*>(k_idx), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    // one pool of num_blocks * block_size rows; boxes of 64 rows (half a tile, inside one block)
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.pages.num_blocks * p.pages.block_size};
    const cuuint64_t strides[1] = {(cuuint64_t)C::ROW_BYTES};
    const cuuint32_t box[2] = {(cuuint32_t)C::BOX_COLS, (cuuint32_t)(kTileM / 2)};
    r = encode_tensor_map(&tm, MX ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(k_idx), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // q_idx rows by TMA when the box of N rows fits inside the T * H_idx rows of the tensor
  CUtensorMap tq;
  memset(&tq, 0, sizeof(tq));
  const int q_by_tma = (int64_t)p.T * p.H_idx >= C::N ? 1 : 0;
  if (q_by_tma) {
    const cuuint64_t qdims[2] = {(cuuint64_t)D, (cuuint64_t)p.T * p.H_idx};
    const cuuint64_t qstrides[1] = {(cuuint64_t)C::ROW_BYTES};
    const cuuint32_t qbox[2] = {(cuuint32_t)C::BOX_COLS, (cuuint32_t)C::N};
    r = encode_tensor_map(&tq, MX ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(q_idx), qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  auto kern = index_score_kernel<MX, D, G, NPAD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t units = (int64_t)((p.T + G - 1) / G) * p.tiles;
  if (units >= (1ll << 31)) return cudaErrorNotSupported;
  // In the fused chain a short launch (fewer than 16 units per resident slot: a decode batch of
  // tens of thousands of positions per query) runs one CTA per SM, so half the slots stay free for
  // the Top-K and attention CTAs of other batches in flight: decode B = 8, L = 32K with six batches
  // in flight, 19.97 -> 18.63 us per step (bf16) and 20.47 -> 18.04 us (MXFP8), at 2-3 us more for
  // one batch alone (grids of 3/4 and 2/3 of the slots fell in between).  Long chain launches (one
  // query over a million positions) take DSA_IDX_LONG_SLOTS_Q quarters of the slots; a launch on
  // its own (dsa_index_score) takes every slot.
  int64_t slots = (int64_t)sms * C::CTAS_PER_SM;
  if (p.share_sms && C::CTAS_PER_SM == 2 && units < 16 * slots) slots = sms;
  else if (p.share_sms && C::CTAS_PER_SM == 2) slots = slots * DSA_IDX_LONG_SLOTS_Q / 4;
  const int grid = (int)(units < slots ? units : slots);
  if (grid <= 0) return cudaSuccess;
  return launch_kernel(kern, dim3(grid), dim3(C::THREADS), C::SMEM, stream, pdl, tm, tq,
                       reinterpret_cast<const uint8_t*>(q_idx), q_by_tma, p);
}

}  // namespace

// queries that share one cache are scored four at a time (N = 4 x 64) when they can be
static bool grouped_launch(int T, int H_idx, int q_per_seq, bool mx) {
  return !mx && H_idx > 32 && q_per_seq % 4 == 0 && T >= 4;
}

bool index_score_builds_hist(int T, int H_idx, int q_per_seq, bool mx) {
  return !grouped_launch(T, H_idx, q_per_seq, mx);
}

cudaError_t launch_index_score(const void* q_idx, const void* k_idx, int64_t k_seq_stride, int n_seq,
                               int d_idx, bool mx, IndexScoreParams p, cudaStream_t stream, bool pdl,
                               bool* hist_filled) {
  const int npad = p.H_idx <= 16 ? 16 : (p.H_idx <= 32 ? 32 : 64);
  const bool grouped = grouped_launch(p.T, p.H_idx, p.q_per_seq, mx);
  if (grouped) p.hist = nullptr;  // the fused histogram is built by the one-query variants only
  if (hist_filled) *hist_filled = p.hist != nullptr;
  if (mx) {
    if (d_idx != 128) return cudaErrorNotSupported;
    // block-scaled MMAs with N = 32 or 64 (fewer heads are padded to 32)
    if (npad <= 32) return launch_cfg<true, 128, 1, 32>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
    return launch_cfg<true, 128, 1, 64>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
  }
  if (d_idx == 128) {
    if (grouped) return launch_cfg<false, 128, 4, 64>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
    if (npad == 16) return launch_cfg<false, 128, 1, 16>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
    if (npad == 32) return launch_cfg<false, 128, 1, 32>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
    return launch_cfg<false, 128, 1, 64>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
  }
  if (d_idx == 64) {
    if (npad == 16) return launch_cfg<false, 64, 1, 16>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
    if (npad == 32) return launch_cfg<false, 64, 1, 32>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
    return launch_cfg<false, 64, 1, 64>(q_idx, k_idx, k_seq_stride, n_seq, p, stream, pdl);
  }
  return cudaErrorNotSupported;
}

}  // namespace dsa
