// Step 3 of the chain: gather the Top-K rows of the latent KV cache and compute exact softmax
// attention over them (only the chosen cache entries are read, and attention over them is
// computed without approximation: Day 0 Support for New LLM Architectures, Step 1; decode gathers
// K/V by the index table then runs a small matrix multiply, "Achieving Day-0 Readiness...",
// section 2.3; FP8 KV cache, Key Optimization 2 of the first page).
//
// One CTA = (split of the K selected rows, query t, group of 16 heads).  Each selected row is
// fetched by a single bulk copy on the TMA engine (cp.async.bulk, completion counted on an
// mbarrier) straight into shared memory; rows are padded by 16 bytes so that ldmatrix reads of 8
// consecutive rows hit distinct banks.  Blocks of 64 rows go to two load slots, so two blocks
// are always in flight.  The 16 heads form the M = 16 side of warp-level bf16 tensor-core MMAs,
// so every gathered row is read from HBM once and used by all heads; softmax is online across
// blocks (running max / sum, log2 domain).
//
// Two groups of 4 warps work on the two slots at the same time and merge their (m, l, o) in shared
// memory at the end, for bf16 and E4M3 rows alike.  E4M3 rows stay raw in shared memory: the tensor
// cores turn them into the bf16 operands of the same MMAs.  An E4M3 MMA of 16 raw rows with a 0/1
// selection matrix yields, in fp32 and exactly, the values in the register layout of a bf16 B
// fragment (the K side of q.K^T with the selection on the right, the V side of P.V with the
// selection on the left); the upper halves of those fp32 are the bf16 values.  The per-row scale is
// folded into the logit and into the probability that multiplies V.
//
// When K is split over S > 1 CTAs (so a small batch still covers every SM), each CTA writes its
// partial (o, m, l) and a second kernel merges them with a log-sum-exp combine.
//
// The 576 / 512 latent row also has a kernel on the 5th-generation tensor cores
// (sparse_attn_tc_kernel below: 128 rows per CTA gathered into a swizzled bf16 tile, the two
// contractions as tcgen05.mma with accumulators in tensor memory).  A call on its own runs E4M3
// rows there (faster alone); the fused chain keeps the kernel above, which costs less SM time when
// several batches are in flight (see DSA_ATTN_TC_MASK).
#include <algorithm>
#include <atomic>

#include "dsa_internal.h"

namespace dsa {

namespace {

constexpr int kHeads = 16;    // heads per CTA (M of m16n8k16)
// Which 576 / 512 latent rows run on the tensor-memory kernel by default (bit 0 bf16, bit 1 E4M3
// rows with row scales, bit 2 E4M3 rows with tile scales), for a call on its own and inside the
// fused chain; dsa_set_attn_kernel(DSA_ATTN_TCGEN05) routes a call on its own there regardless.
// Measured on B = 8, K = 2048, alone: the mma.sync kernel with E4M3 rows widened in registers and
// one CTA per SM takes 12.9 us (tile scales 13.6, one query at L = 1M 11.6) against 15.6 (17.3,
// 13.4) for the tensor-memory kernel, bf16 12.0 against 15.6; in the chain with six batches in
// flight the tensor-memory kernel's 128-row CTAs at 172 KB of shared memory wait for whole SMs
// (earlier: 22.0 against 18.2 us per step).
#ifndef DSA_ATTN_TC_MASK
#define DSA_ATTN_TC_MASK 0
#endif
#ifndef DSA_ATTN_TC_MASK_CHAIN
#define DSA_ATTN_TC_MASK_CHAIN 0
#endif
#ifndef DSA_ATTN_CTA_TARGET
#define DSA_ATTN_CTA_TARGET 76  // attention CTAs aimed for when K is split (about one per two SMs)
#endif
#ifndef DSA_ATTN_CTA_TARGET_ALONE
#define DSA_ATTN_CTA_TARGET_ALONE 152  // the same for a call on its own (dsa_sparse_attn)
#endif
// 1: the attention kernels signal the combine kernel after their row blocks, 0: at their start.
#ifndef DSA_PDL_LATE_ATTN
#define DSA_PDL_LATE_ATTN 1
#endif
constexpr int kRows = 64;     // gathered rows per block
constexpr int kMaxRows = 4096;
constexpr float kLn2 = 0.6931471805599453f;

// 16-byte chunk c of row r of a swizzled tile with `chunks` chunks per row (a multiple of 8).
__device__ __forceinline__ uint32_t swz(int r, int c, int chunks) {
  return (uint32_t)((r * chunks + (c ^ (r & 7))) * 16);
}

// TILED (FP8 only): one fp32 scale per 128-element tile of a row instead of one per row.
template <int DQK, int DV, bool FP8, bool SEPV, bool TILED>
struct Cfg {
  static constexpr int NSC = TILED ? (DQK + 127) / 128 : (FP8 ? 1 : 0);  // scales per row
  static constexpr int PCOPIES = TILED ? DV / 128 : 1;  // P scaled per value tile
  // two independent groups of 4 warps, one block each (E4M3 rows too: the MMAs read them raw)
  static constexpr int GROUPS = 2;
  static_assert(GROUPS == 2, "block b goes to group b % 2 through slot b % 2");
  static constexpr int GW = 4;                           // warps per group
  static constexpr int GT = 32 * GW;                     // threads per group
  static constexpr int THREADS = GT * GROUPS;
  static constexpr int RPW = kRows / GW;                 // S rows per warp: two n-tiles of 8
  static constexpr int CPW = DV / GW;                    // value columns per warp
  static_assert(RPW == 16, "S warp tile");
  static_assert(CPW % 16 == 0 && (!TILED || CPW == 128), "P.V warp tile");
  static constexpr int ROW = DQK * 2 + 16;               // padded bf16 row (bytes)
  static constexpr int VROW = SEPV ? DV * 2 + 16 : 0;    // padded bf16 V row
  static constexpr int RAWROW = FP8 ? DQK + 16 : 0;      // padded E4M3 row
  static constexpr int SLOT = FP8 ? kRows * RAWROW : kRows * (ROW + VROW);  // one load slot
  static constexpr int P_CHUNKS = kRows / 8;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_SLOT = OFF_Q + kHeads * ROW;
  static constexpr int OFF_P = OFF_SLOT + 2 * SLOT;                  // per group
  static constexpr int OFF_RED = OFF_P + GROUPS * PCOPIES * kHeads * kRows * 2;  // per group: max, sum
  static constexpr int OFF_BAR = OFF_RED + GROUPS * 2 * GW * kHeads * 4;
  static constexpr int OFF_IDX = OFF_BAR + 64;
  static int bytes(int rows) { return OFF_IDX + rows * 4 * (1 + NSC); }
  static_assert(!TILED || (FP8 && DV == 512 && DQK % 16 == 0), "tiled scales: the 576/512 latent row");
  // E4M3 rows with whole 32-column chunks per warp: P.V takes V through a transposed ldmatrix of the
  // raw rows, and the accumulators hold even / odd value columns (acc[2g], acc[2g+1] for the warp's
  // 16-column group g)
  static constexpr bool EOV = FP8 && CPW % 32 == 0;
  // E4M3 rows with one scale per row: registers capped for two CTAs per SM (128 per thread, no
  // spills), so that a CTA (about 100 KB of shared memory) fits on an SM beside one index-score
  // CTA (192 threads x 168 registers, about 98 KB).  MXFP8 chain, B = 8, L = 32K, six batches in
  // flight: 15.75 -> 14.95 us per step over 2,400 steps, unchanged over 20, one batch alone 40.8 ->
  // 41.2 us.  With tile scales the cap was slower (16.41 -> 16.77 us per step), so they keep one.
  static constexpr int MINB = FP8 && !TILED ? 2 : 1;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// D = A B for a 16x32 E4M3 A (row-major fragments) and a 32x8 E4M3 B (column-major fragments),
// fp32 result (m16n8k32).  With a 0/1 selection matrix on one side it copies E4M3 values into an
// fp32 fragment exactly: one product of an E4M3 value with 1, all others zero.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// bf16 pair (lo, hi) of two fp32 that hold E4M3 values: such an fp32 has at most 4 significant
// bits, so its upper half is the bf16 of the same value.
__device__ __forceinline__ uint32_t bf16x2_of_e4m3_f32(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
}

// Two E4M3 codes (the bytes of x picked by `sel` into bits 8..15 and 24..31) as two bf16, exactly.
// The code s.eeee.mmm placed as the bf16 pattern s.0000eeee.mmm0000 has 2^-120 times the code's
// value: for e >= 1 both read 2^(e - bias) (1 + m/8), with biases 127 and 7; for e = 0 both are
// subnormal, m/8 x 2^-126 and m/8 x 2^-6.  Scaling by 2^120 is exact.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t x, uint32_t sel) {
  const uint32_t t = __byte_perm(x, 0u, sel);
  const uint32_t pat = (t & 0x80008000u) | ((t & 0x7F007F00u) >> 4);
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(pat), "r"(0x7B807B80u));  // x 2^120
  return r;
}

// Bulk copy of `bytes` (a multiple of 16) from global to shared memory on the TMA engine.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

template <int NTHREADS>
__device__ __forceinline__ void group_sync(int g) {
  asm volatile("bar.sync %0, %1;" ::"r"(g + 1), "n"(NTHREADS) : "memory");
}

template <int DQK, int DV, bool FP8, bool SEPV, bool TILED>
__global__ void __launch_bounds__(Cfg<DQK, DV, FP8, SEPV, TILED>::THREADS, Cfg<DQK, DV, FP8, SEPV, TILED>::MINB)
sparse_attn_kernel(const SparseAttnParams p) {
  using C = Cfg<DQK, DV, FP8, SEPV, TILED>;
  extern __shared__ __align__(128) uint8_t smem[];
  if (!DSA_PDL_LATE_ATTN) pdl_launch_dependents();  // the combine kernel may launch now

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int g = tid / C::GT;              // warp group
  const int gw = (tid >> 5) % C::GW;      // warp within the group
  const int gt = tid % C::GT;             // thread within the group
  const int split = blockIdx.x;
  const int t = blockIdx.y;
  const int h0 = blockIdx.z * kHeads;
  const int seq = (t + p.t_off) / p.q_per_seq;
  const int row_begin = split * p.rows_per_split;
  // rows past the query's selected positions hold -1: the chain's splits stop before them
  const int k_rows = p.valid_prefix
                         ? min(p.K, visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid))
                         : p.K;
  const int row_end = min(k_rows, row_begin + p.rows_per_split);
  const int nrows = max(0, row_end - row_begin);
  const int nblk = (nrows + kRows - 1) / kRows;

  uint8_t* q_s = smem + C::OFF_Q;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);  // [0,1] slots, [2] q
  int* idx_s = reinterpret_cast<int*>(smem + C::OFF_IDX);
  float* scale_s = reinterpret_cast<float*>(smem + C::OFF_IDX + p.rows_per_split * 4);
  uint8_t* p_s = smem + C::OFF_P + g * C::PCOPIES * kHeads * kRows * 2;
  float* red_max = reinterpret_cast<float*>(smem + C::OFF_RED) + g * 2 * C::GW * kHeads;
  float* red_sum = red_max + C::GW * kHeads;

  // paged caches: rows are pool rows found through the page table (no per-sequence base)
  const bool paged = p.pages.table != nullptr;
  const uint8_t* kv_base = p.kv + (paged ? 0 : (int64_t)seq * p.kv_seq_stride);
  const uint8_t* v_base = SEPV ? p.kv_v + (paged ? 0 : (int64_t)seq * p.v_seq_stride) : nullptr;
  const float* scale_base = FP8 ? p.kv_scale + (paged ? 0 : (int64_t)seq * p.L * C::NSC) : nullptr;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // q rows h0 .. h0+15 (a caller input, so fetched before waiting for the previous kernel);
  // rows past H are zero
  if (tid < kHeads) {
    const int h = h0 + tid;
    if (h < p.H) {
      mbar_expect_tx(&bars[2], DQK * 2);
      bulk_g2s(q_s + tid * C::ROW, p.q + ((int64_t)t * p.H + h) * DQK, DQK * 2, &bars[2]);
    } else {
      for (int c = 0; c < DQK / 8; ++c) *reinterpret_cast<uint4*>(q_s + tid * C::ROW + c * 16) = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  if (tid == 0) mbar_arrive(&bars[2]);
  pdl_wait();  // the index rows come from the previous kernel in the stream

  // this CTA's index rows, checked against [-1, L); kept as cache rows
  for (int j = tid; j < nblk * kRows; j += C::THREADS) {
    int i = -1;
    if (j < nrows) {
      i = p.idx[(int64_t)t * p.K + row_begin + j];
      if (p.slice_rows) {  // rows of other slices of the context: not this CTA's to attend
        i -= p.pos_lo;
        if (i < 0 || i >= p.L) i = -1;
      } else if (i < -1 || i >= p.L) {
        record_error(p.err, DSA_DEVERR_INDEX_RANGE);
        i = -1;
      }
      if (i >= 0 && paged) i = (int)page_row(p.pages, seq, i);
    }
    idx_s[j] = i;
  }
  __syncthreads();

  // block b -> slot b & 1, issued by the group that owns the slot; missing rows are zero-filled
  auto issue = [&](int b) {
    uint8_t* slot = smem + C::OFF_SLOT + (b & 1) * C::SLOT;
    uint64_t* bar = &bars[b & 1];
    fence_proxy_async_smem();  // earlier generic reads / zero-fills of this slot come first
    for (int r = gt; r < kRows; r += C::GT) {
      const int i = idx_s[b * kRows + r];
      if (FP8) {
        uint8_t* dst = slot + r * C::RAWROW;
        if (i >= 0) {
          mbar_expect_tx(bar, DQK);
          bulk_g2s(dst, kv_base + (int64_t)i * p.kv_row_stride, DQK, bar);
        } else {
          for (int c = 0; c < DQK / 16; ++c) *reinterpret_cast<uint4*>(dst + c * 16) = make_uint4(0, 0, 0, 0);
        }
      } else {
        uint8_t* dst = slot + r * C::ROW;
        if (i >= 0) {
          mbar_expect_tx(bar, DQK * 2 + (SEPV ? DV * 2 : 0));
          bulk_g2s(dst, kv_base + (int64_t)i * p.kv_row_stride, DQK * 2, bar);
          if (SEPV) bulk_g2s(slot + kRows * C::ROW + r * C::VROW, v_base + (int64_t)i * p.v_row_stride, DV * 2, bar);
        } else {
          for (int c = 0; c < DQK / 8; ++c) *reinterpret_cast<uint4*>(dst + c * 16) = make_uint4(0, 0, 0, 0);
          if (SEPV)
            for (int c = 0; c < DV / 8; ++c)
              *reinterpret_cast<uint4*>(slot + kRows * C::ROW + r * C::VROW + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    group_sync<C::GT>(g);  // every expect_tx of the block precedes the arrival that opens the phase
    if (gt == 0) mbar_arrive(bar);
  };
  if (g < nblk) issue(g);  // group g takes blocks g, g + 2, ... through slot g
  // E4M3 scales of the rows, fetched while the first blocks are on their way
  if constexpr (C::NSC > 0) {
    for (int j = tid; j < nblk * kRows; j += C::THREADS) {  // one row's scales per thread, all in flight
      const int i = idx_s[j];
      float v[C::NSC];
#pragma unroll
      for (int c = 0; c < C::NSC; ++c) v[c] = i >= 0 ? scale_base[(int64_t)i * C::NSC + c] : 0.f;
#pragma unroll
      for (int c = 0; c < C::NSC; ++c) scale_s[j * C::NSC + c] = v[c];
    }
    __syncthreads();
  }
  // selection matrices for the E4M3 expansions.  Byte i of this lane's register is element
  // (4 (lane % 4) + i, lane / 4) of a B fragment (k, n) and element (lane / 4, 4 (lane % 4) + i)
  // of an A fragment (m, k); it holds E4M3 1.0 = 0x38 where the k index equals the other index
  // (sel0) or the other index + 8 (sel8), zero elsewhere
  uint32_t sel0 = 0, sel8 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    sel0 |= (4 * (lane & 3) + i == (lane >> 2) ? 0x38u : 0u) << (8 * i);
    sel8 |= (4 * (lane & 3) + i == (lane >> 2) + 8 ? 0x38u : 0u) << (8 * i);
  }
  bool ok = mbar_wait(&bars[2], 0, p.err);  // q is in shared memory
  if constexpr (FP8) {
    // E4M3 rows: within each group of 16 columns, q is stored in the column order 0,1,4,5,8,9,12,13,
    // 2,3,6,7,10,11,14,15 (32-bit word p <- word {0,2,4,6,1,3,5,7}[p]), the order in which the
    // widened raw rows form B fragments above; the sum over columns does not depend on it
    for (int i = tid; i < kHeads * (DQK / 16); i += C::THREADS) {
      uint4* g = reinterpret_cast<uint4*>(q_s + (i / (DQK / 16)) * C::ROW + (i % (DQK / 16)) * 32);
      const uint4 x = g[0], y = g[1];
      g[0] = make_uint4(x.x, x.z, y.x, y.z);
      g[1] = make_uint4(x.y, x.w, y.y, y.w);
    }
    __syncthreads();
  }

  // per-thread softmax state for heads r0 = lane/4 and r1 = lane/4 + 8
  const int r0 = lane >> 2, r1 = r0 + 8;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  constexpr int NT = C::CPW / 8;  // n-tiles of 8 columns per warp in P.V
  float acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  int use = 0;  // how many blocks this group has consumed (mbarrier phase of its slots)
  for (int b = g; b < nblk; b += C::GROUPS, ++use) {
    const int slot_i = b & 1;
    ok = ok && mbar_wait(&bars[slot_i], (uint32_t)(use & 1), p.err);
    const int* ib = idx_s + b * kRows;
    const float* sb = scale_s + b * kRows * C::NSC;  // C::NSC scales per row
    uint8_t* slot = smem + C::OFF_SLOT + slot_i * C::SLOT;
    uint8_t* kv_s = slot;
    uint8_t* v_s = SEPV ? slot + kRows * C::ROW : kv_s;
    constexpr int VR = SEPV ? C::VROW : C::ROW;

    // ---- S = q . K^T : warp gw owns block rows [16 gw, 16 gw + 16) as two n-tiles of 8
    constexpr int NJ = 2;
    float s[NJ][4];
    {
      const int mat = lane >> 3, rr = lane & 7;
      const uint32_t qa = smem_u32(q_s) + (rr + (mat & 1) * 8) * C::ROW + (mat >> 1) * 16;
      // o = the partial logits over the 32-column chunks [c0, c1) of the rows
      auto s_range = [&](int c0, int c1, float (&o)[NJ][4]) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        if constexpr (FP8) {
          // the warp's 16 raw rows x 32 columns (matrices: rows 0-7 | 8-15 x bytes 0-15 | 16-31):
          // each register holds the codes of columns 4j .. 4j+3 (j = lane % 4) of row lane / 4, and
          // widened exactly to bf16 pairs (4j, 4j+1) and (4j+2, 4j+3) it is the B fragment of a
          // k-step whose columns run in the order q_s was stored in (see the q permutation)
          const uint32_t ka = smem_u32(kv_s) + (gw * 16 + rr + (mat & 1) * 8) * C::RAWROW + (mat >> 1) * 16;
#pragma unroll 2
          for (int cc = c0; cc < c1; ++cc) {
            uint32_t a0, a1, a2, a3, q0, q1, q2, q3;
            ldsm_x4(ka + cc * 32, a0, a1, a2, a3);
            ldsm_x4(qa + (2 * cc) * 32, q0, q1, q2, q3);
            mma_bf16_16816(o[0], q0, q1, q2, q3, e4m3x2_to_bf16x2(a0, 0x1404), e4m3x2_to_bf16x2(a0, 0x3424));
            mma_bf16_16816(o[1], q0, q1, q2, q3, e4m3x2_to_bf16x2(a1, 0x1404), e4m3x2_to_bf16x2(a1, 0x3424));
            ldsm_x4(qa + (2 * cc + 1) * 32, q0, q1, q2, q3);
            mma_bf16_16816(o[0], q0, q1, q2, q3, e4m3x2_to_bf16x2(a2, 0x1404), e4m3x2_to_bf16x2(a2, 0x3424));
            mma_bf16_16816(o[1], q0, q1, q2, q3, e4m3x2_to_bf16x2(a3, 0x1404), e4m3x2_to_bf16x2(a3, 0x3424));
          }
        } else {
          // matrices of one k-step: (rows 0-7 | 8-15) x (k 0-7 | 8-15)
          const uint32_t kb = smem_u32(kv_s) + (gw * 16 + rr + (mat >> 1) * 8) * C::ROW + (mat & 1) * 16;
#pragma unroll 4
          for (int ks = 2 * c0; ks < 2 * c1; ++ks) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(qa + ks * 32, a0, a1, a2, a3);
            ldsm_x4(kb + ks * 32, b0, b1, b2, b3);
            mma_bf16_16816(o[0], a0, a1, a2, a3, b0, b1);
            mma_bf16_16816(o[1], a0, a1, a2, a3, b2, b3);
          }
        }
      };
      static_assert(DQK % 32 == 0, "rows are read in 32-column chunks");
      if constexpr (TILED) {
        // tile c of a row covers chunks [4c, 4c + 4): each tile accumulates alone and is added
        // with the tile's scale of each of this thread's positions
#pragma unroll
        for (int j = 0; j < NJ; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        for (int c = 0; c < C::NSC; ++c) {
          float a_[NJ][4];
          s_range(4 * c, min(DQK / 32, 4 * c + 4), a_);
#pragma unroll
          for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int pos = gw * C::RPW + j * 8 + (lane & 3) * 2 + (e & 1);
              s[j][e] = fmaf(sb[pos * C::NSC + c], a_[j][e], s[j][e]);
            }
        }
      } else {
        s_range(0, DQK / 32, s);
      }
    }

    // ---- block softmax statistics (log2 domain)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pos = gw * C::RPW + j * 8 + (lane & 3) * 2 + (e & 1);
        float x = s[j][e] * p.scale_log2;
        if (FP8 && !TILED) x *= sb[pos];  // the row's scale (tiles: applied per tile above)
        if (ib[pos] < 0) x = -INFINITY;
        s[j][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
    }
    if ((lane & 3) == 0) {
      red_max[gw * kHeads + r0] = mx[0];
      red_max[gw * kHeads + r1] = mx[1];
    }
    group_sync<C::GT>(g);
    float m_use[2], alpha[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = hh ? r1 : r0;
      float mb = red_max[h];
#pragma unroll
      for (int w = 1; w < C::GW; ++w) mb = fmaxf(mb, red_max[w * kHeads + h]);
      const float m_new = fmaxf(m_run[hh], mb);
      m_use[hh] = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[hh] = exp2f(m_run[hh] - m_use[hh]);
      m_run[hh] = m_new;
    }
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int pos0 = gw * C::RPW + j * 8 + (lane & 3) * 2;
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pv[e] = exp2f(s[j][e] - m_use[e >> 1]);
        psum[e >> 1] += pv[e];
        if (FP8 && !TILED) pv[e] *= sb[pos0 + (e & 1)];  // V rows carry the same per-row scale
      }
      // P is stored [head][position], swizzled in 16-byte chunks of 8 positions; with tiled
      // scales one copy per value tile, scaled by that tile
      const int c = pos0 >> 3, within = (pos0 & 7) * 2;
      if constexpr (TILED) {
#pragma unroll
        for (int vt = 0; vt < C::PCOPIES; ++vt) {
          uint8_t* pc = p_s + vt * (kHeads * kRows * 2);
          const float s0 = sb[pos0 * C::NSC + vt], s1 = sb[(pos0 + 1) * C::NSC + vt];
          *reinterpret_cast<uint32_t*>(pc + swz(r0, c, C::P_CHUNKS) + within) = pack_bf16(pv[0] * s0, pv[1] * s1);
          *reinterpret_cast<uint32_t*>(pc + swz(r1, c, C::P_CHUNKS) + within) = pack_bf16(pv[2] * s0, pv[3] * s1);
        }
      } else {
        *reinterpret_cast<uint32_t*>(p_s + swz(r0, c, C::P_CHUNKS) + within) = pack_bf16(pv[0], pv[1]);
        *reinterpret_cast<uint32_t*>(p_s + swz(r1, c, C::P_CHUNKS) + within) = pack_bf16(pv[2], pv[3]);
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], 1);
      psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], 2);
    }
    if ((lane & 3) == 0) {
      red_sum[gw * kHeads + r0] = psum[0];
      red_sum[gw * kHeads + r1] = psum[1];
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      acc[i][0] *= alpha[0];
      acc[i][1] *= alpha[0];
      acc[i][2] *= alpha[1];
      acc[i][3] *= alpha[1];
    }
    group_sync<C::GT>(g);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = hh ? r1 : r0;
      float sum = red_sum[h];
#pragma unroll
      for (int w = 1; w < C::GW; ++w) sum += red_sum[w * kHeads + h];
      l_run[hh] = l_run[hh] * alpha[hh] + sum;
    }

    // ---- O += P . V : warp gw owns value columns [CPW gw, CPW gw + CPW), inside one value tile
    {
      const int mat = lane >> 3, rr = lane & 7;
      const uint32_t p_base = smem_u32(p_s) + (TILED ? (gw * C::CPW / 128) * (kHeads * kRows * 2) : 0);
#pragma unroll(FP8 ? 1 : kRows / 16)
      for (int kk = 0; kk < kRows / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(p_base + swz(rr + (mat & 1) * 8, 2 * kk + (mat >> 1), C::P_CHUNKS), a0, a1, a2, a3);
        if constexpr (C::EOV) {
          // raw rows 16kk .. 16kk+15 read transposed as 16-bit pairs of value columns (matrices:
          // rows 0-7 | 8-15 x bytes 0-15 | 16-31 of the chunk): a register holds rows 2j and 2j+1
          // (j = lane % 4) of value columns 2c and 2c+1 (c = lane / 4).  Widened exactly, bytes
          // (0, 2) are the B fragment of column 2c and bytes (1, 3) that of column 2c+1, so 16
          // value columns form two n-tiles: the even columns (acc[2g]) and the odd ones (acc[2g+1])
          const uint32_t vb = smem_u32(kv_s) + (16 * kk + rr + (mat & 1) * 8) * C::RAWROW + (mat >> 1) * 16;
#pragma unroll
          for (int ch = 0; ch < C::CPW / 32; ++ch) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(vb + gw * C::CPW + 32 * ch, v0, v1, v2, v3);
            mma_bf16_16816(acc[4 * ch], a0, a1, a2, a3, e4m3x2_to_bf16x2(v0, 0x2404), e4m3x2_to_bf16x2(v1, 0x2404));
            mma_bf16_16816(acc[4 * ch + 1], a0, a1, a2, a3, e4m3x2_to_bf16x2(v0, 0x3414), e4m3x2_to_bf16x2(v1, 0x3414));
            mma_bf16_16816(acc[4 * ch + 2], a0, a1, a2, a3, e4m3x2_to_bf16x2(v2, 0x2404), e4m3x2_to_bf16x2(v3, 0x2404));
            mma_bf16_16816(acc[4 * ch + 3], a0, a1, a2, a3, e4m3x2_to_bf16x2(v2, 0x3414), e4m3x2_to_bf16x2(v3, 0x3414));
          }
        } else if constexpr (FP8) {
          // 16-column warps (64-wide rows): raw rows 16kk .. 16kk+15 x 32 value columns as E4M3 B
          // fragments (matrices: rows 0-7 | 8-15 x bytes 0-15 | 16-31); the selections on the left
          // (value columns 0-15 or 16-31 of the chunk) give the V fragments of two n-tiles
          const uint32_t vb = smem_u32(kv_s) + (16 * kk + rr + (mat >> 1) * 8) * C::RAWROW + (mat & 1) * 16;
          constexpr int CH = C::CPW >= 32 ? C::CPW / 32 : 1;  // chunks of the warp's columns
#pragma unroll
          for (int ch = 0; ch < CH; ++ch) {
            const int col = gw * C::CPW + 32 * ch;  // first value column (16-column warps: may be mid-chunk)
            uint32_t v0, v1, v2, v3;
            ldsm_x4(vb + (col & ~31), v0, v1, v2, v3);
#pragma unroll
            for (int half = 0; half < (C::CPW >= 32 ? 2 : 1); ++half) {
              const bool upper = C::CPW >= 32 ? half == 1 : (col & 16) != 0;
              const uint32_t l0 = upper ? 0u : sel0, l8 = upper ? 0u : sel8;
              const uint32_t u0 = upper ? sel0 : 0u, u8 = upper ? sel8 : 0u;
              float f0[4], f8[4];  // value rows 0-7 and 8-15 of the k-step
              mma_e4m3_16832(f0, l0, l8, u0, u8, v0, v1);
              mma_e4m3_16832(f8, l0, l8, u0, u8, v2, v3);
              const int nt = (C::CPW >= 32 ? 4 * ch : 0) + 2 * half;
              mma_bf16_16816(acc[nt], a0, a1, a2, a3, bf16x2_of_e4m3_f32(f0[0], f0[1]), bf16x2_of_e4m3_f32(f8[0], f8[1]));
              mma_bf16_16816(acc[nt + 1], a0, a1, a2, a3, bf16x2_of_e4m3_f32(f0[2], f0[3]), bf16x2_of_e4m3_f32(f8[2], f8[3]));
            }
          }
        } else {
          const uint32_t vb = smem_u32(v_s) + (rr + (mat & 1) * 8) * VR + (gw * C::CPW + (mat >> 1) * 8) * 2;
#pragma unroll
          for (int nt = 0; nt < NT; nt += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vb + kk * 16 * VR + nt * 16, b0, b1, b2, b3);
            mma_bf16_16816(acc[nt], a0, a1, a2, a3, b0, b1);
            mma_bf16_16816(acc[nt + 1], a0, a1, a2, a3, b2, b3);
          }
        }
      }
    }
    group_sync<C::GT>(g);  // the slot and P are rewritten next
    if (ok && b + 2 < nblk) issue(b + 2);
  }
  if (DSA_PDL_LATE_ATTN) pdl_launch_dependents();
  // ---- merge the second group into the first
  {
    __syncthreads();  // all slots are idle: reuse slot 1 as staging
    float* stage = reinterpret_cast<float*>(smem + C::OFF_SLOT + C::SLOT);
    float2* ml = reinterpret_cast<float2*>(smem + C::OFF_P);  // P of group 0 is idle as well
    if (g == 1) {
      // element i of thread gt at [i][gt]: consecutive lanes hit consecutive 16-byte words
      float4* st = reinterpret_cast<float4*>(stage) + gt;
#pragma unroll
      for (int i = 0; i < NT; ++i) st[i * C::GT] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      if (gw == 0 && (lane & 3) == 0) {
        ml[r0] = make_float2(m_run[0], l_run[0]);
        ml[r1] = make_float2(m_run[1], l_run[1]);
      }
    }
    __syncthreads();
    if (g == 1) return;
    const float4* st = reinterpret_cast<const float4*>(stage) + gt;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float2 o = ml[hh ? r1 : r0];
      const float m_new = fmaxf(m_run[hh], o.x);
      const float mu = (m_new == -INFINITY) ? 0.f : m_new;
      const float a0 = exp2f(m_run[hh] - mu), a1 = exp2f(o.x - mu);
      l_run[hh] = l_run[hh] * a0 + o.y * a1;
      m_run[hh] = m_new;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const float4 v = st[i * C::GT];
        acc[i][2 * hh] = acc[i][2 * hh] * a0 + (hh ? v.z : v.x) * a1;
        acc[i][2 * hh + 1] = acc[i][2 * hh + 1] * a0 + (hh ? v.w : v.y) * a1;
      }
    }
  }

  const int col0 = gw * C::CPW + (lane & 3) * 2;
  // even / odd accumulators (C::EOV): slot s of acc[2g] is value column 16g + 2s, of acc[2g + 1]
  // column 16g + 2s + 1, so a thread holds 4 consecutive columns of each group
  const int colq = gw * C::CPW + (lane & 3) * 4;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = h0 + (hh ? r1 : r0);
    if (h >= p.H) continue;
    if (p.splits == 1) {
      const float inv = l_run[hh] > 0.f ? 1.f / l_run[hh] : 0.f;
      if (p.out_f32) {
        float* o = p.out_f32 + ((int64_t)t * p.H + h) * DV;
        if constexpr (C::EOV) {
#pragma unroll
          for (int g2 = 0; g2 < NT / 2; ++g2)
            *reinterpret_cast<float4*>(o + colq + 16 * g2) =
                make_float4(acc[2 * g2][2 * hh] * inv, acc[2 * g2 + 1][2 * hh] * inv, acc[2 * g2][2 * hh + 1] * inv,
                            acc[2 * g2 + 1][2 * hh + 1] * inv);
        } else {
#pragma unroll
          for (int i = 0; i < NT; ++i)
            *reinterpret_cast<float2*>(o + col0 + i * 8) = make_float2(acc[i][2 * hh] * inv, acc[i][2 * hh + 1] * inv);
        }
      } else {
        __nv_bfloat16* o = p.out + ((int64_t)t * p.H + h) * DV;
        if constexpr (C::EOV) {
#pragma unroll
          for (int g2 = 0; g2 < NT / 2; ++g2)
            *reinterpret_cast<uint2*>(o + colq + 16 * g2) =
                make_uint2(pack_bf16(acc[2 * g2][2 * hh] * inv, acc[2 * g2 + 1][2 * hh] * inv),
                           pack_bf16(acc[2 * g2][2 * hh + 1] * inv, acc[2 * g2 + 1][2 * hh + 1] * inv));
        } else {
#pragma unroll
          for (int i = 0; i < NT; ++i)
            *reinterpret_cast<uint32_t*>(o + col0 + i * 8) = pack_bf16(acc[i][2 * hh] * inv, acc[i][2 * hh + 1] * inv);
        }
      }
      if (p.lse && (lane & 3) == 0 && gw == 0)
        p.lse[(int64_t)t * p.H + h] = l_run[hh] > 0.f ? (m_run[hh] + log2f(l_run[hh])) * kLn2 : -INFINITY;
    } else {
      const int64_t row = ((int64_t)t * p.H + h) * p.splits + split;
      float* o = p.part_o + row * DV;
      if constexpr (C::EOV) {
#pragma unroll
        for (int g2 = 0; g2 < NT / 2; ++g2)
          *reinterpret_cast<float4*>(o + colq + 16 * g2) =
              make_float4(acc[2 * g2][2 * hh], acc[2 * g2 + 1][2 * hh], acc[2 * g2][2 * hh + 1], acc[2 * g2 + 1][2 * hh + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < NT; ++i)
          *reinterpret_cast<float2*>(o + col0 + i * 8) = make_float2(acc[i][2 * hh], acc[i][2 * hh + 1]);
      }
      if ((lane & 3) == 0 && gw == 0)
        *reinterpret_cast<float2*>(p.part_ml + row * 2) = make_float2(m_run[hh], l_run[hh]);
    }
  }
}

// Merges split partials: out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j and
// lse = (M + log2 sum_j 2^(m_j - M) l_j) * ln 2.  One CTA per (query, head); each thread owns four
// value columns.  The partials are read eight splits per batch (all loads of a batch in flight
// at once) and merged with an online rescale, so a batch costs one memory round trip.
template <int DV>
__global__ void __launch_bounds__(DV / 4) lse_combine_kernel(const SparseAttnParams p) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int kBatch = 8;
  const int t = blockIdx.x, h = blockIdx.y;
  const int64_t row = ((int64_t)t * p.H + h) * p.splits;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + row;
  const int c = threadIdx.x * 4;
  float M = -INFINITY, lsum = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < p.splits; j0 += kBatch) {
    float2 mlb[kBatch];
    float4 ob[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const bool in = j0 + k < p.splits;
      mlb[k] = in ? ml[j0 + k] : make_float2(-INFINITY, 0.f);
      ob[k] = in ? *reinterpret_cast<const float4*>(p.part_o + (row + j0 + k) * DV + c)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float Mb = M;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) Mb = fmaxf(Mb, mlb[k].x);
    const float Mu = (Mb == -INFINITY) ? 0.f : Mb;
    const float a = exp2f(M - Mu);  // rescales what the earlier batches gave (0 when empty)
    lsum *= a;
    o.x *= a, o.y *= a, o.z *= a, o.w *= a;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const float wj = exp2f(mlb[k].x - Mu);
      lsum += wj * mlb[k].y;
      o.x += wj * ob[k].x;
      o.y += wj * ob[k].y;
      o.z += wj * ob[k].z;
      o.w += wj * ob[k].w;
    }
    M = Mb;
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  if (p.out_f32) {
    *reinterpret_cast<float4*>(p.out_f32 + ((int64_t)t * p.H + h) * DV + c) =
        make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
  } else {
    __nv_bfloat16* out = p.out + ((int64_t)t * p.H + h) * DV + c;
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
  }
  if (p.lse && threadIdx.x == 0)
    p.lse[(int64_t)t * p.H + h] = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
}

// ---------------------------------------------------------------------------------------------
// The 576 / 512 latent row on the 5th-generation tensor cores.  One CTA = 128 selected rows of one
// query (the M = 128 side of tcgen05.mma) and 16 heads:
//   * the rows are gathered into one 128-byte-swizzled, K-major bf16 tile (9 boxes of 64 columns):
//     bf16 rows by 16-byte cp.async chunks placed at their swizzled addresses; E4M3 rows loaded 16
//     codes at a time and widened exactly to bf16 in registers on the way;
//   * S^T[128 rows x 16 heads] = K q^T: 36 MMAs (M = 128, N = 16, K = 16) into tensor memory
//     (one accumulator per 128-element scale tile for tile-scaled FP8 rows);
//   * four warps (one row per thread, the tensor-memory lane of that row) take the softmax of the
//     tile: per-head maxima and sums over the 128 rows with warp butterflies and a 4-warp exchange,
//     and write P^T (bf16, scaled per row or per value tile) as the K-major B operand;
//   * O^T[512 values x 16 heads] = V^T P: the same tile read as an MN-major A operand (values along
//     M, rows along K), 4 accumulators of 128 values x 8 K steps;
//   * the four warps read O^T back (one value column per thread) and write this split's partial
//     (o, m, l), merged over the splits by lse_combine_kernel (or the output when K <= 128).
// No warp-level mma.sync: the E4M3 rows cost one ALU widening per element, not tensor-core work.
constexpr int kTcRows = 128;

template <bool FP8, bool TILED>
struct TcCfg {
  static constexpr int DQK = 576, DV = 512;
  static constexpr int BOXES = DQK / 64;                 // 64 bf16 columns = one 128-byte atom row
  static constexpr int NSC = TILED ? (DQK + 127) / 128 : (FP8 ? 1 : 0);
  static constexpr int SACC = TILED ? NSC : 1;           // S accumulators (one per scale tile)
  static constexpr int PCOPIES = TILED ? DV / 128 : 1;   // P per value tile
  static constexpr int THREADS = 256;
  static constexpr int TILE_BOX = kTcRows * 128;         // 16 KB per box of the row tile
  static constexpr int Q_BOX = kHeads * 128;             // 2 KB per box of q
  static constexpr int P_BYTES = 2 * Q_BOX;              // P^T: 16 heads x 128 rows bf16
  static constexpr int OFF_TILE = 0;
  static constexpr int OFF_Q = OFF_TILE + BOXES * TILE_BOX;
  static constexpr int OFF_P = OFF_Q + BOXES * Q_BOX;
  static constexpr int OFF_RED = OFF_P + PCOPIES * P_BYTES;  // [2][4 warps][16] fp32
  static constexpr int OFF_IDX = OFF_RED + 2 * 4 * kHeads * 4;
  static constexpr int OFF_SC = OFF_IDX + kTcRows * 4;
  static constexpr int OFF_BAR = OFF_SC + kTcRows * 4 * (NSC > 0 ? NSC : 1);
  static constexpr int SMEM = OFF_BAR + 64 + 1024;       // + alignment slack (1024-byte atoms)
  static constexpr int TMEM_COLS = 256;                  // S at [0, 16 SACC), O^T at [128, 192)
  static constexpr int O_COL = 128;
  static_assert(16 * SACC <= O_COL, "S accumulators");
};

// Butterfly over a warp: v[0..15] are this lane's values for heads 0..15; afterwards v[0] holds the
// reduction over all 32 lanes of head (lane >> 1) & 15.
template <bool MAX>
__device__ __forceinline__ void warp_reduce16(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
  auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
#pragma unroll
  for (int n = 8; n >= 1; n >>= 1) {  // offsets 16, 8, 4, 2: halve the heads per lane
    const int off = 2 * n;
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = hi ? v[i + n] : v[i];
      const float send = hi ? v[i] : v[i + n];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
  v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

template <bool FP8, bool TILED>
__global__ void __launch_bounds__(256, 1) sparse_attn_tc_kernel(const SparseAttnParams p) {
  using C = TcCfg<FP8, TILED>;
  constexpr int DQK = C::DQK, DV = C::DV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tile = smem + C::OFF_TILE;
  uint8_t* q_s = smem + C::OFF_Q;
  uint8_t* p_s = smem + C::OFF_P;
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);  // [0]: max, [1]: sum; [warp][head]
  int* idx_s = reinterpret_cast<int*>(smem + C::OFF_IDX);
  float* scale_s = reinterpret_cast<float*>(smem + C::OFF_SC);  // [row][NSC]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);  // [0] S done, [1] O done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  if (!DSA_PDL_LATE_ATTN) pdl_launch_dependents();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, t = blockIdx.y, h0 = blockIdx.z * kHeads;
  const int seq = (t + p.t_off) / p.q_per_seq;
  const int row_begin = split * kTcRows;
  const int k_rows = p.valid_prefix
                         ? min(p.K, visible_len(t + p.t_off, p.L, p.q_per_seq, p.q_pos0, p.n_valid))
                         : p.K;
  const int nrows = max(0, min(kTcRows, k_rows - row_begin));
  const bool paged = p.pages.table != nullptr;
  const uint8_t* kv_base = p.kv + (paged ? 0 : (int64_t)seq * p.kv_seq_stride);
  const float* scale_base = FP8 ? p.kv_scale + (paged ? 0 : (int64_t)seq * p.L * C::NSC) : nullptr;

  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  // q rows h0 .. h0+15 (a caller input, so read before waiting for the previous kernel) into the
  // swizzled K-major B layout; rows past H are zero
  for (int i = tid; i < kHeads * (DQK / 8); i += C::THREADS) {
    const int h = i / (DQK / 8), c = i - h * (DQK / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (h0 + h < p.H) v = *reinterpret_cast<const uint4*>(p.q + ((int64_t)t * p.H + h0 + h) * DQK + 8 * c);
    *reinterpret_cast<uint4*>(q_s + (c >> 3) * C::Q_BOX + h * 128 + (((c & 7) ^ (h & 7)) << 4)) = v;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the index rows come from the previous kernel in the stream

  // ---- this CTA's index rows (checked against [-1, L), or taken from this slice of the context)
  // and their scales
  if (tid < kTcRows) {
    int i = -1;
    if (tid < nrows) {
      i = p.idx[(int64_t)t * p.K + row_begin + tid];
      if (p.slice_rows) {
        i -= p.pos_lo;
        if (i < 0 || i >= p.L) i = -1;
      } else if (i < -1 || i >= p.L) {
        record_error(p.err, DSA_DEVERR_INDEX_RANGE);
        i = -1;
      }
      if (i >= 0 && paged) i = (int)page_row(p.pages, seq, i);
    }
    idx_s[tid] = i;
    if constexpr (C::NSC > 0) {
#pragma unroll
      for (int c = 0; c < C::NSC; ++c) scale_s[tid * C::NSC + c] = i >= 0 ? scale_base[(int64_t)i * C::NSC + c] : 0.f;
    }
  }
  __syncthreads();

  // ---- gather the rows into the swizzled bf16 tile: element (r, col) at box col / 64, byte
  // r * 128 + ((col % 64 / 8) ^ (r % 8)) * 16 + (col % 8) * 2
  if constexpr (!FP8) {
    for (int i = tid; i < kTcRows * (DQK / 8); i += C::THREADS) {
      const int r = i / (DQK / 8), c = i - r * (DQK / 8);  // 16-byte chunk c of row r
      const int row = idx_s[r];
      uint8_t* dst = tile + (c >> 3) * C::TILE_BOX + r * 128 + (((c & 7) ^ (r & 7)) << 4);
      cp_async16(dst, kv_base + (int64_t)(row >= 0 ? row : 0) * p.kv_row_stride + 16 * c, row >= 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
  } else {
    constexpr int CH = DQK / 16;  // 16-code chunks per row
    constexpr int BATCH = 6;      // loads in flight per thread
    constexpr int TOTAL = kTcRows * CH;
    static_assert(TOTAL % (BATCH * C::THREADS) == 0, "whole batches");
#pragma unroll 1
    for (int i0 = tid; i0 < TOTAL; i0 += BATCH * C::THREADS) {
      uint4 raw[BATCH];
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int i = i0 + b * C::THREADS;
        const int r = i / CH, c = i - r * CH;
        const int row = idx_s[r];
        raw[b] = row >= 0 ? __ldg(reinterpret_cast<const uint4*>(kv_base + (int64_t)row * p.kv_row_stride + 16 * c))
                          : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int i = i0 + b * C::THREADS;
        const int r = i / CH, c = i - r * CH;  // codes 16c .. 16c + 15: bf16 chunks 2c and 2c + 1
        const uint4 lo = make_uint4(e4m3x2_to_bf16x2(raw[b].x, 0x1404), e4m3x2_to_bf16x2(raw[b].x, 0x3424),
                                    e4m3x2_to_bf16x2(raw[b].y, 0x1404), e4m3x2_to_bf16x2(raw[b].y, 0x3424));
        const uint4 hi = make_uint4(e4m3x2_to_bf16x2(raw[b].z, 0x1404), e4m3x2_to_bf16x2(raw[b].z, 0x3424),
                                    e4m3x2_to_bf16x2(raw[b].w, 0x1404), e4m3x2_to_bf16x2(raw[b].w, 0x3424));
        const int c0 = 2 * c, c1 = 2 * c + 1;
        *reinterpret_cast<uint4*>(tile + (c0 >> 3) * C::TILE_BOX + r * 128 + (((c0 & 7) ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(tile + (c1 >> 3) * C::TILE_BOX + r * 128 + (((c1 & 7) ^ (r & 7)) << 4)) = hi;
      }
    }
  }
  fence_proxy_async_smem();  // the generic-proxy writes of tile and q are seen by the tensor cores
  __syncthreads();

  // ---- S^T = K q^T (one elected thread issues; completion arrives on bar[0])
  if (warp == 0) {
    tc_fence_after();
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(1, 1, kTcRows, kHeads);
      const uint32_t tb = smem_u32(tile), qb = smem_u32(q_s);
#pragma unroll 1
      for (int b = 0; b < C::BOXES; ++b) {
        const int acc = TILED ? b / 2 : 0;  // 128-element scale tile of this box
        const bool first = TILED ? (b % 2 == 0) : (b == 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_f16(tmem + 16 * acc, smem_desc_sw128(tb + b * C::TILE_BOX + 32 * k),
                  smem_desc_sw128(qb + b * C::Q_BOX + 32 * k), idesc, (first && k == 0) ? 0u : 1u);
      }
      tc_commit(&bar[0]);
    }
    __syncwarp();
  }

  float m_fin = -INFINITY, l_fin = 0.f;  // head (tid & 15) of warp 0: this split's (m, l)
  if (warp < 4) {
    // ---- softmax over the tile's 128 rows: thread = row r = tensor-memory lane r
    const int r = tid;
    bool ok = mbar_wait(&bar[0], 0, p.err);
    tc_fence_after();
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    float x[16];
    const bool valid = idx_s[r] >= 0;
    if constexpr (TILED) {
#pragma unroll
      for (int h = 0; h < 16; ++h) x[h] = 0.f;
#pragma unroll
      for (int c = 0; c < C::SACC; ++c) {
        float s[16];
        tmem_ld_sync(lane_base + 16 * c, s);
        const float sc = scale_s[r * C::NSC + c];
#pragma unroll
        for (int h = 0; h < 16; ++h) x[h] = fmaf(sc, s[h], x[h]);
      }
#pragma unroll
      for (int h = 0; h < 16; ++h) x[h] = valid && ok ? x[h] * p.scale_log2 : -INFINITY;
    } else {
      tmem_ld_sync(lane_base, x);
      const float f = p.scale_log2 * (FP8 ? scale_s[r] : 1.f);
#pragma unroll
      for (int h = 0; h < 16; ++h) x[h] = valid && ok ? x[h] * f : -INFINITY;
    }
    // per-head maxima over the 128 rows
    float v[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) v[h] = x[h];
    warp_reduce16<true>(v);
    if ((lane & 1) == 0) red[warp * kHeads + ((lane >> 1) & 15)] = v[0];
    asm volatile("bar.sync 1, 128;" ::: "memory");
    float mu[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      const float m = fmaxf(fmaxf(red[h], red[kHeads + h]), fmaxf(red[2 * kHeads + h], red[3 * kHeads + h]));
      mu[h] = m == -INFINITY ? 0.f : m;
      x[h] = exp2f(x[h] - mu[h]);  // the probability of this row, unnormalised
      v[h] = x[h];
    }
    if (lane < 16 && warp == 0) m_fin = fmaxf(fmaxf(red[lane], red[kHeads + lane]), fmaxf(red[2 * kHeads + lane], red[3 * kHeads + lane]));
    warp_reduce16<false>(v);
    if ((lane & 1) == 0) red[4 * kHeads + warp * kHeads + ((lane >> 1) & 15)] = v[0];
    // P^T as the K-major B operand: element (head h, row r) at box r / 64, byte
    // h * 128 + ((r % 64 / 8) ^ (h % 8)) * 16 + (r % 8) * 2; one copy per value tile when scaled by tile
#pragma unroll
    for (int pc = 0; pc < C::PCOPIES; ++pc) {
      const float sc = TILED ? scale_s[r * C::NSC + pc] : (FP8 ? scale_s[r] : 1.f);  // V carries the row's scale
      uint8_t* pb = p_s + pc * C::P_BYTES + (r >> 6) * C::Q_BOX + (r & 7) * 2;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        *reinterpret_cast<__nv_bfloat16*>(pb + h * 128 + ((((r & 63) >> 3) ^ (h & 7)) << 4)) = __float2bfloat16_rn(x[h] * sc);
    }
    fence_proxy_async_smem();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (lane < 16 && warp == 0)
      l_fin = red[4 * kHeads + lane] + red[5 * kHeads + lane] + red[6 * kHeads + lane] + red[7 * kHeads + lane];

    // ---- O^T = V^T P: values along M (4 blocks of 128), rows along K (8 steps of 16)
    if (warp == 0) {
      tc_fence_after();
      if (lane == 0 && ok) {
        constexpr uint32_t idesc_pv = make_idesc(1, 1, kTcRows, kHeads) | (1u << 15);  // A MN-major
        const uint32_t tb = smem_u32(tile), pbase = smem_u32(p_s);
#pragma unroll 1
        for (int j = 0; j < DV / 128; ++j) {
          const uint32_t pj = pbase + (TILED ? j : 0) * C::P_BYTES;
#pragma unroll
          for (int ks = 0; ks < kTcRows / 16; ++ks)
            mma_f16(tmem + C::O_COL + 16 * j, smem_desc_sw128_mn(tb + 2 * j * C::TILE_BOX + ks * 2048, C::TILE_BOX, 1024),
                    smem_desc_sw128(pj + (ks >> 2) * C::Q_BOX + 32 * (ks & 3)), idesc_pv, ks > 0 ? 1u : 0u);
        }
      }
      if (lane == 0) tc_commit(&bar[1]);  // (arrives at once when nothing was issued)
      __syncwarp();
    }
    ok = mbar_wait(&bar[1], 0, p.err) && ok;
    tc_fence_after();
    // ---- this split's output: thread = value column 128 j + 32 warp + lane of every head
    float inv[16];
    if (p.splits == 1) {
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float l = red[4 * kHeads + h] + red[5 * kHeads + h] + red[6 * kHeads + h] + red[7 * kHeads + h];
        inv[h] = l > 0.f ? 1.f / l : 0.f;
      }
    }
#pragma unroll 1
    for (int j = 0; j < DV / 128; ++j) {
      float o[16];
      tmem_ld_sync(lane_base + C::O_COL + 16 * j, o);
      const int v = 128 * j + 32 * warp + lane;
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        if (h0 + h >= p.H) continue;
        const int64_t hr = (int64_t)t * p.H + h0 + h;
        const float oh = ok ? o[h] : 0.f;
        if (p.splits == 1) {
          if (p.out_f32) p.out_f32[hr * DV + v] = oh * inv[h];
          else p.out[hr * DV + v] = __float2bfloat16_rn(oh * inv[h]);
        } else {
          p.part_o[(hr * p.splits + split) * DV + v] = oh;
        }
      }
    }
    if (warp == 0 && lane < 16 && h0 + lane < p.H) {
      const int64_t hr = (int64_t)t * p.H + h0 + lane;
      if (p.splits == 1) {
        if (p.lse) p.lse[hr] = l_fin > 0.f ? (m_fin + log2f(l_fin)) * kLn2 : -INFINITY;
      } else {
        *reinterpret_cast<float2*>(p.part_ml + (hr * p.splits + split) * 2) = make_float2(m_fin, l_fin);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (DSA_PDL_LATE_ATTN) pdl_launch_dependents();
}

template <bool FP8, bool TILED>
cudaError_t launch_tc(const SparseAttnParams& p, cudaStream_t stream, bool pdl) {
  using C = TcCfg<FP8, TILED>;
  auto kern = sparse_attn_tc_kernel<FP8, TILED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, p.T, (p.H + kHeads - 1) / kHeads);
  e = launch_kernel(kern, grid, dim3(C::THREADS), C::SMEM, stream, pdl, p);
  if (e != cudaSuccess || p.splits == 1) return e;
  return launch_kernel(lse_combine_kernel<512>, dim3(p.T, p.H), dim3(512 / 4), 0, stream, true, p);
}

template <int DQK, int DV, bool FP8, bool SEPV, bool TILED = false>
cudaError_t launch_variant(const SparseAttnParams& p, cudaStream_t stream, bool pdl) {
  using C = Cfg<DQK, DV, FP8, SEPV, TILED>;
  auto kern = sparse_attn_kernel<DQK, DV, FP8, SEPV, TILED>;
  const int smem = C::bytes(p.rows_per_split);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, p.T, (p.H + kHeads - 1) / kHeads);
  e = launch_kernel(kern, grid, dim3(C::THREADS), smem, stream, pdl, p);
  if (e != cudaSuccess || p.splits == 1) return e;
  return launch_kernel(lse_combine_kernel<DV>, dim3(p.T, p.H), dim3(DV / 4), 0, stream, true, p);
}

// ---------------------------------------------------------------------------------------------
// Merge of the partial outputs of G context slices: slice g attended over the selected positions
// it holds and gave o_g (normalised over its own rows) and lse_g (natural log; -inf when it held
// none).  With M = max_g lse_g:  out = sum_g e^(lse_g - M) o_g / sum_g e^(lse_g - M) and
// lse = M + ln sum_g e^(lse_g - M).  One CTA per (query, head), four value columns per thread.
__global__ void __launch_bounds__(128) slice_combine_kernel(const SliceCombineParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x, h = blockIdx.y;
  const int64_t row = (int64_t)t * p.H + h;
  float M = -INFINITY;
  for (int g = 0; g < p.G; ++g) M = fmaxf(M, p.lse_parts[g * p.lse_stride + row]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float wsum = 0.f;
  for (int g = 0; g < p.G; ++g) wsum += expf(p.lse_parts[g * p.lse_stride + row] - Mu);
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  for (int c = 4 * threadIdx.x; c < p.D_v; c += 4 * blockDim.x) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < p.G; ++g) {
      const float lg = p.lse_parts[g * p.lse_stride + row];
      if (lg == -INFINITY) continue;  // a slice with no selected row contributes nothing
      const float wg = expf(lg - Mu);
      const float4 v = *reinterpret_cast<const float4*>(p.o_parts + g * p.o_stride + row * p.D_v + c);
      o.x = fmaf(wg, v.x, o.x);
      o.y = fmaf(wg, v.y, o.y);
      o.z = fmaf(wg, v.z, o.z);
      o.w = fmaf(wg, v.w, o.w);
    }
    __nv_bfloat16* out = p.out + row * p.D_v + c;
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
  }
  if (p.lse && threadIdx.x == 0) p.lse[row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_slice_combine(const SliceCombineParams& p, cudaStream_t stream, bool pdl) {
  if (p.T <= 0 || p.H <= 0) return cudaSuccess;
  return launch_kernel(slice_combine_kernel, dim3(p.T, p.H), dim3(128), 0, stream, pdl, p);
}

int sparse_attn_splits(int T, int H, int K, bool chain) {
  // Inside the fused chain about one CTA per two SMs of a 152-SM part.  A CTA's time is mostly the
  // gather's round trips (index rows, then the selected rows), not its MMAs, so fewer CTAs with
  // more blocks each cost less SM time; with independent batches in flight the other SMs score the
  // next batches (measured on the decode chain, B = 8, L = 32K: 64 CTAs of 256 rows gave 7 % more
  // queries/s than 128 CTAs of 128 rows, at 3 % more latency for one batch alone).  A call on its
  // own aims at one CTA per SM: each CTA's rows arrive in one round.
  const int blocks = (K + kRows - 1) / kRows;
  const int ctas_per_split = T * ((H + kHeads - 1) / kHeads);
  if (ctas_per_split <= 0) return 1;
  const int target = chain ? DSA_ATTN_CTA_TARGET : DSA_ATTN_CTA_TARGET_ALONE;
  int s = (target + ctas_per_split - 1) / ctas_per_split;
  s = s < 1 ? 1 : (s > 64 ? 64 : s);
  // at least two blocks per split: a CTA's two warp groups take alternate blocks, so a one-block
  // split leaves one group idle (one query, K = 2048: 16 CTAs of 128 rows instead of 32 of 64)
  if (s > blocks / 2) s = blocks / 2 > 1 ? blocks / 2 : 1;
  // whole blocks per split, and no empty split
  const int rows = ((blocks + s - 1) / s) * kRows;
  return (K + rows - 1) / rows;
}

static int rows_per_split(int K, int splits) {
  const int blocks = (K + kRows - 1) / kRows;
  return ((blocks + splits - 1) / splits) * kRows;
}

// Which rows go to the tensor-memory kernel: the 576 / 512 latent row, per storage format (bit 0
// bf16, bit 1 E4M3 with row scales, bit 2 E4M3 with 128-element tile scales).
std::atomic<int> g_attn_kernel{0};  // DSA_ATTN_AUTO or DSA_ATTN_TCGEN05 (dsa_set_attn_kernel)

bool attn_uses_tc(int D_qk, int D_v, bool fp8, bool sepv, bool tiled, bool chain) {
  if (D_qk != 576 || D_v != 512 || sepv) return false;
  if (!chain && g_attn_kernel.load(std::memory_order_relaxed) == 1) return true;
  const int bit = tiled ? 4 : (fp8 ? 2 : 1);
  return ((chain ? DSA_ATTN_TC_MASK_CHAIN : DSA_ATTN_TC_MASK) & bit) != 0;
}

bool set_attn_kernel(int kernel) {
  if (kernel != 0 && kernel != 1) return false;
  g_attn_kernel.store(kernel, std::memory_order_relaxed);
  return true;
}

static int routed_splits(int T, int H, int K, bool tc, bool chain) {
  return tc ? (K + kTcRows - 1) / kTcRows : sparse_attn_splits(T, H, K, chain);
}

int sparse_attn_launches(int T, int H, int K, int D_qk, int D_v, bool fp8, bool sepv, bool tiled, bool chain) {
  return routed_splits(T, H, K, attn_uses_tc(D_qk, D_v, fp8, sepv, tiled, chain), chain) > 1 ? 2 : 1;
}

size_t sparse_attn_ws_bytes(int T, int H, int K, int D_v) {
  // sized for every kernel a call can be routed to now (the storage format is not an argument
  // here): the mma.sync kernel's splits, in the chain and alone, and the tensor-memory kernel's
  // 128-row splits when it can be selected
  int splits = std::max(sparse_attn_splits(T, H, K, true), sparse_attn_splits(T, H, K, false));
  if (D_v == 512 && ((DSA_ATTN_TC_MASK | DSA_ATTN_TC_MASK_CHAIN) != 0 || g_attn_kernel.load() == 1))
    splits = std::max(splits, routed_splits(T, H, K, true, false));
  if (splits <= 1) return 0;
  const size_t rows = (size_t)T * H * splits;
  return align_up(rows * D_v * sizeof(float), 256) + align_up(rows * 2 * sizeof(float), 256);
}

cudaError_t launch_sparse_attn(SparseAttnParams p, int D_qk, int D_v, bool fp8, bool sepv, void* ws,
                               cudaStream_t stream, bool pdl, bool tiled) {
  const bool tc = attn_uses_tc(D_qk, D_v, fp8, sepv, tiled, p.valid_prefix);
  p.splits = routed_splits(p.T, p.H, p.K, tc, p.valid_prefix);
  p.rows_per_split = tc ? kTcRows : rows_per_split(p.K, p.splits);
  if (p.rows_per_split > kMaxRows) return cudaErrorNotSupported;
  if (p.splits > 1) {
    if (!ws) return cudaErrorInvalidValue;
    const size_t rows = (size_t)p.T * p.H * p.splits;
    p.part_o = reinterpret_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + align_up(rows * D_v * sizeof(float), 256));
  }
  if (tc) {
    if (tiled) return launch_tc<true, true>(p, stream, pdl);
    return fp8 ? launch_tc<true, false>(p, stream, pdl) : launch_tc<false, false>(p, stream, pdl);
  }
  if (tiled) {  // FP8 with one scale per 128-element tile: the 576/512 latent row only
    if (!fp8 || D_qk != 576 || D_v != 512 || sepv) return cudaErrorNotSupported;
    return launch_variant<576, 512, true, false, true>(p, stream, pdl);
  }
  if (D_qk == 576 && D_v == 512 && !sepv) {
    return fp8 ? launch_variant<576, 512, true, false>(p, stream, pdl)
               : launch_variant<576, 512, false, false>(p, stream, pdl);
  }
  if (D_qk == 64 && D_v == 64) {
    if (sepv) return fp8 ? cudaErrorNotSupported : launch_variant<64, 64, false, true>(p, stream, pdl);
    return fp8 ? launch_variant<64, 64, true, false>(p, stream, pdl)
               : launch_variant<64, 64, false, false>(p, stream, pdl);
  }
  return cudaErrorNotSupported;
}

}  // namespace dsa
