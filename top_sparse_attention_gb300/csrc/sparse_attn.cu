// Step 3 of the chain: gather the Top-K rows of the latent KV cache and compute exact softmax
// attention over them ("a sparse-attention kernel then reads only the selected KV entries to
// perform exact computation", Day 0 Support for New LLM Architectures, Step 1; decode gathers
// K/V by the index table then runs a small matrix multiply, "Achieving Day-0 Readiness...",
// section 2.3; FP8 KV cache, Key Optimization 2 of the first page).
//
// One CTA = (query t, split of the K selected rows, group of 16 heads).  Rows arrive in blocks
// of 64 by 16-byte copies straight into shared memory (no DRAM staging buffer); the 16 heads
// form the M = 16 side of warp-level bf16 tensor-core MMAs, so every gathered row is read from
// HBM once and used by all heads.  Softmax is online across blocks (running max / sum); when K
// is split over several CTAs each writes (o, m, l) partials and a second kernel merges them
// with a log-sum-exp combine.  FP8 rows are widened to bf16 in registers on the way into shared
// memory (exact: every E4M3 value is a bf16 value); the per-row scale is folded into the logit
// and into the probability that multiplies V.
#include "dsa_internal.h"

namespace dsa {

namespace {

constexpr int kThreads = 128;
constexpr int kHeads = 16;   // heads per CTA (M of m16n8k16)
constexpr int kRows = 64;    // gathered rows per block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Byte offset of 16-byte chunk c of row r in a swizzled bf16 tile whose rows hold `chunks`
// chunks (a multiple of 8): the chunk index is XORed with (r & 7) so that the 8 rows an
// ldmatrix phase touches fall in distinct banks.
__device__ __forceinline__ uint32_t swz(int r, int c, int chunks) {
  return (uint32_t)((r * chunks + (c ^ (r & 7))) * 16);
}

template <int DQK, int DV, bool FP8, bool SEPV>
struct Smem {
  static constexpr int QK_CHUNKS = DQK / 8;
  static constexpr int V_CHUNKS = DV / 8;
  static constexpr int P_CHUNKS = kRows / 8;
  static constexpr int Q_BYTES = kHeads * DQK * 2;
  static constexpr int KV_BYTES = kRows * DQK * 2;
  static constexpr int V_BYTES = SEPV ? kRows * DV * 2 : 0;
  static constexpr int P_BYTES = kHeads * kRows * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_KV + KV_BYTES;
  static constexpr int OFF_P = OFF_V + V_BYTES;
  static constexpr int OFF_IDX = OFF_P + P_BYTES;
  static constexpr int OFF_SCALE = OFF_IDX + kRows * 4;
  static constexpr int OFF_RED = OFF_SCALE + kRows * 4;
  static constexpr int BYTES = OFF_RED + 2 * 4 * kHeads * 4;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 4 E4M3 codes (one 32-bit word) -> 4 bf16 values (two 32-bit words), exact.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  __half2_raw h0 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
  __half2_raw h1 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  float2 f0 = __half22float2(*reinterpret_cast<__half2*>(&h0));
  float2 f1 = __half22float2(*reinterpret_cast<__half2*>(&h1));
  return make_uint2(pack_bf16(f0.x, f0.y), pack_bf16(f1.x, f1.y));
}

template <int DQK, int DV, bool FP8, bool SEPV>
__global__ void __launch_bounds__(kThreads, 2)
sparse_attn_kernel(const SparseAttnParams p) {
  using S = Smem<DQK, DV, FP8, SEPV>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* q_s = smem + S::OFF_Q;
  uint8_t* kv_s = smem + S::OFF_KV;
  uint8_t* v_s = SEPV ? smem + S::OFF_V : kv_s;
  uint8_t* p_s = smem + S::OFF_P;
  int* idx_s = reinterpret_cast<int*>(smem + S::OFF_IDX);
  float* scale_s = reinterpret_cast<float*>(smem + S::OFF_SCALE);
  float* red_max = reinterpret_cast<float*>(smem + S::OFF_RED);
  float* red_sum = red_max + 4 * kHeads;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int split = blockIdx.x;
  const int t = blockIdx.y;
  const int h0 = blockIdx.z * kHeads;
  const int seq = (t + p.t_off) / p.q_per_seq;
  const int row_begin = split * p.rows_per_split;
  const int row_end = min(p.K, row_begin + p.rows_per_split);

  const uint8_t* kv_base = p.kv + (int64_t)seq * p.kv_seq_stride;
  const uint8_t* v_base = SEPV ? p.kv_v + (int64_t)seq * p.v_seq_stride : nullptr;
  const float* scale_base = FP8 ? p.kv_scale + (int64_t)seq * p.L : nullptr;

  // q rows h0 .. h0+15 (rows past H are zero); q is a caller input, so it is fetched before
  // waiting for the kernel that produces the index rows
  {
    const __nv_bfloat16* qg = p.q + ((int64_t)t * p.H) * DQK;
    for (int id = tid; id < kHeads * S::QK_CHUNKS; id += kThreads) {
      const int r = id / S::QK_CHUNKS, c = id % S::QK_CHUNKS;
      const bool ok = (h0 + r) < p.H;
      const void* src = ok ? (const void*)(qg + (int64_t)(h0 + r) * DQK + c * 8) : (const void*)p.q;
      cp_async16(q_s + swz(r, c, S::QK_CHUNKS), src, ok);
    }
    cp_async_commit();
  }
  pdl_wait();  // the index rows come from the previous kernel in the stream

  // per-thread softmax state for heads r0 = lane/4 and r1 = lane/4 + 8
  const int r0 = lane >> 2, r1 = r0 + 8;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  constexpr int NT = DV / 32;  // n-tiles of 8 columns per warp in P.V
  float acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  for (int blk = row_begin; blk < row_end; blk += kRows) {
    const int nrows = min(kRows, row_end - blk);
    if (tid < kRows) {
      int i = -1;
      if (tid < nrows) {
        i = p.idx[(int64_t)t * p.K + blk + tid];
        if (i < -1 || i >= p.L) {
          record_error(p.err, DSA_DEVERR_INDEX_RANGE);
          i = -1;
        }
      }
      idx_s[tid] = i;
      if (FP8) scale_s[tid] = (i >= 0) ? scale_base[i] : 0.f;
    }
    __syncthreads();

    // gather: 16-byte pieces, consecutive threads on consecutive pieces of one row
    if (!FP8) {
      for (int id = tid; id < kRows * S::QK_CHUNKS; id += kThreads) {
        const int r = id / S::QK_CHUNKS, c = id % S::QK_CHUNKS;
        const int i = idx_s[r];
        const uint8_t* src = (i >= 0) ? kv_base + (int64_t)i * p.kv_row_stride + c * 16 : p.kv;
        cp_async16(kv_s + swz(r, c, S::QK_CHUNKS), src, i >= 0);
      }
      if (SEPV) {
        for (int id = tid; id < kRows * S::V_CHUNKS; id += kThreads) {
          const int r = id / S::V_CHUNKS, c = id % S::V_CHUNKS;
          const int i = idx_s[r];
          const uint8_t* src = (i >= 0) ? v_base + (int64_t)i * p.v_row_stride + c * 16 : p.kv;
          cp_async16(v_s + swz(r, c, S::V_CHUNKS), src, i >= 0);
        }
      }
      cp_async_commit();
    } else {
      // E4M3 row = DQK bytes = DQK/16 pieces of 16 codes; each piece becomes two bf16 chunks
      constexpr int PIECES = DQK / 16;
      constexpr int PER_THREAD = (kRows * PIECES + kThreads - 1) / kThreads;
      constexpr int BATCH = 6;
#pragma unroll
      for (int b0 = 0; b0 < PER_THREAD; b0 += BATCH) {
        uint4 raw[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
          const int id = tid + (b0 + j) * kThreads;
          raw[j] = make_uint4(0, 0, 0, 0);
          if (b0 + j < PER_THREAD && id < kRows * PIECES) {
            const int r = id / PIECES, c = id % PIECES;
            const int i = idx_s[r];
            if (i >= 0)
              raw[j] = __ldg(reinterpret_cast<const uint4*>(kv_base + (int64_t)i * p.kv_row_stride +
                                                            c * 16));
          }
        }
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
          const int id = tid + (b0 + j) * kThreads;
          if (b0 + j < PER_THREAD && id < kRows * PIECES) {
            const int r = id / PIECES, c = id % PIECES;
            const uint2 a = e4m3x4_to_bf16x4(raw[j].x), b = e4m3x4_to_bf16x4(raw[j].y);
            const uint2 cc = e4m3x4_to_bf16x4(raw[j].z), d = e4m3x4_to_bf16x4(raw[j].w);
            *reinterpret_cast<uint4*>(kv_s + swz(r, 2 * c, S::QK_CHUNKS)) = make_uint4(a.x, a.y, b.x, b.y);
            *reinterpret_cast<uint4*>(kv_s + swz(r, 2 * c + 1, S::QK_CHUNKS)) = make_uint4(cc.x, cc.y, d.x, d.y);
          }
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- S = q . K^T : warp w owns block rows [16w, 16w+16) as two n-tiles of 8
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mat = lane >> 3, rr = lane & 7;
      const uint32_t q_base = smem_u32(q_s);
      const uint32_t kv_base_s = smem_u32(kv_s);
      const int qa_row = rr + (mat & 1) * 8;
      const int kb_row = warp * 16 + rr + (mat >> 1) * 8;
#pragma unroll 4
      for (int ks = 0; ks < DQK / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(q_base + swz(qa_row, 2 * ks + (mat >> 1), S::QK_CHUNKS), a0, a1, a2, a3);
        ldsm_x4(kv_base_s + swz(kb_row, 2 * ks + (mat & 1), S::QK_CHUNKS), b0, b1, b2, b3);
        mma_bf16_16816(s[0], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(s[1], a0, a1, a2, a3, b2, b3);
      }
    }

    // ---- block softmax statistics (log2 domain)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pos = warp * 16 + j * 8 + (lane & 3) * 2 + (e & 1);
        float x = s[j][e] * p.scale_log2;
        if (FP8) x *= scale_s[pos];
        if (idx_s[pos] < 0) x = -INFINITY;
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
      red_max[warp * kHeads + r0] = mx[0];
      red_max[warp * kHeads + r1] = mx[1];
    }
    __syncthreads();
    float m_use[2], alpha[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = hh ? r1 : r0;
      float mb = fmaxf(fmaxf(red_max[h], red_max[kHeads + h]),
                       fmaxf(red_max[2 * kHeads + h], red_max[3 * kHeads + h]));
      const float m_new = fmaxf(m_run[hh], mb);
      m_use[hh] = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[hh] = exp2f(m_run[hh] - m_use[hh]);
      m_run[hh] = m_new;
    }
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int pos0 = warp * 16 + j * 8 + (lane & 3) * 2;
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pv[e] = exp2f(s[j][e] - m_use[e >> 1]);
        psum[e >> 1] += pv[e];
        if (FP8) pv[e] *= scale_s[pos0 + (e & 1)];  // V rows carry the same per-row scale
      }
      // P is stored [head][position], swizzled in 16-byte chunks of 8 positions
      const int c = pos0 >> 3, within = (pos0 & 7) * 2;
      *reinterpret_cast<uint32_t*>(p_s + swz(r0, c, S::P_CHUNKS) + within) = pack_bf16(pv[0], pv[1]);
      *reinterpret_cast<uint32_t*>(p_s + swz(r1, c, S::P_CHUNKS) + within) = pack_bf16(pv[2], pv[3]);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], 1);
      psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], 2);
    }
    if ((lane & 3) == 0) {
      red_sum[warp * kHeads + r0] = psum[0];
      red_sum[warp * kHeads + r1] = psum[1];
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      acc[i][0] *= alpha[0];
      acc[i][1] *= alpha[0];
      acc[i][2] *= alpha[1];
      acc[i][3] *= alpha[1];
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = hh ? r1 : r0;
      const float sb = red_sum[h] + red_sum[kHeads + h] + red_sum[2 * kHeads + h] + red_sum[3 * kHeads + h];
      l_run[hh] = l_run[hh] * alpha[hh] + sb;
    }

    // ---- O += P . V : warp w owns value columns [w*DV/4, (w+1)*DV/4)
    {
      const int mat = lane >> 3, rr = lane & 7;
      const uint32_t p_base = smem_u32(p_s);
      const uint32_t v_base_s = smem_u32(v_s);
      constexpr int VCH = SEPV ? S::V_CHUNKS : S::QK_CHUNKS;  // chunks per smem row holding V
#pragma unroll
      for (int kk = 0; kk < kRows / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(p_base + swz(rr + (mat & 1) * 8, 2 * kk + (mat >> 1), S::P_CHUNKS), a0, a1, a2, a3);
        const int vrow = kk * 16 + rr + (mat & 1) * 8;
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
          const int col_chunk = (warp * (DV / 4)) / 8 + nt + (mat >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(v_base_s + swz(vrow, col_chunk, VCH), b0, b1, b2, b3);
          mma_bf16_16816(acc[nt], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(acc[nt + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();  // smem is rewritten by the next block
  }

  // ---- results for heads h0 + r0, h0 + r1
  const int col0 = warp * (DV / 4) + (lane & 3) * 2;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = h0 + (hh ? r1 : r0);
    if (h >= p.H) continue;
    if (p.splits == 1) {
      const float inv = l_run[hh] > 0.f ? 1.f / l_run[hh] : 0.f;
      __nv_bfloat16* o = p.out + ((int64_t)t * p.H + h) * DV;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        *reinterpret_cast<uint32_t*>(o + col0 + i * 8) =
            pack_bf16(acc[i][2 * hh] * inv, acc[i][2 * hh + 1] * inv);
      }
      if (p.lse && (lane & 3) == 0 && warp == 0)
        p.lse[(int64_t)t * p.H + h] = l_run[hh] > 0.f ? (m_run[hh] + log2f(l_run[hh])) * kLn2 : -INFINITY;
    } else {
      const int64_t row = ((int64_t)t * p.H + h) * p.splits + split;
      float* o = p.part_o + row * DV;
#pragma unroll
      for (int i = 0; i < NT; ++i)
        *reinterpret_cast<float2*>(o + col0 + i * 8) = make_float2(acc[i][2 * hh], acc[i][2 * hh + 1]);
      if ((lane & 3) == 0 && warp == 0)
        *reinterpret_cast<float2*>(p.part_ml + row * 2) = make_float2(m_run[hh], l_run[hh]);
    }
  }
  pdl_launch_dependents();
}

// Merge split partials: out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j,
// lse = (M + log2 sum_j 2^(m_j - M) l_j) * ln 2.  One CTA per (query, head).
template <int DV>
__global__ void __launch_bounds__(DV / 4) lse_combine_kernel(const SparseAttnParams p) {
  pdl_wait();
  const int t = blockIdx.x, h = blockIdx.y;
  const int64_t row = ((int64_t)t * p.H + h) * p.splits;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + row;
  float M = -INFINITY;
  for (int j = 0; j < p.splits; ++j) M = fmaxf(M, ml[j].x);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float lsum = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  const int c = threadIdx.x * 4;
  for (int j = 0; j < p.splits; ++j) {
    const float2 mlj = ml[j];
    const float wj = exp2f(mlj.x - Mu);
    lsum += wj * mlj.y;
    const float4 v = *reinterpret_cast<const float4*>(p.part_o + (row + j) * DV + c);
    o.x += wj * v.x;
    o.y += wj * v.y;
    o.z += wj * v.z;
    o.w += wj * v.w;
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  __nv_bfloat16* out = p.out + ((int64_t)t * p.H + h) * DV + c;
  *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
  if (p.lse && threadIdx.x == 0)
    p.lse[(int64_t)t * p.H + h] = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
  pdl_launch_dependents();
}

template <int DQK, int DV, bool FP8, bool SEPV>
cudaError_t launch_variant(const SparseAttnParams& p, cudaStream_t stream, bool pdl) {
  using S = Smem<DQK, DV, FP8, SEPV>;
  auto kern = sparse_attn_kernel<DQK, DV, FP8, SEPV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, p.T, (p.H + kHeads - 1) / kHeads);
  e = launch_kernel(kern, grid, dim3(kThreads), S::BYTES, stream, pdl, p);
  if (e != cudaSuccess || p.splits == 1) return e;
  return launch_kernel(lse_combine_kernel<DV>, dim3(p.T, p.H), dim3(DV / 4), 0, stream, true, p);
}

}  // namespace

int sparse_attn_splits(int T, int H, int K) {
  // enough CTAs to cover the SMs about twice; each split holds whole 64-row blocks
  const int blocks = (K + kRows - 1) / kRows;
  const int head_groups = (H + kHeads - 1) / kHeads;
  const int ctas_per_split = T * head_groups;
  if (ctas_per_split <= 0) return 1;
  int want = (2 * 152 + ctas_per_split - 1) / ctas_per_split;
  if (want < 1) want = 1;
  if (want > blocks) want = blocks;
  if (want > 64) want = 64;
  return want;
}

size_t sparse_attn_ws_bytes(int T, int H, int K, int D_v) {
  const int splits = sparse_attn_splits(T, H, K);
  if (splits <= 1) return 0;
  const size_t rows = (size_t)T * H * splits;
  return align_up(rows * D_v * sizeof(float), 256) + align_up(rows * 2 * sizeof(float), 256);
}

cudaError_t launch_sparse_attn(SparseAttnParams p, int D_qk, int D_v, bool fp8, bool sepv,
                               void* ws, cudaStream_t stream, bool pdl) {
  p.splits = sparse_attn_splits(p.T, p.H, p.K);
  const int blocks = (p.K + kRows - 1) / kRows;
  p.rows_per_split = ((blocks + p.splits - 1) / p.splits) * kRows;
  p.splits = (p.K + p.rows_per_split - 1) / p.rows_per_split;
  if (p.splits > 1) {
    const size_t rows = (size_t)p.T * p.H * p.splits;
    p.part_o = reinterpret_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) +
                                         align_up(rows * D_v * sizeof(float), 256));
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
