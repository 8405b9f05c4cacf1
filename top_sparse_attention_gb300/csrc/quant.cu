// Online quantisation that writes the caches the chain reads (the step before the indexer scores
// and the gather): indexer rows to MXFP8, latent KV rows to FP8 with one scale per row ("Day 0
// Support for New LLM Architectures", Key Optimization 2: MXFP8 with groups of 32 sharing one
// scale for the indexer, FP8 for the sparse-attention KV cache).
//
// Group scales follow the OCP Microscaling Formats specification v1.0: the shared exponent is
// floor(log2 amax) - 8 (8 is E4M3's largest exponent), clamped to E8M0's range [-127, 127], and 0
// for an all-zero group; the exponent byte is that exponent + 127.  Elements are rounded to the
// nearest E4M3 value, ties to even, saturating to +-448.  Dividing by the power-of-two group scale
// is exact, so the element codes depend on no rounding of ours.  FP8 rows use s = amax / 448 (1
// for an all-zero row) and the codes of x / s, both IEEE fp32 divisions (round to nearest).  (A
// reciprocal 448 / amax would save the per-element division but leaves fp32's range for rows
// whose amax is below 448 / FLT_MAX, e.g. rows of bf16 subnormals.)
//
// One warp per input row.  Generic forms: lane j holds elements j, j + 32, ..., so a group of 32
// is one warp-wide max and every store is coalesced; vector forms (below) move four elements per
// lane.  Input row r goes to destination row dst_rows[r] (or r; a negative entry drops the row),
// which makes the same kernels the cache append: destination row = sequence * L + position.
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kRowsPerCta = 8;  // one warp each

__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// |v| of finite floats orders like the bit patterns, so the warp max runs on integers.
__device__ __forceinline__ float warp_amax(float a) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(a))));
}

// The E4M3 code of the IEEE quotient x / s (fp32, round to nearest), without a division per
// element.  Per row: r = 1/s correctly rounded, usable when s and r are normal floats.  Per element:
// q0 = x * r lies within 2.5 fp32 ulps of x / s rounded, and E4M3 rounding is monotone, so the two
// give the same code unless an E4M3 rounding midpoint lies that close to q0.  A midpoint of two
// normal E4M3 values (those two a binade apart included) has fp32 mantissa bit 19 set and bits
// 18..0 clear, so a q0 whose low 20 bits are within 4 of 0x80000 takes the division, and so does
// a q0 in E4M3's subnormal range (below 2^-6), whose midpoints sit elsewhere.
struct Quotient {
  float s, r;
  bool fast;
  __device__ explicit Quotient(float s_) : s(s_) {
    r = __frcp_rn(s_);
    fast = s_ >= 0x1p-126f && r >= 0x1p-126f && r <= 0x1p126f;
  }
  // q0, and whether it gives the code of the IEEE quotient
  __device__ __forceinline__ float fast_part(float x, bool* exact) const {
    const float q0 = x * r;
    const uint32_t low = __float_as_uint(q0) & 0xFFFFFu;
    *exact = fast && !(low - 0x7FFFCu <= 8u || fabsf(q0) < 0x1p-6f);
    return q0;
  }
  __device__ __forceinline__ float operator()(float x) const {
    bool exact;
    const float q0 = fast_part(x, &exact);
    return exact ? q0 : __fdiv_rn(x, s);
  }
};

__global__ void __launch_bounds__(32 * kRowsPerCta) mxfp8_quant_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t x_row_stride, int rows, int d,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, const int64_t* __restrict__ dst_rows) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int64_t dst = dst_rows ? dst_rows[r] : r;
  if (dst < 0) return;
  const __nv_bfloat16* src = x + (int64_t)r * x_row_stride;
  uint8_t* out = codes + dst * d;
  uint8_t* out_sf = sf + dst * (d / 32);
  for (int g = 0; g < d / 32; ++g) {
    const float v = __bfloat162float(src[g * 32 + lane]);
    const float amax = warp_amax(v);
    int e = 0;
    if (amax > 0.f) e = min(max(ilogbf(amax) - 8, -127), 127);
    out[g * 32 + lane] = to_e4m3(v * ldexpf(1.f, -e));  // a power of two: exact
    if (lane == 0) out_sf[g] = (uint8_t)(e + 127);
  }
}

__global__ void __launch_bounds__(32 * kRowsPerCta) fp8_rows_quant_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t x_row_stride, int rows, int width,
    uint8_t* __restrict__ codes, int64_t code_row_stride, float* __restrict__ scales,
    const int64_t* __restrict__ dst_rows) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int64_t dst = dst_rows ? dst_rows[r] : r;
  if (dst < 0) return;
  const __nv_bfloat16* src = x + (int64_t)r * x_row_stride;
  float a = 0.f;
  for (int j = lane; j < width; j += 32) a = fmaxf(a, fabsf(__bfloat162float(src[j])));
  const float amax = warp_amax(a);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint8_t* out = codes + dst * code_row_stride;
  const Quotient div(s);
  for (int j = lane; j < width; j += 32) out[j] = to_e4m3(div(__bfloat162float(src[j])));
  if (lane == 0) scales[dst] = s;
}

// Vector forms: each lane moves four elements (8 bytes of bf16 in, 4 code bytes out), so a warp
// covers 128 elements per step.  MXFP8 rows with d a multiple of 128: a group of 32 is 8 lanes
// and its max takes three shuffles.  FP8 rows with width a multiple of 4.  Both need 8-byte
// aligned source rows and 4-byte aligned code rows (checked on the host).

__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  v[0] = a.x, v[1] = a.y, v[2] = b.x, v[3] = b.y;
}

__device__ __forceinline__ uint32_t pack4(uint8_t a, uint8_t b, uint8_t c, uint8_t d) {
  return (uint32_t)a | (uint32_t)b << 8 | (uint32_t)c << 16 | (uint32_t)d << 24;
}

__global__ void __launch_bounds__(32 * kRowsPerCta) mxfp8_quant_vec_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t x_row_stride, int rows, int d,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, const int64_t* __restrict__ dst_rows) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int64_t dst = dst_rows ? dst_rows[r] : r;
  if (dst < 0) return;
  const __nv_bfloat16* src = x + (int64_t)r * x_row_stride;
  uint8_t* out = codes + dst * d;
  uint8_t* out_sf = sf + dst * (d / 32);
  for (int c = 0; c < d; c += 128) {
    float v[4];
    load4(src + c + 4 * lane, v);
    float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));  // 8 lanes
    int e = 0;
    if (a > 0.f) e = min(max(ilogbf(a) - 8, -127), 127);
    const float inv = ldexpf(1.f, -e);  // a power of two: exact
    *reinterpret_cast<uint32_t*>(out + c + 4 * lane) =
        pack4(to_e4m3(v[0] * inv), to_e4m3(v[1] * inv), to_e4m3(v[2] * inv), to_e4m3(v[3] * inv));
    if ((lane & 7) == 0) out_sf[c / 32 + (lane >> 3)] = (uint8_t)(e + 127);
  }
}

__global__ void __launch_bounds__(32 * kRowsPerCta) fp8_rows_quant_vec_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t x_row_stride, int rows, int width,
    uint8_t* __restrict__ codes, int64_t code_row_stride, float* __restrict__ scales,
    const int64_t* __restrict__ dst_rows) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int64_t dst = dst_rows ? dst_rows[r] : r;
  if (dst < 0) return;
  const __nv_bfloat16* src = x + (int64_t)r * x_row_stride;
  float a = 0.f;
  for (int j = 4 * lane; j < width; j += 128) {
    float v[4];
    load4(src + j, v);
    a = fmaxf(a, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
  }
  const float amax = warp_amax(a);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint8_t* out = codes + dst * code_row_stride;
  const Quotient div(s);
  for (int j = 4 * lane; j < width; j += 128) {
    float v[4];
    load4(src + j, v);
    *reinterpret_cast<uint32_t*>(out + j) = pack4(to_e4m3(div(v[0])), to_e4m3(div(v[1])), to_e4m3(div(v[2])),
                                                  to_e4m3(div(v[3])));
  }
  if (lane == 0) scales[dst] = s;
}

// Wide forms: 16-byte loads (eight elements per lane) and 8-byte code stores.
//  * MXFP8: a warp takes kRowsPerWarp8 consecutive rows as one flat run of 8-element chunks; four
//    consecutive lanes hold a group of 32 (d is a multiple of 32, so groups never straddle rows)
//    and its max takes two shuffles.
//  * FP8 rows (width a multiple of 8, at most 32 * 8 * kMaxChunks8): two passes, the second
//    re-reading the row from L2.

constexpr int kRowsPerWarp8 = 8;
constexpr int kMaxChunks8 = 4;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    v[2 * i] = f.x, v[2 * i + 1] = f.y;
  }
}

__global__ void __launch_bounds__(32 * kRowsPerCta) mxfp8_quant_v8_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t x_row_stride, int rows, int d,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, const int64_t* __restrict__ dst_rows) {
  const int lane = threadIdx.x & 31;
  const int r0 = (blockIdx.x * kRowsPerCta + (threadIdx.x >> 5)) * kRowsPerWarp8;
  if (r0 >= rows) return;
  const int cpr = d / 8;  // chunks per row
  const int nrows = min(kRowsPerWarp8, rows - r0);
  for (int c0 = 0; c0 < nrows * cpr; c0 += 32) {
    const int c = c0 + lane;
    const bool in = c < nrows * cpr;  // whole groups of four lanes agree (cpr % 4 == 0)
    const int r = r0 + (in ? c / cpr : 0), k = c % cpr;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (in) load8(x + (int64_t)r * x_row_stride + 8 * k, v);
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    const int64_t dst = in ? (dst_rows ? dst_rows[r] : r) : -1;
    if (dst < 0) continue;
    int e = 0;
    if (a > 0.f) e = min(max(ilogbf(a) - 8, -127), 127);
    const float inv = ldexpf(1.f, -e);  // a power of two: exact
    uint8_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = to_e4m3(v[i] * inv);
    *reinterpret_cast<uint2*>(codes + dst * d + 8 * k) =
        make_uint2(pack4(q[0], q[1], q[2], q[3]), pack4(q[4], q[5], q[6], q[7]));
    if ((k & 3) == 0) sf[dst * (d / 32) + k / 4] = (uint8_t)(e + 127);
  }
}

__global__ void __launch_bounds__(32 * kRowsPerCta) fp8_rows_quant_v8_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t x_row_stride, int rows, int width,
    uint8_t* __restrict__ codes, int64_t code_row_stride, float* __restrict__ scales,
    const int64_t* __restrict__ dst_rows) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int64_t dst = dst_rows ? dst_rows[r] : r;
  if (dst < 0) return;
  const __nv_bfloat16* src = x + (int64_t)r * x_row_stride;
  const int nch = width / 8;
  // two passes over the row: the first (from HBM) keeps only the running max, the second re-reads
  // the row from L2; few registers per thread keep many rows in flight per SM
  float a = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxChunks8; ++j) {
    const int c = lane + 32 * j;
    if (c < nch) {
      float v[8];
      load8(src + 8 * c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    }
  }
  const float amax = warp_amax(a);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint8_t* out = codes + dst * code_row_stride;
  const Quotient div(s);
#pragma unroll 1
  for (int c = lane; c < nch; c += 32) {
    float v[8];
    load8(src + 8 * c, v);
    uint8_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = to_e4m3(div(v[i]));
    *reinterpret_cast<uint2*>(out + 8 * c) = make_uint2(pack4(q[0], q[1], q[2], q[3]), pack4(q[4], q[5], q[6], q[7]));
  }
  if (lane == 0) scales[dst] = s;
}

// Tiles: one warp per (row, tile); the tile is quantised as a row of fp8_rows_quant_kernel.
__global__ void __launch_bounds__(32 * kRowsPerCta) fp8_tiles_quant_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t x_row_stride, int rows, int width, int tile,
    uint8_t* __restrict__ codes, int64_t code_row_stride, float* __restrict__ scales,
    const int64_t* __restrict__ dst_rows) {
  const int lane = threadIdx.x & 31;
  const int ntile = (width + tile - 1) / tile;
  const int64_t w = (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);  // (row, tile) index
  if (w >= (int64_t)rows * ntile) return;
  const int r = (int)(w / ntile), c = (int)(w % ntile);
  const int64_t dst = dst_rows ? dst_rows[r] : r;
  if (dst < 0) return;
  const int lo = c * tile, n = min(tile, width - lo);
  const __nv_bfloat16* src = x + (int64_t)r * x_row_stride + lo;
  float a = 0.f;
  for (int j = lane; j < n; j += 32) a = fmaxf(a, fabsf(__bfloat162float(src[j])));
  const float amax = warp_amax(a);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint8_t* out = codes + dst * code_row_stride + lo;
  const Quotient div(s);
  for (int j = lane; j < n; j += 32) out[j] = to_e4m3(div(__bfloat162float(src[j])));
  if (lane == 0) scales[dst * ntile + c] = s;
}

bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }
bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

dsa_status dsa_quantize_mxfp8(const void* x, int64_t x_row_stride, int rows, int d, uint8_t* codes,
                              uint8_t* sf, const int64_t* dst_rows, void* stream) {
  if (rows < 0 || d <= 0 || d % 32 != 0 || x_row_stride < d) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!x || !codes || !sf || !aligned2(x)) return DSA_ERR_INVALID_ARG;
  dsa_status s = check_device_arch();
  if (s != DSA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  if (aligned(x, 16) && x_row_stride % 8 == 0 && aligned(codes, 8)) {
    const int per_cta = kRowsPerCta * kRowsPerWarp8;
    mxfp8_quant_v8_kernel<<<(rows + per_cta - 1) / per_cta, 32 * kRowsPerCta, 0, st>>>(
        xb, x_row_stride, rows, d, codes, sf, dst_rows);
  } else {
    const int grid = (rows + kRowsPerCta - 1) / kRowsPerCta;
    auto kern = (d % 128 == 0 && aligned(x, 8) && x_row_stride % 4 == 0 && aligned(codes, 4))
                    ? mxfp8_quant_vec_kernel : mxfp8_quant_kernel;
    kern<<<grid, 32 * kRowsPerCta, 0, st>>>(xb, x_row_stride, rows, d, codes, sf, dst_rows);
  }
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_quantize_fp8_rows(const void* x, int64_t x_row_stride, int rows, int width,
                                 uint8_t* codes, int64_t code_row_stride, float* scales,
                                 const int64_t* dst_rows, void* stream) {
  if (rows < 0 || width <= 0 || x_row_stride < width || code_row_stride < width)
    return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!x || !codes || !scales || !aligned2(x)) return DSA_ERR_INVALID_ARG;
  dsa_status s = check_device_arch();
  if (s != DSA_OK) return s;
  const int grid = (rows + kRowsPerCta - 1) / kRowsPerCta;
  auto kern = (width % 8 == 0 && width <= 256 * kMaxChunks8 && aligned(x, 16) && x_row_stride % 8 == 0 &&
               aligned(codes, 8) && code_row_stride % 8 == 0)
                  ? fp8_rows_quant_v8_kernel
                  : (width % 4 == 0 && aligned(x, 8) && x_row_stride % 4 == 0 && aligned(codes, 4) &&
                     code_row_stride % 4 == 0)
                        ? fp8_rows_quant_vec_kernel : fp8_rows_quant_kernel;
  kern<<<grid, 32 * kRowsPerCta, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), x_row_stride, rows, width, codes, code_row_stride,
      scales, dst_rows);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_quantize_fp8_tiles(const void* x, int64_t x_row_stride, int rows, int width, int tile,
                                  uint8_t* codes, int64_t code_row_stride, float* scales,
                                  const int64_t* dst_rows, void* stream) {
  if (rows < 0 || width <= 0 || tile < 1 || tile > 1024 || x_row_stride < width || code_row_stride < width)
    return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!x || !codes || !scales || !aligned2(x)) return DSA_ERR_INVALID_ARG;
  dsa_status s = check_device_arch();
  if (s != DSA_OK) return s;
  const int64_t items = (int64_t)rows * ((width + tile - 1) / tile);
  const int64_t grid = (items + kRowsPerCta - 1) / kRowsPerCta;
  if (grid >= (1ll << 31)) return DSA_ERR_UNSUPPORTED;
  fp8_tiles_quant_kernel<<<(unsigned)grid, 32 * kRowsPerCta, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), x_row_stride, rows, width, tile, codes, code_row_stride,
      scales, dst_rows);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // extern "C"
