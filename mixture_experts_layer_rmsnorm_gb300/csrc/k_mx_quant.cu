// k_mx_quant.cu -- MXFP8 quantization: bf16 rows -> E4M3 codes + E8M0 scales;
// MXFP4 quantization of the expert weights: bf16 rows -> E2M1 codes + E8M0 scales.
//
// Block scaling over 32 consecutive elements ("CuTeDSL chez Perplexity",
// "Prise en charge de Blackwell": MXFP8 with an absolute maximum over 32
// elements).  Recipe (the OCP Microscaling rule; the pages give none): for a
// block with absolute maximum amax, X = 2^E with E = floor(log2(amax)) - 8
// (8 = the largest E4M3 exponent), clamped to [-127, 127], E = -127 for an
// all-zero block; each element is stored as the E4M3 code of x / X, rounded
// to nearest even and clamped to +-448 (cvt.rn.satfinite); the scale byte is
// E + 127.
//
// MXFP4 (the same pages name Blackwell's block-scaled 4-bit formats beside
// MXFP8; the same OCP rule): E = floor(log2(amax)) - 2 (2 = the largest E2M1
// exponent), codes E2M1 of x / X rounded to nearest even and clamped to +-6.
//
// Codes keep the rows' layout ([rows, K], one byte per element; MXFP4: [rows,
// K/2] bytes, element 2i in the low nibble of byte i).  Scales are
// stored for the tensor cores' block-scaled MMA: per 128-row group and per
// 128-element chunk of K, one 512-byte tile of 32 rows x 16 bytes in which
// byte r*16 + 4*j + b is the scale of row 32*j + r of the group and K-block b
// of the chunk -- the layout tcgen05.cp .32x128b.warpx4 copies into TMEM so
// that the MMA finds row m's scale in lane m, column m/32, byte b.
// Scale row of a matrix row: W13 rows are reordered into the gate/up GEMM's
// tile rows (64 features per tile: 16 gate rows, the matching 16 up rows, x 4);
// W2 keeps its row index.  Token rows (gathered inputs, activations) are
// grouped by the expert GEMMs' token chunks instead: the rows
// [offsets[e] + c*bn, +bn) of expert e form chunk unit_off[e] / tiles + c, and
// its scales ceil(bn / 128) 512-byte tiles per 128 elements of K, tile h with
// byte r*16 + 4*j + b for row offsets[e] + c*bn + 128*h + 32*j + r (bn <= 128,
// or 256 for CTA-pair units; offsets multiples of 32), so that a unit's token
// scales start at TMEM column 0.
#include <cuda_bf16.h>

#include <cstdint>

#include "moe_kernels.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kQuantWarps = 8;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// two E4M3 codes (round to nearest even, saturating): lo in bits 0-7, hi in 8-15
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// eight E2M1 codes (round to nearest even, saturating to +-6): element i in
// bits 4i .. 4i+3
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// byte offset of the scale of (scale row R, K-block kb) for K elements per row
__device__ __forceinline__ size_t scale_offset(int64_t R, int kb, int K) {
  const int64_t g = R >> 7;
  const int rr = static_cast<int>(R & 127);
  return (static_cast<size_t>(g) * (K / 128) + kb / 4) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (kb & 3);
}

// Token row p (< offsets[E]) -> chunk-relative scale position: the "scale row"
// chunk * 128 * G + in_chunk with G = ceil(bn / 128) tiles per chunk, so that
// scale_offset() lands in tile G * chunk + in_chunk / 128.
__device__ __forceinline__ int64_t token_scale_row(int p, const int32_t* offsets, const int32_t* unit_off, int E,
                                                   int tiles, int bn) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldcg(offsets + mid) <= p)
      lo = mid;
    else
      hi = mid;
  }
  const int within = p - __ldcg(offsets + lo);
  const int c = within / bn, in_chunk = within - c * bn;
  const int64_t chunk = __ldcg(unit_off + lo) / tiles + c;
  return chunk * 128 * ((bn + 127) / 128) + in_chunk;  // in_chunk % 128 = 32 * j + r
}

// One warp per row.  MODE 0: rows of a matrix (W2); MODE 1: gathered token
// rows (row p <- h[sorted_ids[p] / k], zeros for padding rows), rows below
// offsets[E] only, chunk-grouped scales; MODE 2: rows of W13, scales in gate/up
// tile-row order; MODE 3: activation rows below offsets[E], chunk-grouped scales.
// FP4: E2M1 codes, packed two per byte, and the block exponent
// floor(log2 amax) - 2 (2 = the largest E2M1 exponent): the weights of both
// FP4 layers (MODE 0 and 2), the token rows and activations of the MXFP4 layer
// (MODE 1 and 3).
template <int MODE, bool FP4 = false>
__global__ void __launch_bounds__(kQuantWarps * 32)
    mx_quantize_kernel(const uint16_t* __restrict__ src, int64_t rows, int K, const int32_t* __restrict__ sorted_ids,
                       const int32_t* __restrict__ offsets, const int32_t* __restrict__ unit_off, int tiles, int bn,
                       int E, int N, int k, int I, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  pdl_wait();  // the rows (and routing tables) may come from the previous kernel
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  if ((MODE == 1 || MODE == 3) && row >= __ldcg(offsets + E)) return;
  const uint16_t* s = nullptr;
  int64_t R = row;  // scale row
  if (MODE == 1 || MODE == 3) R = token_scale_row(static_cast<int>(row), offsets, unit_off, E, tiles, bn);
  if (MODE == 1) {
    const int id = __ldcg(sorted_ids + row);
    if (id >= 0 && id < N) s = src + static_cast<int64_t>(id / k) * K;
  } else {
    s = src + row * K;
    if (MODE == 2) {
      const int64_t e = row / (2 * I);
      const int i = static_cast<int>(row - e * 2 * I);
      const int up = i >= I, f = up ? i - I : i;
      const int m = 32 * ((f & 63) >> 4) + 16 * up + (f & 15);
      R = (e * (I / 64) + (f >> 6)) * 128 + m;
    }
  }
  const int nch = K >> 3;  // 8-element chunks; a 32-block is 4 neighbouring lanes
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int c = c0 + lane;
    const bool on = c < nch;  // whole 4-lane groups are on or off (nch is a multiple of 4)
    float x[8];
    unpack8(on && s ? *reinterpret_cast<const uint4*>(s + c * 8) : make_uint4(0, 0, 0, 0), x);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    int ex = amax > 0.0f ? ilogbf(amax) - (FP4 ? 2 : 8) : -127;
    ex = ex < -127 ? -127 : (ex > 127 ? 127 : ex);
    const float inv = ldexpf(1.0f, -ex);  // exact power of two
    if (FP4) {
      float y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) y[i] = x[i] * inv;
      const uint32_t w = e2m1x8(y);
      if (on) *reinterpret_cast<uint32_t*>(codes + row * (K / 2) + c * 4) = w;
    } else {
      const uint32_t w0 = e4m3x2(x[0] * inv, x[1] * inv) | (e4m3x2(x[2] * inv, x[3] * inv) << 16);
      const uint32_t w1 = e4m3x2(x[4] * inv, x[5] * inv) | (e4m3x2(x[6] * inv, x[7] * inv) << 16);
      if (on) *reinterpret_cast<uint2*>(codes + row * K + c * 8) = make_uint2(w0, w1);
    }
    if (on && (lane & 3) == 0) scales[scale_offset(R, c >> 2, K)] = static_cast<uint8_t>(ex + 127);
  }
}

// ------------------------------------------------------------------ NVFP4
// E2M1 codes (two per byte), one E4M3 scale per 16 elements, one fp32 scale
// per tensor (NVFP4's two-level scaling; the same pages name NVFP4 with an
// absolute maximum over 16 elements): g = amax_tensor / (448 * 6) (1 for an
// all-zero tensor), s = E4M3(amax_16 / (6 g)), q = E2M1(x / (value(s) g)), 0
// where value(s) g = 0.  The scales are not powers of two, so each step is one
// explicitly rounded fp32 operation in this order.  Scale tiles: per 128-row
// group and 64-element chunk of K one 512-byte tile, byte r*16 + 4*j + b = row
// 32*j + r, 16-element block b of the chunk (the MXFP8 tile with 16-element
// blocks: a 32-bit TMEM word then holds the 4 scales of one K = 64 MMA).

__device__ __forceinline__ float nv4_global_of(float amax) {
  return amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
}

// E4M3 code of a non-negative fp32 value (nearest even, saturating to 448) and its value
__device__ __forceinline__ uint32_t e4m3_code(float u) { return e4m3x2(u, 0.0f) & 0xFFu; }
// value of a non-negative E4M3 code (exponent bias 7, 3 mantissa bits; exponent
// field 0: m * 2^-9), built exactly as fp32 bits
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0x1p-9f;
}

__device__ __forceinline__ size_t nv4_scale_offset(int64_t R, int blk, int K) {
  const int64_t g = R >> 7;
  const int rr = static_cast<int>(R & 127);
  return (static_cast<size_t>(g) * (K / 64) + blk / 4) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (blk & 3);
}

// Per expert matrix, the absolute maximum of its rows (rows_per_tensor rows
// each) into amax[e] (zeroed before; fp32 bit patterns of non-negative values
// order as integers).  One warp per row.
__global__ void __launch_bounds__(kQuantWarps * 32)
    nv4_amax_kernel(const uint16_t* __restrict__ src, int64_t rows, int K, int64_t rows_per_tensor,
                    float* __restrict__ amax) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint16_t* s = src + row * K;
  float m = 0.0f;
  for (int c = lane; c < K / 8; c += 32) {
    float x[8];
    unpack8(*reinterpret_cast<const uint4*>(s + c * 8), x);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) atomicMax(reinterpret_cast<int*>(amax + row / rows_per_tensor), __float_as_int(m));
}

// amax[e] -> g[e] in place
__global__ void nv4_global_kernel(float* __restrict__ amax_to_g, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) amax_to_g[i] = nv4_global_of(amax_to_g[i]);
}

// One warp per row.  MODE 0: matrix rows, g from tensor_amax[row / rows_per_tensor];
// MODE 1: gathered token rows, MODE 3: activation rows (rows below offsets[E],
// chunk-grouped scales, g of the row itself, written to g_rows[row]); MODE 2:
// W13 rows in gate/up tile-row order, g from tensor_amax[expert].
template <int MODE>
__global__ void __launch_bounds__(kQuantWarps * 32)
    nv4_quantize_kernel(const uint16_t* __restrict__ src, int64_t rows, int K, const int32_t* __restrict__ sorted_ids,
                        const int32_t* __restrict__ offsets, const int32_t* __restrict__ unit_off, int tiles, int bn,
                        int E, int N, int k, int I, int64_t rows_per_tensor, const float* __restrict__ tensor_amax,
                        uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, float* __restrict__ g_rows) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  if ((MODE == 1 || MODE == 3) && row >= __ldcg(offsets + E)) return;
  const uint16_t* s = nullptr;
  int64_t R = row;  // scale row
  if (MODE == 1 || MODE == 3) R = token_scale_row(static_cast<int>(row), offsets, unit_off, E, tiles, bn);
  if (MODE == 1) {
    const int id = __ldcg(sorted_ids + row);
    if (id >= 0 && id < N) s = src + static_cast<int64_t>(id / k) * K;
  } else {
    s = src + row * K;
    if (MODE == 2) {
      const int64_t e = row / (2 * I);
      const int i = static_cast<int>(row - e * 2 * I);
      const int up = i >= I, f = up ? i - I : i;
      const int m = 32 * ((f & 63) >> 4) + 16 * up + (f & 15);
      R = (e * (I / 64) + (f >> 6)) * 128 + m;
    }
  }
  const int nch = K >> 3;  // 8-element chunks; a 16-block is 2 neighbouring lanes
  float g;
  if (MODE == 1 || MODE == 3) {
    float m = 0.0f;
    for (int c = lane; c < nch; c += 32) {
      float x[8];
      unpack8(s ? *reinterpret_cast<const uint4*>(s + c * 8) : make_uint4(0, 0, 0, 0), x);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    g = nv4_global_of(m);
    if (lane == 0) g_rows[row] = g;
  } else {
    g = nv4_global_of(__ldg(tensor_amax + row / rows_per_tensor));
  }
  const float six_g = __fmul_rn(6.0f, g);
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int c = c0 + lane;
    const bool on = c < nch;  // whole lane pairs are on or off (nch is even: K is a multiple of 128)
    float x[8];
    unpack8(on && s ? *reinterpret_cast<const uint4*>(s + c * 8) : make_uint4(0, 0, 0, 0), x);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    const uint32_t sc = e4m3_code(__fdiv_rn(amax, six_g));
    const float X = __fmul_rn(e4m3_value(sc), g);
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = X > 0.0f ? __fdiv_rn(x[i], X) : 0.0f;
    uint32_t w = e2m1x8(y);
    if (!(X > 0.0f)) w = 0;  // code 0 (not a signed zero) where the block scale is 0
    if (on) {
      *reinterpret_cast<uint32_t*>(codes + row * (K / 2) + c * 4) = w;
      if ((lane & 1) == 0) scales[nv4_scale_offset(R, c >> 1, K)] = static_cast<uint8_t>(sc);
    }
  }
}

}  // namespace

cudaError_t launch_nv4_weight_amax(const uint16_t* src, int64_t rows, int K, int64_t rows_per_tensor, float* amax,
                                   int n_tensors, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float) * n_tensors, stream);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  nv4_amax_kernel<<<static_cast<unsigned>(blocks), kQuantWarps * 32, 0, stream>>>(src, rows, K, rows_per_tensor,
                                                                                   amax);
  return cudaGetLastError();
}

cudaError_t launch_nv4_global(float* amax_to_g, int n, cudaStream_t stream) {
  nv4_global_kernel<<<(n + 127) / 128, 128, 0, stream>>>(amax_to_g, n);
  return cudaGetLastError();
}

cudaError_t launch_nv4_quantize_rows(const uint16_t* src, int64_t rows, int K, int64_t rows_per_tensor,
                                     const float* tensor_amax, uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(nv4_quantize_kernel<0>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0, stream,
                    src, rows, K, nullptr, nullptr, nullptr, 1, 32, 0, 0, 1, 0, rows_per_tensor, tensor_amax, codes,
                    scales, nullptr);
}

cudaError_t launch_nv4_quantize_w13(const uint16_t* w13, int E, int H, int I, const float* tensor_amax,
                                    uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(E) * 2 * I;
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(nv4_quantize_kernel<2>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0, stream,
                    w13, rows, H, nullptr, nullptr, nullptr, 1, 32, 0, 0, 1, I, static_cast<int64_t>(2) * I,
                    tensor_amax, codes, scales, nullptr);
}

cudaError_t launch_nv4_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets,
                              const int32_t* unit_off, int tiles, int bn, int E, int N, int k, int H, int64_t rows,
                              uint8_t* codes, uint8_t* scales, float* g_rows, cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(nv4_quantize_kernel<1>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0, stream,
                    h, rows, H, sorted_ids, offsets, unit_off, tiles, bn, E, N, k, 0, static_cast<int64_t>(1),
                    nullptr, codes, scales, g_rows);
}

cudaError_t launch_nv4_quantize_act(const uint16_t* act, int64_t rows, int K, const int32_t* offsets,
                                    const int32_t* unit_off, int tiles, int bn, int E, uint8_t* codes,
                                    uint8_t* scales, float* g_rows, cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(nv4_quantize_kernel<3>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0, stream,
                    act, rows, K, nullptr, offsets, unit_off, tiles, bn, E, 0, 1, 0, static_cast<int64_t>(1), nullptr,
                    codes, scales, g_rows);
}

cudaError_t launch_mx_quantize_rows(const uint16_t* src, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(mx_quantize_kernel<0>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0, stream,
                    src, rows, K, nullptr, nullptr, nullptr, 1, 32, 0, 0, 1, 0, codes, scales);
}

cudaError_t launch_mx_quantize_act(const uint16_t* act, int64_t rows, int K, const int32_t* offsets,
                                   const int32_t* unit_off, int tiles, int bn, int E, uint8_t* codes, uint8_t* scales,
                                   cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(mx_quantize_kernel<3>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0, stream,
                    act, rows, K, nullptr, offsets, unit_off, tiles, bn, E, 0, 1, 0, codes, scales);
}

cudaError_t launch_mx_quantize_w13(const uint16_t* w13, int E, int H, int I, uint8_t* codes, uint8_t* scales,
                                   cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(E) * 2 * I;
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(mx_quantize_kernel<2>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0, stream,
                    w13, rows, H, nullptr, nullptr, nullptr, 1, 32, 0, 0, 1, I, codes, scales);
}

cudaError_t launch_mx4_quantize_rows(const uint16_t* src, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                                     cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(mx_quantize_kernel<0, true>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0,
                    stream, src, rows, K, nullptr, nullptr, nullptr, 1, 32, 0, 0, 1, 0, codes, scales);
}

cudaError_t launch_mx4_quantize_w13(const uint16_t* w13, int E, int H, int I, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(E) * 2 * I;
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(mx_quantize_kernel<2, true>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0,
                    stream, w13, rows, H, nullptr, nullptr, nullptr, 1, 32, 0, 0, 1, I, codes, scales);
}

cudaError_t launch_mx4_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets,
                              const int32_t* unit_off, int tiles, int bn, int E, int N, int k, int H, int64_t rows,
                              uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(mx_quantize_kernel<1, true>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0,
                    stream, h, rows, H, sorted_ids, offsets, unit_off, tiles, bn, E, N, k, 0, codes, scales);
}

cudaError_t launch_mx4_quantize_act(const uint16_t* act, int64_t rows, int K, const int32_t* offsets,
                                    const int32_t* unit_off, int tiles, int bn, int E, uint8_t* codes,
                                    uint8_t* scales, cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(mx_quantize_kernel<3, true>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0,
                    stream, act, rows, K, nullptr, offsets, unit_off, tiles, bn, E, 0, 1, 0, codes, scales);
}

cudaError_t launch_mx_gather(const uint16_t* h, const int32_t* sorted_ids, const int32_t* offsets,
                             const int32_t* unit_off, int tiles, int bn, int E, int N, int k, int H, int64_t rows,
                             uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantWarps - 1) / kQuantWarps;
  return launch_pdl(mx_quantize_kernel<1>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0, stream,
                    h, rows, H, sorted_ids, offsets, unit_off, tiles, bn, E, N, k, 0, codes, scales);
}

}  // namespace moe
