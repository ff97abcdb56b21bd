// k_qk_norm.cu -- QK-norm: RMSNorm of every attention head of Q and K, in place.
//
// "CuTeDSL chez Perplexity", "Norme QK": the norm of recent Qwen attention
// layers, applied per head over head_dim = 64, 128 or 256 elements, with one
// weight vector for the heads of Q and one for the heads of K and a constant
// weight bias:
//   out_j = (w_j + weight_bias) * (x_j * rstd),  rstd = 1/sqrt(mean_j x_j^2 + eps).
// Heads are small, so no shared memory is needed: each thread takes 128 bits
// (8 bf16) of a head, D/8 consecutive lanes hold one head (a half-warp for
// D = 128, several heads per warp for D = 64), and the sum of squares is
// reduced across those lanes with an xor butterfly of shuffles.
//
// Precision: fp32, one fixed order -- each thread sums the squares of its 8
// elements in index order (fused multiply-add from +0), then
// v += shfl_xor(v, off) for off = D/16, ..., 1; mean = ss / D,
// rstd = 1 / sqrt(mean + eps) with IEEE division and square root; then
// bf16((w_j + weight_bias) * (x_j * rstd)) -- all roundings explicit.
#include <cuda_bf16.h>

#include <cstdint>

#include "moe_kernels.cuh"

namespace moe {
namespace {

constexpr int kQkThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t bf16_bits_rn(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// q [T, Hq, D] is a flat list of T*Hq heads and k of T*Hk heads, all heads of
// a tensor sharing its weight vector; the kernel walks the n_q + n_k heads (q's
// first) without any division.  Each thread keeps its 16-byte part of the two
// weight vectors in registers; block b takes the V
// groups of kQkThreads / TPH consecutive heads starting at head b * V * HPB
// (then + gridDim.x * V * HPB), issuing all V loads before the first
// reduction.
template <int D, int V>
__global__ void __launch_bounds__(kQkThreads, 4)
    qk_norm_kernel(uint16_t* __restrict__ q, uint16_t* __restrict__ k, const uint16_t* __restrict__ q_weight,
                   const uint16_t* __restrict__ k_weight, uint32_t n_q, uint32_t n_k, float weight_bias, float eps) {
  constexpr int TPH = D / 8;              // lanes per head
  constexpr int HPB = kQkThreads / TPH;   // heads per block and pass
  static_assert(TPH >= 1 && TPH <= 32 && (32 % TPH) == 0, "head_dim");
  const uint32_t part = threadIdx.x % TPH;
  const uint32_t local = threadIdx.x / TPH;
  const uint32_t n = n_q + n_k;
  // this thread's 8 elements of the two weight vectors (bf16, kept packed)
  const uint4 wq = n_q ? __ldg(reinterpret_cast<const uint4*>(q_weight + part * 8)) : make_uint4(0, 0, 0, 0);
  const uint4 wk = n_k ? __ldg(reinterpret_cast<const uint4*>(k_weight + part * 8)) : make_uint4(0, 0, 0, 0);
  for (uint32_t base = blockIdx.x * (V * HPB); base < n; base += gridDim.x * (V * HPB)) {
    uint4 xv[V];
    uint16_t* row[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const uint32_t h = base + v * HPB + local;  // whole head groups are in range or not
      row[v] = h < n_q ? q + static_cast<size_t>(h) * D : k + static_cast<size_t>(h - n_q) * D;
      xv[v] = h < n ? *reinterpret_cast<const uint4*>(row[v] + part * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const uint32_t h = base + v * HPB + local;
      const bool is_q = h < n_q;
      float x[8];
      unpack8(xv[v], x);
      float ss = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = __fmaf_rn(x[i], x[i], ss);
#pragma unroll
      for (int off = TPH / 2; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
      const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), eps)));
      float w[8];
      unpack8(is_q ? wq : wk, w);
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float g0 = __fadd_rn(w[2 * i], weight_bias), g1 = __fadd_rn(w[2 * i + 1], weight_bias);
        o[i] = bf16_bits_rn(__fmul_rn(g0, __fmul_rn(x[2 * i], rstd))) |
               (bf16_bits_rn(__fmul_rn(g1, __fmul_rn(x[2 * i + 1], rstd))) << 16);
      }
      if (h < n) *reinterpret_cast<uint4*>(row[v] + part * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

template <int D>
cudaError_t launch_qk_t(uint16_t* q, uint16_t* k, const uint16_t* qw, const uint16_t* kw, int64_t T, int Hq, int Hk,
                        float wb, float eps, cudaStream_t stream) {
  constexpr int V = 4;
  constexpr int HPB = kQkThreads / (D / 8);
  const int64_t n_q = T * Hq, n_k = T * Hk;
  if (n_q + n_k >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int64_t blocks = (n_q + n_k + V * HPB - 1) / (V * HPB);
  qk_norm_kernel<D, V><<<static_cast<unsigned>(blocks), kQkThreads, 0, stream>>>(
      q, k, qw, kw, static_cast<uint32_t>(n_q), static_cast<uint32_t>(n_k), wb, eps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm(uint16_t* q, uint16_t* k, const uint16_t* q_weight, const uint16_t* k_weight, int64_t T,
                           int Hq, int Hk, int D, float weight_bias, float eps, cudaStream_t stream) {
  switch (D) {
    case 64: return launch_qk_t<64>(q, k, q_weight, k_weight, T, Hq, Hk, weight_bias, eps, stream);
    case 128: return launch_qk_t<128>(q, k, q_weight, k_weight, T, Hq, Hk, weight_bias, eps, stream);
    case 256: return launch_qk_t<256>(q, k, q_weight, k_weight, T, Hq, Hk, weight_bias, eps, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
