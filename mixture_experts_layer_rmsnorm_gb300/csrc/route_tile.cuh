// route_tile.cuh -- RMSNorm + router logits of one tile of tokens x experts
// (used by the router kernel and by the single-launch decode front end).
//
// RMSNorm ("4 · La fusion de noyaux", §4.2 "Réduction + élémentaire"; "CuTeDSL
// chez Perplexity", "Norme QK"): one warp per token row, 128-bit loads of 8
// bf16 per lane, fp32 sum of squares reduced by an xor butterfly of warp
// shuffles, h = bf16((x * rstd) * g) with rstd = 1/sqrt(mean + eps).
//
// Router: l_e = sum_j h_j Wr[e,j] (+ b_e) in fp32.  Every dot product (and
// the sum of squares) is taken in one fixed order so that the routing
// decision is reproducible bit for bit:
//   chunk c = elements [8c, 8c+8) belongs to lane c mod 32; a lane runs over
//   its chunks in increasing c, one fused multiply-add per element in
//   increasing index, from +0; the 32 lane sums are combined by
//   v += shfl_xor(v, off) for off = 16, 8, 4, 2, 1.
// All roundings are explicit (__fmaf_rn, __fadd_rn, __fmul_rn, __fdiv_rn,
// __fsqrt_rn), so the compiler cannot contract or reorder them.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace moe {
namespace rt {

constexpr int kRouteWarps = 8;  // warps of a CTA running a tile
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

__device__ __forceinline__ float warp_butterfly_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
  return v;
}

// Pull the router rows [e0, e_hi) and the norm gain into L2 (they do not
// depend on earlier kernels).  All threads of the CTA.
__device__ __forceinline__ void route_prefetch(const float* w_router, const uint16_t* g, int H, int e0, int e_hi) {
  const char* wb = reinterpret_cast<const char*>(w_router + static_cast<size_t>(e0) * H);
  const size_t wbytes = static_cast<size_t>(max(e_hi - e0, 0)) * H * 4;
  for (size_t off = static_cast<size_t>(threadIdx.x) * 128; off < wbytes; off += 128 * blockDim.x)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(wb + off));
  const char* gb = reinterpret_cast<const char*>(g);
  for (int off = threadIdx.x * 128; off < H * 2; off += 128 * blockDim.x)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(gb + off));
}

// h = bf16((x * rstd) * g) for the chunks [8c, 8c+8) of one row
__device__ __forceinline__ uint4 norm_chunk(const uint4& xv, const uint4& gv, float rstd) {
  float f[8], gg[8];
  unpack8(xv, f);
  unpack8(gv, gg);
  uint4 o;
  o.x = pack2_bf16(__fmul_rn(__fmul_rn(f[0], rstd), gg[0]), __fmul_rn(__fmul_rn(f[1], rstd), gg[1]));
  o.y = pack2_bf16(__fmul_rn(__fmul_rn(f[2], rstd), gg[2]), __fmul_rn(__fmul_rn(f[3], rstd), gg[3]));
  o.z = pack2_bf16(__fmul_rn(__fmul_rn(f[4], rstd), gg[4]), __fmul_rn(__fmul_rn(f[5], rstd), gg[5]));
  o.w = pack2_bf16(__fmul_rn(__fmul_rn(f[6], rstd), gg[6]), __fmul_rn(__fmul_rn(f[7], rstd), gg[7]));
  return o;
}

__device__ __forceinline__ float rms_rstd(float ss, int H, float eps) {
  ss = warp_butterfly_sum(ss);
  const float ms = __fdiv_rn(ss, static_cast<float>(H));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// One round of the logits loop: chunks c0 + 32 d (d < DEPTH) of TE router
// rows, all loaded before the first FMA, then accumulated in chunk order.
// MASKED: skip the chunks at or past nch.
template <int TT, int TE, int DEPTH, bool MASKED>
__device__ __forceinline__ void gemv_round(const float4* const (&wrow)[TE], const uint4* h_s, int nch, int c0,
                                           float (&acc)[TT][TE]) {
  float4 wv[DEPTH][TE][2];
#pragma unroll
  for (int d = 0; d < DEPTH; ++d)
#pragma unroll
    for (int b = 0; b < TE; ++b) {
      if (!MASKED || c0 + 32 * d < nch) {
        wv[d][b][0] = __ldg(wrow[b] + 2 * (c0 + 32 * d));
        wv[d][b][1] = __ldg(wrow[b] + 2 * (c0 + 32 * d) + 1);
      }
    }
#pragma unroll
  for (int d = 0; d < DEPTH; ++d) {
    const int c = c0 + 32 * d;
    if (!MASKED || c < nch) {
#pragma unroll
      for (int a = 0; a < TT; ++a) {
        float hv[8];
        unpack8(h_s[a * nch + c], hv);
#pragma unroll
        for (int b = 0; b < TE; ++b) {
          const float w[8] = {wv[d][b][0].x, wv[d][b][0].y, wv[d][b][0].z, wv[d][b][0].w,
                              wv[d][b][1].x, wv[d][b][1].y, wv[d][b][1].z, wv[d][b][1].w};
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[a][b] = __fmaf_rn(hv[i], w[i], acc[a][b]);
        }
      }
    }
  }
}

// The same round for tokens taken two at a time: one paired fp32 FMA
// (fma.rn.f32x2, each half rounded exactly as a single fused multiply-add)
// updates the accumulators of tokens 2p and 2p+1 for one expert, so every
// accumulator still sees its products in the canonical order and the logits
// are bit for bit those of gemv_round, in half the FMA instructions.
template <int TT, int TE, int DEPTH, bool MASKED>
__device__ __forceinline__ void gemv_round_paired(const float4* const (&wrow)[TE], const uint4* h_s, int nch, int c0,
                                                  float2 (&acc)[TT / 2][TE]) {
  float4 wv[DEPTH][TE][2];
#pragma unroll
  for (int d = 0; d < DEPTH; ++d)
#pragma unroll
    for (int b = 0; b < TE; ++b) {
      if (!MASKED || c0 + 32 * d < nch) {
        wv[d][b][0] = __ldg(wrow[b] + 2 * (c0 + 32 * d));
        wv[d][b][1] = __ldg(wrow[b] + 2 * (c0 + 32 * d) + 1);
      }
    }
#pragma unroll
  for (int d = 0; d < DEPTH; ++d) {
    const int c = c0 + 32 * d;
    if (!MASKED || c < nch) {
#pragma unroll
      for (int p = 0; p < TT / 2; ++p) {
        const uint4 ha = h_s[(2 * p) * nch + c], hb = h_s[(2 * p + 1) * nch + c];
        const uint32_t wa[4] = {ha.x, ha.y, ha.z, ha.w}, wb[4] = {hb.x, hb.y, hb.z, hb.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // elements 2j and 2j+1 of both tokens' chunk (bf16 -> fp32 is exact)
          const float2 h0 = make_float2(__uint_as_float(wa[j] << 16), __uint_as_float(wb[j] << 16));
          const float2 h1 = make_float2(__uint_as_float(wa[j] & 0xFFFF0000u), __uint_as_float(wb[j] & 0xFFFF0000u));
#pragma unroll
          for (int b = 0; b < TE; ++b) {
            const float w[8] = {wv[d][b][0].x, wv[d][b][0].y, wv[d][b][0].z, wv[d][b][0].w,
                                wv[d][b][1].x, wv[d][b][1].y, wv[d][b][1].z, wv[d][b][1].w};
            acc[p][b] = __ffma2_rn(h0, make_float2(w[2 * j], w[2 * j]), acc[p][b]);
            acc[p][b] = __ffma2_rn(h1, make_float2(w[2 * j + 1], w[2 * j + 1]), acc[p][b]);
          }
        }
      }
    }
  }
}

// Tokens [t0, t0+TT) x experts [e0, e0+experts_per_cta): RMSNorm of the
// tokens into h_s (TT*H bf16 of shared memory; also to h_out when write_h),
// then the fp32 logits.  Each warp computes TE experts x TT tokens at a time.
// The CTA's kRouteWarps*32 threads call it together (it synchronises them).
// Both phases are bound by memory latency at small T, so a lane issues the
// loads of a whole pass (up to kRegChunks chunks of x and g, DEPTH chunks of
// router weights per expert) before it uses any of them.  DEEP = false halves
// both depths, for callers that need the registers for other work.  PAIRED
// (TT even): the logits loop takes tokens two at a time (gemv_round_paired),
// one chunk of router weights per round.
template <int TT, int TE, bool DEEP = true, bool PAIRED = false>
__device__ __forceinline__ void norm_router_tile(const uint16_t* __restrict__ x, const uint16_t* __restrict__ g,
                                                 const float* __restrict__ w_router, const float* __restrict__ bias,
                                                 int T, int H, int E, float eps, int t0, int e0, int experts_per_cta,
                                                 bool write_h, uint16_t* __restrict__ h_out,
                                                 float* __restrict__ logits, uint4* h_s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = H >> 3;
  // ---- RMSNorm: one warp per token
  constexpr int kRegChunks = (TT >= 8 || !DEEP) ? 8 : 16;  // per lane: rows up to 256 * kRegChunks elements in registers
  for (int tt = warp; tt < TT; tt += kRouteWarps) {
    const int t = t0 + tt;
    if (t >= T) break;
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    const uint4* gr = reinterpret_cast<const uint4*>(g);
    uint4* hrow = reinterpret_cast<uint4*>(h_out + static_cast<size_t>(t) * H);
    if (TT < 8 && nch <= 32 * kRegChunks) {
      // the whole row: x and g loads all in flight, one pass
      uint4 xv[kRegChunks], gv[kRegChunks];
#pragma unroll
      for (int d = 0; d < kRegChunks; ++d) {
        const int c = lane + 32 * d;
        if (c < nch) {
          xv[d] = __ldg(xr + c);
          gv[d] = __ldg(gr + c);
        }
      }
      float ss = 0.0f;
#pragma unroll
      for (int d = 0; d < kRegChunks; ++d) {
        if (lane + 32 * d < nch) {
          float f[8];
          unpack8(xv[d], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) ss = __fmaf_rn(f[i], f[i], ss);
        }
      }
      const float rstd = rms_rstd(ss, H, eps);
#pragma unroll
      for (int d = 0; d < kRegChunks; ++d) {
        const int c = lane + 32 * d;
        if (c < nch) {
          const uint4 o = norm_chunk(xv[d], gv[d], rstd);
          h_s[tt * nch + c] = o;
          if (write_h) hrow[c] = o;
        }
      }
    } else {
      // longer rows: 8 chunks' loads in flight, then their FMAs in chunk order;
      // a second pass for h
      float ss = 0.0f;
      int c = lane;
      for (; c + 32 * 7 < nch; c += 32 * 8) {
        uint4 v[8];
#pragma unroll
        for (int d = 0; d < 8; ++d) v[d] = __ldg(xr + c + 32 * d);
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          float f[8];
          unpack8(v[d], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) ss = __fmaf_rn(f[i], f[i], ss);
        }
      }
      for (; c < nch; c += 32) {
        float f[8];
        unpack8(__ldg(xr + c), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = __fmaf_rn(f[i], f[i], ss);
      }
      const float rstd = rms_rstd(ss, H, eps);
#pragma unroll 4
      for (int c2 = lane; c2 < nch; c2 += 32) {
        const uint4 o = norm_chunk(__ldg(xr + c2), __ldg(gr + c2), rstd);
        h_s[tt * nch + c2] = o;
        if (write_h) hrow[c2] = o;
      }
    }
  }
  __syncthreads();

  // ---- logits: warp w takes expert groups e0 + (w + 8 r) * TE .. + TE
  const int e_end = min(E, e0 + experts_per_cta);
  const int ntok = min(TT, T - t0);
  // DEPTH chunks of router weights in flight per lane (32 B each per expert),
  // consumed in chunk order, so every accumulator keeps the canonical sequence
  constexpr int DEPTH = ((TE >= 4) ? 2 : (TE == 2 ? 8 : 16)) / (DEEP || TE >= 4 ? 1 : 2);
  if constexpr (PAIRED) {
    static_assert(TT % 2 == 0, "tokens are paired");
    for (int eg = e0 + warp * TE; eg < e_end; eg += kRouteWarps * TE) {
      float2 acc[TT / 2][TE];
#pragma unroll
      for (int p = 0; p < TT / 2; ++p)
#pragma unroll
        for (int b = 0; b < TE; ++b) acc[p][b] = make_float2(0.0f, 0.0f);
      const float4* wrow[TE];
#pragma unroll
      for (int b = 0; b < TE; ++b)
        wrow[b] = reinterpret_cast<const float4*>(w_router + static_cast<size_t>(min(eg + b, E - 1)) * H);
      for (int c0 = lane; c0 < nch; c0 += 32) gemv_round_paired<TT, TE, 1, false>(wrow, h_s, nch, c0, acc);
#pragma unroll
      for (int p = 0; p < TT / 2; ++p)
#pragma unroll
        for (int b = 0; b < TE; ++b) {
          float v0 = warp_butterfly_sum(acc[p][b].x);
          float v1 = warp_butterfly_sum(acc[p][b].y);
          const int e = eg + b;
          if (lane == 0 && e < e_end) {
            if (bias) {
              v0 = __fadd_rn(v0, bias[e]);
              v1 = __fadd_rn(v1, bias[e]);
            }
            if (2 * p < ntok) logits[static_cast<size_t>(t0 + 2 * p) * E + e] = v0;
            if (2 * p + 1 < ntok) logits[static_cast<size_t>(t0 + 2 * p + 1) * E + e] = v1;
          }
        }
    }
    return;
  }
  for (int eg = e0 + warp * TE; eg < e_end; eg += kRouteWarps * TE) {
    float acc[TT][TE];
#pragma unroll
    for (int a = 0; a < TT; ++a)
#pragma unroll
      for (int b = 0; b < TE; ++b) acc[a][b] = 0.0f;
    const float4* wrow[TE];
#pragma unroll
    for (int b = 0; b < TE; ++b) {
      const int e = min(eg + b, E - 1);  // clamp: a tail expert's duplicate is computed but not stored
      wrow[b] = reinterpret_cast<const float4*>(w_router + static_cast<size_t>(e) * H);
    }
    // full rounds of DEPTH chunks, then one round with the chunks past the row masked off
    int c0 = lane;
    for (; c0 + 32 * (DEPTH - 1) < nch; c0 += 32 * DEPTH) gemv_round<TT, TE, DEPTH, false>(wrow, h_s, nch, c0, acc);
    if constexpr (DEPTH > 2) {
      if (c0 < nch) gemv_round<TT, TE, DEPTH, true>(wrow, h_s, nch, c0, acc);
    } else {
      for (; c0 < nch; c0 += 32) gemv_round<TT, TE, 1, false>(wrow, h_s, nch, c0, acc);
    }
#pragma unroll
    for (int a = 0; a < TT; ++a)
#pragma unroll
      for (int b = 0; b < TE; ++b) {
        float v = warp_butterfly_sum(acc[a][b]);
        const int e = eg + b;
        if (lane == 0 && a < ntok && e < e_end) {
          if (bias) v = __fadd_rn(v, bias[e]);
          logits[static_cast<size_t>(t0 + a) * E + e] = v;
        }
      }
  }
}

}  // namespace rt
}  // namespace moe
