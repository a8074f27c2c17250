// The output side of a KDA layer: y = RMSNorm(o~) (*) sigma(u).
//
// Kimi K3 wiki, "Notations mathématiques": o~_t is the raw output of the recurrence, before the
// gate; table "Fonctions": RMSNorm(x) = x / sqrt(mean_i x_i^2 + eps) (*) w and
// Sigmoid(x) = 1 / (1 + e^-x). Chapter 03: RMSNorm is applied to KDA's recurrent output;
// "Tableau des spécifications": RMSNorm epsilon 1e-5, and a full-rank KDA output gate, whose
// pre-activation u (one value per output channel) is an input here. The norm runs over the d_v
// channels of each (token, head); w has d_v entries shared by the heads.
//
// The tensor-core prefill applies this in its output epilogue (kda_chunk_tc.cuh); this file holds
// the pieces it shares with the standalone kernel below, which serves the other paths (the
// CUDA-core prefill, decode outputs): one pass over [rows, H, d_v], 16 threads per (token, head)
// with 8 channels each (16-byte accesses for bf16), the sum of squares reduced over the 16 lanes.
#pragma once

#include "kda_common.cuh"

namespace kda {
namespace post {

// sigma(x) = (1 + tanh(x / 2)) / 2 with the hardware tanh approximation (PTX tanh.approx.f32,
// relative error about 2^-11), for bf16 outputs.
__device__ __forceinline__ float sigmoid_fast(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
  return fmaf(0.5f, t, 0.5f);
}

// sigma(x) to fp32 accuracy, for fp32 outputs.
__device__ __forceinline__ float sigmoid_exact(float x) { return 1.f / (1.f + expf(-x)); }

template <typename TIn>
__device__ __forceinline__ float sigmoid_for(float x) {
  if constexpr (sizeof(TIn) == 2) return sigmoid_fast(x);
  else return sigmoid_exact(x);
}

// Sum over the 16 lanes of each half-warp (lanes 0-15 and 16-31 reduce separately).
__device__ __forceinline__ float sum16(float x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ void unpack8(const uint4& r, float (&x)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The 8 weights of one chunk (16-byte aligned: w is, and chunks start at multiples of 8)
__device__ __forceinline__ void load_w8(const float* p, float (&w)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// y = o / sqrt(mean(o^2) + eps) * w * sigma(u) for one 8-channel chunk of a 128-channel row held
// by 16 lanes; `valid` rows take part in the reduction either way (their lanes are in the same
// half-warp) but their values are only used when valid.
template <typename TIn = __nv_bfloat16>
__device__ __forceinline__ void gate_chunk(float (&x)[8], const float (&u)[8], const float (&w)[8],
                                           float eps, int d) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
  ss = sum16(ss);
  // bf16 outputs: the hardware reciprocal square root (about 2 ulp of fp32, far below the
  // output's rounding) instead of a correctly rounded square root and division
  const float ms = ss / (float)d + eps;
  const float inv = sizeof(TIn) == 2 ? rsqrtf(ms) : 1.f / sqrtf(ms);
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = x[e] * inv * w[e] * sigmoid_for<TIn>(u[e]);
}

// Standalone kernel: 256 threads = 16 rows of (token, head) per CTA, 16 threads x 8 channels per
// row (d_v = 128). bf16 or fp32 tensors; y may alias o.
template <typename TIn>
__global__ void __launch_bounds__(256)
    output_gate_kernel(const TIn* o, const TIn* __restrict__ u, const float* __restrict__ w,
                       float eps, TIn* y, long long n_rows) {
  const long long row = (long long)blockIdx.x * 16 + (threadIdx.x >> 4);
  const int q = threadIdx.x & 15;
  const bool valid = row < n_rows;
  const size_t base = (size_t)(valid ? row : 0) * 128 + 8 * q;
  float x[8], uu[8], ww[8];
  load_w8(w + 8 * q, ww);
  if constexpr (sizeof(TIn) == 2) {
    uint4 ro = make_uint4(0, 0, 0, 0), ru = ro;
    if (valid) {
      ro = *reinterpret_cast<const uint4*>(o + base);
      ru = *reinterpret_cast<const uint4*>(u + base);
    }
    unpack8(ro, x);
    unpack8(ru, uu);
  } else {
#pragma unroll
    for (int e = 0; e < 8; e += 4) {
      float4 a = valid ? *reinterpret_cast<const float4*>(o + base + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      float4 b = valid ? *reinterpret_cast<const float4*>(u + base + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      x[e] = a.x; x[e + 1] = a.y; x[e + 2] = a.z; x[e + 3] = a.w;
      uu[e] = b.x; uu[e + 1] = b.y; uu[e + 2] = b.z; uu[e + 3] = b.w;
    }
  }
  gate_chunk<TIn>(x, uu, ww, eps, 128);
  if (!valid) return;
  if constexpr (sizeof(TIn) == 2) {
    *reinterpret_cast<uint4*>(y + base) = pack8(x);
  } else {
#pragma unroll
    for (int e = 0; e < 8; e += 4)
      *reinterpret_cast<float4*>(y + base + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
  }
}

// d_v = 64: 8 threads x 8 channels per row, 32 rows per CTA. The 8-lane reduction runs inside
// each group of 8 lanes.
template <typename TIn>
__global__ void __launch_bounds__(256)
    output_gate64_kernel(const TIn* o, const TIn* __restrict__ u, const float* __restrict__ w,
                         float eps, TIn* y, long long n_rows) {
  const long long row = (long long)blockIdx.x * 32 + (threadIdx.x >> 3);
  const int q = threadIdx.x & 7;
  const bool valid = row < n_rows;
  const size_t base = (size_t)(valid ? row : 0) * 64 + 8 * q;
  float x[8], uu[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[e] = valid ? to_f32(o[base + e]) : 0.f;
    uu[e] = valid ? to_f32(u[base + e]) : 0.f;
  }
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float ms = ss / 64.f + eps;
  const float inv = sizeof(TIn) == 2 ? rsqrtf(ms) : 1.f / sqrtf(ms);  // as gate_chunk
  if (!valid) return;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    y[base + e] = from_f32<TIn>(x[e] * inv * w[8 * q + e] * sigmoid_for<TIn>(uu[e]));
}

}  // namespace post
}  // namespace kda
