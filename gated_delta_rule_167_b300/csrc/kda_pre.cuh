// The input side of a KDA layer: the inputs of the recurrence from the raw projections.
//
// Kimi K3 wiki, "Notations mathématiques", table "Fonctions": ShortConv is a causal convolution
// with a kernel of size 4, L2Norm(x) = x / ||x||_2, Sigmoid(x) = 1 / (1 + e^-x); table
// "Attention et KDA": q, k are L2-normalised, A_h is a learned per-head log scale, b_alpha^h a
// per-head decay bias and z_t the decay logit; "Glossaire", entry "Décroissance bornée":
// g = g_min sigma(e^A z) with g_min = -5; "Tableau des spécifications": ShortConv kernel 4.
//   q = L2Norm(ShortConv(q~)), k = L2Norm(ShortConv(k~)), v = ShortConv(v~),
//   g = g_min sigma(e^{A_h} z + b_alpha^h),
// ShortConv depthwise (one 4-tap filter per channel; the weights are tap-major, w[h, j, c] on the
// token j steps back), with zeros before the first token of each sequence.
//
// This file holds the pieces shared with the fused path of the tensor-core prefill and a
// standalone kernel for every shape: d / 8 threads per (token, head) row, 8 channels and 4
// consecutive tokens per thread; the norm's sum of squares is reduced over the lanes of the row.
#pragma once

#include "kda_common.cuh"
#include "kda_post.cuh"

namespace kda {
namespace pre {

constexpr float G_MIN = -5.0f;

// g = g_min * sigma(s), s = e^A z + b: to fp32 accuracy for fp32 outputs, with the hardware tanh
// form of the sigmoid for bf16 outputs.
template <typename TIn = __nv_bfloat16>
__device__ __forceinline__ float decay_gate(float z, float eA, float b) {
  return G_MIN * post::sigmoid_for<TIn>(fmaf(eA, z, b));
}

// Raw row pointers of the standalone kernel.
struct PreParams {
  const void *q_raw, *k_raw, *v_raw, *z;
  const float *conv_q, *conv_k, *conv_v;  // [H, 4, d], tap-major
  const float *A_log, *b_decay;           // [H], [H, d]
  void *q, *k, *v, *g;                    // outputs, [rows, H, d]
  const int32_t* cu_seqlens;              // null: dense, sequences of T tokens
  int n_seq, H, T;                        // dense: B; packed: N and T_total
};

// Position of token `tok` (an index along the token axis) inside its sequence.
__device__ __forceinline__ int position_in_sequence(const PreParams& P, long long tok) {
  if (P.cu_seqlens == nullptr) return (int)(tok % P.T);
  int lo = 0, hi = P.n_seq;  // largest s with cu[s] <= tok
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (P.cu_seqlens[mid] <= tok) lo = mid; else hi = mid;
  }
  return (int)(tok - P.cu_seqlens[lo]);
}

template <typename TIn>
__device__ __forceinline__ void load8(const TIn* p, float (&x)[8]) {
  if constexpr (sizeof(TIn) == 2) {
    post::unpack8(*reinterpret_cast<const uint4*>(p), x);
  } else {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

template <typename TIn>
__device__ __forceinline__ void store8(TIn* p, const float (&x)[8]) {
  if constexpr (sizeof(TIn) == 2) {
    *reinterpret_cast<uint4*>(p) = post::pack8(x);
  } else {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
}

// The four taps of 8 channels [c0, c0 + 8) of head h: w[j][e] multiplies the token j steps back
// (tap-major weights: the 16 lanes of a row read one contiguous 512-byte span per tap).
template <int D>
__device__ __forceinline__ void load_taps(const float* w, int h, int c0, float (&t)[4][8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4* p = reinterpret_cast<const float4*>(w + ((size_t)h * 4 + j) * D + c0);
    const float4 a = p[0], b = p[1];
    t[j][0] = a.x; t[j][1] = a.y; t[j][2] = a.z; t[j][3] = a.w;
    t[j][4] = b.x; t[j][5] = b.y; t[j][6] = b.z; t[j][7] = b.w;
  }
}

// Four consecutive outputs of the causal convolution, one 8-channel chunk: x[m] holds input row
// m - 3 relative to the first output (x[0..2] the three rows before it); output i takes tap j
// (from x[i + 3 - j]) only when j <= pos[i], its position in its sequence, so that nothing
// reaches across a sequence start.
__device__ __forceinline__ void conv4x8(const float (&t)[4][8], const float (&x)[7][8],
                                        const int (&pos)[4], float (&y)[4][8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j <= pos[i]) a = fmaf(t[j][e], x[i + 3 - j][e], a);
      y[i][e] = a;
    }
}

// Sum over the lanes of one row: 16 lanes for d = 128, 8 for d = 64.
template <int D>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int o = D / 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D, bool kExact = true>
__device__ __forceinline__ void l2norm8(float (&x)[8]) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
  ss = row_sum<D>(ss);
  const float inv = ss > 0.f ? (kExact ? 1.f / sqrtf(ss) : rsqrtf(ss)) : 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] *= inv;
}

// Standalone kernel: one CTA per (head, tile of 4 * 256 / (D / 8) tokens, output tensor), heads
// fastest, so that the CTAs resident at one time read neighbouring heads of the same tokens
// (contiguous memory); blockIdx.z picks q, k, v (convolution, and the norm for q and k) or g
// (the decay gate), so that a thread holds one tensor's rows and many CTAs fit on an SM. D / 8
// threads per token row, 8 channels and 4 consecutive tokens per thread: each thread reads the
// 7 rows it needs once (the rows shared with neighbouring threads hit L1). With bf16 inputs
// three CTAs share an SM (registers capped at 85, a few spills): more loads in flight per SM.
template <typename TIn, int D>
__global__ void __launch_bounds__(256, sizeof(TIn) == 2 ? 3 : 2) pre_core_kernel(PreParams P, long long n_tok) {
  constexpr int TPR = D / 8;            // threads per token row
  constexpr int TOK = 4 * (256 / TPR);  // tokens per CTA
  const int h = blockIdx.x;
  const int ts = blockIdx.z;  // 0 q, 1 k, 2 v, 3 g
  const int cg = threadIdx.x % TPR, rg = threadIdx.x / TPR;
  const int c0 = 8 * cg;
  const int H = P.H;
  const long long n_tiles = (n_tok + TOK - 1) / TOK;
  for (long long tile = blockIdx.y; tile < n_tiles; tile += gridDim.y) {
    const long long tok0 = tile * TOK + 4 * rg;  // first of this thread's tokens
    bool live[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) live[i] = tok0 + i < n_tok;
    if (ts == 3) {  // the decay gate
      const float eA = expf(P.A_log[h]);
      float b8[8];
      {
        const float4* bp = reinterpret_cast<const float4*>(P.b_decay + (size_t)h * D + c0);
        const float4 a = bp[0], b = bp[1];
        b8[0] = a.x; b8[1] = a.y; b8[2] = a.z; b8[3] = a.w; b8[4] = b.x; b8[5] = b.y; b8[6] = b.z; b8[7] = b.w;
      }
      float z[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (live[i]) load8(static_cast<const TIn*>(P.z) + ((size_t)(tok0 + i) * H + h) * D + c0, z[i]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (!live[i]) continue;
#pragma unroll
        for (int e = 0; e < 8; ++e) z[i][e] = decay_gate<TIn>(z[i][e], eA, b8[e]);
        store8(static_cast<TIn*>(P.g) + ((size_t)(tok0 + i) * H + h) * D + c0, z[i]);
      }
      continue;
    }
    int pos[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pos[i] = live[i] ? position_in_sequence(P, tok0 + i) : 0;
    const TIn* src = static_cast<const TIn*>(ts == 0 ? P.q_raw : (ts == 1 ? P.k_raw : P.v_raw));
    const float* w = ts == 0 ? P.conv_q : (ts == 1 ? P.conv_k : P.conv_v);
    TIn* dst = static_cast<TIn*>(ts == 0 ? P.q : (ts == 1 ? P.k : P.v));
    float t[4][8], y[4][8];
    if constexpr (sizeof(TIn) == 2) {  // rows kept packed (bf16 pairs) until used
      uint4 xr[7];
#pragma unroll
      for (int m = 0; m < 7; ++m) {  // every load is issued before any arithmetic
        const long long r = tok0 + m - 3;
        xr[m] = (r >= 0 && r < n_tok)
                    ? *reinterpret_cast<const uint4*>(src + ((size_t)r * H + h) * D + c0)
                    : make_uint4(0, 0, 0, 0);
      }
      load_taps<D>(w, h, c0, t);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float xe[7];
#pragma unroll
        for (int m = 0; m < 7; ++m) {
          const uint32_t wd = e < 2 ? xr[m].x : (e < 4 ? xr[m].y : (e < 6 ? xr[m].z : xr[m].w));
          xe[m] = __uint_as_float((e & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j <= pos[i]) a = fmaf(t[j][e], xe[i + 3 - j], a);
          y[i][e] = a;
        }
      }
    } else {
      float x[7][8];
#pragma unroll
      for (int m = 0; m < 7; ++m) {  // every load is issued before any arithmetic
        const long long r = tok0 + m - 3;
        if (r >= 0 && r < n_tok) {
          load8(src + ((size_t)r * H + h) * D + c0, x[m]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[m][e] = 0.f;
        }
      }
      load_taps<D>(w, h, c0, t);
      conv4x8(t, x, pos, y);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (ts < 2) l2norm8<D, sizeof(TIn) == 4>(y[i]);  // every lane of the row joins
      if (live[i]) store8(dst + ((size_t)(tok0 + i) * H + h) * D + c0, y[i]);
    }
  }  // tiles
}

}  // namespace pre
}  // namespace kda
