// One-token KDA decode step, state resident in HBM and updated in place.
//
// Kimi K3 wiki, "Glossaire", entry "Decode": generation advances one token at a time and is
// bound by memory bandwidth. Per (sequence, head) the step reads and writes the whole fp32
// state (d_k x d_v x 4 bytes each way) and only a few hundred bytes of token inputs, so the
// kernel is a streaming pass over S at HBM speed:
//
//   S' = Diag(alpha) S,  c = S'^T k,  S'' = S' + beta k (v - c)^T,  o = S''^T q
//
// (Notations mathématiques, table "Attention et KDA": M_t, S_t, o_t.) Each column of S is
// independent, so the only cross-thread step is the reduction over the key channel i. The
// read-out folds into the same reduction:
//   o_j = sum_i q_i S''_ij = sum_i (alpha_i q_i) S_ij + (q . k) beta (v_j - c_j),
// so S is read once, reduced once (two dot products per column), updated and written once.
//
// Layout: one CTA per (sequence, head). A warp covers a row slab of DV columns with one
// float4 per lane (128-bit, fully coalesced 512-byte rows); the CTA's row groups split the
// d_k rows. Every thread issues all of its state loads before any arithmetic, so each CTA
// keeps its whole 64 KiB state slice in flight.
#pragma once

#include "kda_common.cuh"

namespace kda {

template <typename TIn, int DK, int DV, int THREADS>
__global__ void __launch_bounds__(THREADS)
    decode_step_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                       const TIn* __restrict__ v, const TIn* __restrict__ g,
                       const TIn* __restrict__ beta, float* __restrict__ S,
                       TIn* __restrict__ out) {
  constexpr int CG = DV / 4;        // float4 column groups per row
  constexpr int RG = THREADS / CG;  // row groups
  constexpr int RPT = DK / RG;      // rows per thread
  static_assert(DV % 4 == 0 && THREADS % CG == 0 && DK % RG == 0, "bad decode tiling");

  __shared__ float s_alpha[DK], s_k[DK], s_ak[DK], s_aq[DK], s_q[DK];
  __shared__ float4 s_redc[RG][CG];
  __shared__ float4 s_redp[RG][CG];
  __shared__ float s_qk;

  const int p = blockIdx.x;  // n * H + h
  const int tid = threadIdx.x;
  const int cg = tid % CG;
  const int rg = tid / CG;

  float4* Sp = reinterpret_cast<float4*>(S + (size_t)p * DK * DV);
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = __ldcs(&Sp[(rg * RPT + i) * CG + cg]);

  for (int i = tid; i < DK; i += THREADS) {
    const float a = expf(to_f32(g[(size_t)p * DK + i]));
    const float kk = to_f32(k[(size_t)p * DK + i]);
    const float qq = to_f32(q[(size_t)p * DK + i]);
    s_alpha[i] = a;
    s_k[i] = kk;
    s_q[i] = qq;
    s_ak[i] = a * kk;
    s_aq[i] = a * qq;
  }
  __syncthreads();

  float4 c = make_float4(0.f, 0.f, 0.f, 0.f), pq = c;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg * RPT + i;
    const float ak = s_ak[r], aq = s_aq[r];
    c.x = fmaf(ak, s[i].x, c.x); c.y = fmaf(ak, s[i].y, c.y);
    c.z = fmaf(ak, s[i].z, c.z); c.w = fmaf(ak, s[i].w, c.w);
    pq.x = fmaf(aq, s[i].x, pq.x); pq.y = fmaf(aq, s[i].y, pq.y);
    pq.z = fmaf(aq, s[i].z, pq.z); pq.w = fmaf(aq, s[i].w, pq.w);
  }
  s_redc[rg][cg] = c;
  s_redp[rg][cg] = pq;
  if (tid < 32) {
    float acc = 0.f;
    for (int i = tid; i < DK; i += 32) acc = fmaf(s_q[i], s_k[i], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (tid == 0) s_qk = acc;
  }
  __syncthreads();

  float4 C = make_float4(0.f, 0.f, 0.f, 0.f), P = C;
#pragma unroll
  for (int r = 0; r < RG; ++r) {
    const float4 a = s_redc[r][cg], b = s_redp[r][cg];
    C.x += a.x; C.y += a.y; C.z += a.z; C.w += a.w;
    P.x += b.x; P.y += b.y; P.z += b.z; P.w += b.w;
  }
  const float bt = to_f32(beta[p]);
  const TIn* vp = v + (size_t)p * DV + 4 * cg;
  float4 d;  // beta (v - c)
  d.x = bt * (to_f32(vp[0]) - C.x);
  d.y = bt * (to_f32(vp[1]) - C.y);
  d.z = bt * (to_f32(vp[2]) - C.z);
  d.w = bt * (to_f32(vp[3]) - C.w);

#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg * RPT + i;
    const float a = s_alpha[r], kk = s_k[r];
    float4 x = s[i];
    x.x = fmaf(kk, d.x, a * x.x);
    x.y = fmaf(kk, d.y, a * x.y);
    x.z = fmaf(kk, d.z, a * x.z);
    x.w = fmaf(kk, d.w, a * x.w);
    __stcs(&Sp[r * CG + cg], x);
  }
  if (rg == 0) {
    const float qk = s_qk;
    TIn* op = out + (size_t)p * DV + 4 * cg;
    op[0] = from_f32<TIn>(fmaf(qk, d.x, P.x));
    op[1] = from_f32<TIn>(fmaf(qk, d.y, P.y));
    op[2] = from_f32<TIn>(fmaf(qk, d.z, P.z));
    op[3] = from_f32<TIn>(fmaf(qk, d.w, P.w));
  }
}

}  // namespace kda

namespace kda {

// K decode tokens per (sequence, head) in one pass over the state: the same step as
// decode_step_kernel applied K times while the CTA's slice of S stays in registers, so S is read
// from and written to HBM once whatever K is (speculative verification of K draft tokens, or
// any short run of tokens). Inputs are [N, K, H, d] (token t of sequence n at (n K + t) H + h);
// out receives o for every token. Per token: the read-out reductions go through shared memory
// (one barrier each), as in the single-step kernel.
template <typename TIn, int DK, int DV, int THREADS>
__global__ void __launch_bounds__(THREADS)
    decode_tokens_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                         const TIn* __restrict__ v, const TIn* __restrict__ g,
                         const TIn* __restrict__ beta, float* __restrict__ S,
                         TIn* __restrict__ out, int K, int H) {
  constexpr int CG = DV / 4;
  constexpr int RG = THREADS / CG;
  constexpr int RPT = DK / RG;
  static_assert(DV % 4 == 0 && THREADS % CG == 0 && DK % RG == 0, "bad decode tiling");

  __shared__ float s_alpha[DK], s_k[DK], s_ak[DK], s_aq[DK], s_q[DK];
  __shared__ float4 s_redc[RG][CG];
  __shared__ float4 s_redp[RG][CG];
  __shared__ float s_qk;

  const int p = blockIdx.x;  // n * H + h
  const int n = p / H, h = p % H;
  const int tid = threadIdx.x;
  const int cg = tid % CG;
  const int rg = tid / CG;

  float4* Sp = reinterpret_cast<float4*>(S + (size_t)p * DK * DV);
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = __ldcs(&Sp[(rg * RPT + i) * CG + cg]);

  for (int t = 0; t < K; ++t) {
    const size_t tok = ((size_t)n * K + t) * H + h;  // token row of (n, t, h)
    if (t > 0) __syncthreads();  // the previous token's shared arrays are no longer read
    for (int i = tid; i < DK; i += THREADS) {
      const float a = expf(to_f32(g[tok * DK + i]));
      const float kk = to_f32(k[tok * DK + i]);
      const float qq = to_f32(q[tok * DK + i]);
      s_alpha[i] = a;
      s_k[i] = kk;
      s_q[i] = qq;
      s_ak[i] = a * kk;
      s_aq[i] = a * qq;
    }
    __syncthreads();
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f), pq = c;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = rg * RPT + i;
      const float ak = s_ak[r], aq = s_aq[r];
      c.x = fmaf(ak, s[i].x, c.x); c.y = fmaf(ak, s[i].y, c.y);
      c.z = fmaf(ak, s[i].z, c.z); c.w = fmaf(ak, s[i].w, c.w);
      pq.x = fmaf(aq, s[i].x, pq.x); pq.y = fmaf(aq, s[i].y, pq.y);
      pq.z = fmaf(aq, s[i].z, pq.z); pq.w = fmaf(aq, s[i].w, pq.w);
    }
    s_redc[rg][cg] = c;
    s_redp[rg][cg] = pq;
    if (tid < 32) {
      float acc = 0.f;
      for (int i = tid; i < DK; i += 32) acc = fmaf(s_q[i], s_k[i], acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (tid == 0) s_qk = acc;
    }
    __syncthreads();
    float4 C = make_float4(0.f, 0.f, 0.f, 0.f), Pq = C;
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      const float4 a = s_redc[r][cg], b = s_redp[r][cg];
      C.x += a.x; C.y += a.y; C.z += a.z; C.w += a.w;
      Pq.x += b.x; Pq.y += b.y; Pq.z += b.z; Pq.w += b.w;
    }
    const float bt = to_f32(beta[tok]);
    const TIn* vp = v + tok * DV + 4 * cg;
    float4 d;  // beta (v - c)
    d.x = bt * (to_f32(vp[0]) - C.x);
    d.y = bt * (to_f32(vp[1]) - C.y);
    d.z = bt * (to_f32(vp[2]) - C.z);
    d.w = bt * (to_f32(vp[3]) - C.w);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = rg * RPT + i;
      const float a = s_alpha[r], kk = s_k[r];
      s[i].x = fmaf(kk, d.x, a * s[i].x);
      s[i].y = fmaf(kk, d.y, a * s[i].y);
      s[i].z = fmaf(kk, d.z, a * s[i].z);
      s[i].w = fmaf(kk, d.w, a * s[i].w);
    }
    if (rg == 0) {
      const float qk = s_qk;
      TIn* op = out + tok * DV + 4 * cg;
      op[0] = from_f32<TIn>(fmaf(qk, d.x, Pq.x));
      op[1] = from_f32<TIn>(fmaf(qk, d.y, Pq.y));
      op[2] = from_f32<TIn>(fmaf(qk, d.z, Pq.z));
      op[3] = from_f32<TIn>(fmaf(qk, d.w, Pq.w));
    }
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) __stcs(&Sp[(rg * RPT + i) * CG + cg], s[i]);
}

}  // namespace kda
