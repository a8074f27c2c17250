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
#include "kda_sm100.cuh"

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
// out receives o for every token. The inputs of up to KB tokens are staged in shared memory in
// one go (their loads overlap the state loads instead of following each token), with the q . k
// products of the staged tokens. The value columns are independent (the reductions run over the
// key channel), so each warp owns 16 value columns over all DK rows: lane = row group rg (8) x
// column group (4), rows rg RPT .. rg RPT + RPT - 1 of lane rg (the row slabs of
// decode_step_kernel; the staged rows, with alpha k and alpha q formed once per token and
// channel, are read as float4 and padded by four words per slab, so that the eight row groups'
// reads fall in distinct banks). The two column sums of a token are xor-shuffles inside
// the warp (the row groups' partial sums added pairwise, where decode_step_kernel adds them in
// sequence: the two agree to fp32 rounding, not bit for bit), and tokens take no barrier of the
// CTA. CTAs of 128 threads (64 columns, 32 KiB of state) keep four in flight per SM.
template <typename TIn, int DK, int DV, int THREADS>
__global__ void __launch_bounds__(THREADS, 512 / THREADS)
    decode_tokens_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                         const TIn* __restrict__ v, const TIn* __restrict__ g,
                         const TIn* __restrict__ beta, float* __restrict__ S,
                         TIn* __restrict__ out, int K, int H) {
  constexpr int WARPS = THREADS / 32;
  constexpr int DVC = 16 * WARPS;   // value columns per CTA
  constexpr int NSPLIT = DV / DVC;  // CTAs per (sequence, head)
  constexpr int RPT = DK / 8;       // rows per lane
  constexpr int KB = 8;             // tokens staged per pass
  constexpr int DKP = DK + 32;      // staged row stride: four pad words after each row slab
  static_assert(THREADS % 32 == 0 && DV % DVC == 0 && DK % 8 == 0 && RPT % 4 == 0,
                "bad decode tiling");

  // per staged token and key channel: alpha, k, q and the products alpha k, alpha q
  __shared__ __align__(16) float s_alpha[KB][DKP], s_k[KB][DKP], s_q[KB][DKP];
  __shared__ __align__(16) float s_ak[KB][DKP], s_aq[KB][DKP];
  __shared__ float4 s_v[KB][DVC / 4];
  __shared__ float s_beta[KB], s_qk[KB];

  const int p = blockIdx.x / NSPLIT;              // n * H + h
  const int c_off = (blockIdx.x % NSPLIT) * DVC;  // first value column of this CTA
  const int n = p / H, h = p % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cgl = lane & 3, rg = lane >> 2;
  const int col4 = c_off / 4 + 4 * warp + cgl;  // this lane's float4 column in a row of S
  auto token_row = [&](int t) { return ((size_t)n * K + t) * H + h; };

  float4* Sp = reinterpret_cast<float4*>(S + (size_t)p * DK * DV);
  constexpr int ROW4 = DV / 4;
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = __ldcs(&Sp[(rg * RPT + i) * ROW4 + col4]);
  // padded position of row r: a lane's slab starts on 16 bytes (read as float4), and the eight
  // slabs of a warp's row groups fall in distinct banks
  auto slot = [](int r) { return r + 4 * (r / RPT); };
  const int slab = slot(rg * RPT);  // this lane's first row

  for (int t0 = 0; t0 < K; t0 += KB) {
    const int kn = min(KB, K - t0);
    if (t0 > 0) __syncthreads();  // the previous pass's staged inputs are no longer read
    for (int e = tid; e < kn * DK; e += THREADS) {
      const int tt = e / DK, i = e % DK;
      const size_t o = token_row(t0 + tt) * DK + i;
      const float a = expf(to_f32(g[o])), kk = to_f32(k[o]), qq = to_f32(q[o]);
      s_alpha[tt][slot(i)] = a;
      s_k[tt][slot(i)] = kk;
      s_q[tt][slot(i)] = qq;
      s_ak[tt][slot(i)] = a * kk;
      s_aq[tt][slot(i)] = a * qq;
    }
    for (int e = tid; e < kn * (DVC / 4); e += THREADS) {
      const int tt = e / (DVC / 4), j = e % (DVC / 4);
      const TIn* vp = v + token_row(t0 + tt) * DV + c_off + 4 * j;
      s_v[tt][j] = make_float4(to_f32(vp[0]), to_f32(vp[1]), to_f32(vp[2]), to_f32(vp[3]));
    }
    if (tid < kn) s_beta[tid] = to_f32(beta[token_row(t0 + tid)]);
    __syncthreads();
    for (int tt = warp; tt < kn; tt += WARPS) {  // q . k, one warp per token
      float acc = 0.f;
      for (int i = lane; i < DK; i += 32) acc = fmaf(s_q[tt][slot(i)], s_k[tt][slot(i)], acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) s_qk[tt] = acc;
    }
    __syncthreads();
    for (int tt = 0; tt < kn; ++tt) {
      // column sums over this lane's rows, on fp32 pairs: c = (alpha k)^T S, pq = (alpha q)^T S
      float2 c01 = make_float2(0.f, 0.f), c23 = c01, p01 = c01, p23 = c01;
#pragma unroll
      for (int i4 = 0; i4 < RPT; i4 += 4) {
        const float4 ak4 = *reinterpret_cast<const float4*>(&s_ak[tt][slab + i4]);
        const float4 aq4 = *reinterpret_cast<const float4*>(&s_aq[tt][slab + i4]);
        const float akv[4] = {ak4.x, ak4.y, ak4.z, ak4.w}, aqv[4] = {aq4.x, aq4.y, aq4.z, aq4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float ak = akv[u], aq = aqv[u];
          const float4 si = s[i4 + u];
          const float2 s01 = make_float2(si.x, si.y), s23 = make_float2(si.z, si.w);
          c01 = sm100::fma2(make_float2(ak, ak), s01, c01);
          c23 = sm100::fma2(make_float2(ak, ak), s23, c23);
          p01 = sm100::fma2(make_float2(aq, aq), s01, p01);
          p23 = sm100::fma2(make_float2(aq, aq), s23, p23);
        }
      }
      // over the eight row groups of the warp (lane bits 2..4), pairwise
      float red[8] = {c01.x, c01.y, c23.x, c23.y, p01.x, p01.y, p23.x, p23.y};
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
#pragma unroll
        for (int j = 0; j < 8; ++j) red[j] += __shfl_xor_sync(0xffffffffu, red[j], off);
      const float bt = s_beta[tt];
      const float4 vv = s_v[tt][4 * warp + cgl];
      // beta (v - c)
      const float2 d01 = make_float2(bt * (vv.x - red[0]), bt * (vv.y - red[1]));
      const float2 d23 = make_float2(bt * (vv.z - red[2]), bt * (vv.w - red[3]));
#pragma unroll
      for (int i4 = 0; i4 < RPT; i4 += 4) {  // S <- Diag(alpha) S + k d^T
        const float4 a4 = *reinterpret_cast<const float4*>(&s_alpha[tt][slab + i4]);
        const float4 k4 = *reinterpret_cast<const float4*>(&s_k[tt][slab + i4]);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float a = av[u], kk = kv[u];
          const int i = i4 + u;
          const float2 x01 = sm100::fma2(make_float2(kk, kk), d01,
                                         sm100::mul2(make_float2(a, a), make_float2(s[i].x, s[i].y)));
          const float2 x23 = sm100::fma2(make_float2(kk, kk), d23,
                                         sm100::mul2(make_float2(a, a), make_float2(s[i].z, s[i].w)));
          s[i] = make_float4(x01.x, x01.y, x23.x, x23.y);
        }
      }
      if (rg == 0) {  // o = S'^T q = pq + (q . k) d
        const float qk = s_qk[tt];
        TIn* op = out + token_row(t0 + tt) * DV + 4 * col4;
        op[0] = from_f32<TIn>(fmaf(qk, d01.x, red[4]));
        op[1] = from_f32<TIn>(fmaf(qk, d01.y, red[5]));
        op[2] = from_f32<TIn>(fmaf(qk, d23.x, red[6]));
        op[3] = from_f32<TIn>(fmaf(qk, d23.y, red[7]));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) __stcs(&Sp[(rg * RPT + i) * ROW4 + col4], s[i]);
}

}  // namespace kda
