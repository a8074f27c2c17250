// Chunkwise KDA prefill on CUDA cores, fp32 arithmetic throughout.
//
// This is the exact path for fp32 inputs (and for shapes the tensor-core kernel does not take).
// The block algebra is the UT-transform form of the recurrence (Kimi K3 wiki, "Glossaire",
// entries "Chunkwise" and "UT"; the recurrence is in "Notations mathématiques", table
// "Attention et KDA"). For one block of L tokens with incoming state S:
//   Gamma_r = inclusive cumulative sum of g along the block, per key channel
//   A_rj  = beta_r sum_c k_rc k_jc exp(Gamma_rc - Gamma_jc), j < r     (strictly lower)
//   T     = (I + A)^{-1}                                              (forward substitution)
//   W     = T Diag(beta) (K * exp(Gamma)),  U~ = T Diag(beta) V,  U = U~ - W S
//   P_rj  = sum_c q_rc k_jc exp(Gamma_rc - Gamma_jc), j <= r          (Tril keeps the diagonal)
//   O     = (Q * exp(Gamma)) S + P U
//   S'    = Diag(exp(Gamma_L)) S + Khat^T U,  Khat_j = k_j * exp(Gamma_L - Gamma_j)
// Every exp(Gamma_r - Gamma_j) here has a non-positive exponent (j <= r, g <= 0), so it is
// evaluated directly per element and never overflows; exp(Gamma_r) may underflow to 0 only
// when its true value is below 1e-38, where it no longer matters next to O(1) terms.
//
// One CTA owns one (batch, head) or (sequence, head) problem and walks its blocks in order;
// the fp32 state stays in shared memory for the whole sequence. The kernel works in L-token
// sub-blocks (L <= 32 keeps everything in one CTA's shared memory); a caller's C of 64 or 128
// is processed as consecutive L-token blocks, which is the same mathematics (the block form is
// exact for any block size).
#pragma once

#include "kda_common.cuh"

namespace kda {

struct SeqParams {
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* beta;
  const float* S0;
  void* out;                  // null: outputs are not written
  float* S_final;
  const int32_t* cu_seqlens;  // null for a dense batch
  int n_seq;                  // dense: B; packed: N
  int H;
  int T;  // dense: tokens per sequence; packed: T_total
  // Segments of dense sequences (seg_len > 0): problem (s, h) with s = sigma * n_seq + b covers
  // tokens [sigma * seg_len, min((sigma + 1) * seg_len, T)) of sequence b, sigma < n_seg.
  int seg_len;
  int n_seg;
  // Transition launches (n_ident > 0): problems p < n_ident start from the identity with v = 0,
  // so their final state is the product of the segment's M_t (written to M_out); problems
  // p >= n_ident cover the same segments from S0 (or zero) with the real v (final state to
  // S_final).
  int n_ident;
  float* M_out;
  // Nonzero: only the last segment of a sequence writes its final state, at (sequence, head).
  int sf_last_only;
  // Output side (null gate_u: out receives the raw output o~): out receives
  // RMSNorm(o~) * norm_w * sigma(gate_u), gate_u shaped like out, norm_w [d_v] fp32.
  const void* gate_u;
  const float* norm_w;
  float norm_eps;
  // Input side (null conv_q: q, k, v, g are the inputs of the recurrence). Otherwise q, k, v, g
  // hold the raw projections q~, k~, v~ and the decay logit z, and the kernel forms
  // q = L2Norm(ShortConv(q~)), k = L2Norm(ShortConv(k~)), v = ShortConv(v~) and
  // g = g_min sigma(e^{A_h} z + b_h): conv_* [H, d, 4], A_log [H], b_decay [H, d], fp32.
  const float* conv_q;
  const float* conv_k;
  const float* conv_v;
  const float* A_log;
  const float* b_decay;
};

// One (sequence or segment, head) problem of a launch.
struct Problem {
  int h;
  size_t row0;     // first token row in the [rows, H] token grid
  int len;         // tokens
  bool ident;      // initial state I and v = 0; S0 is not read
  int pos0;        // position of the first token inside its sequence (segments start inside)
  long long s0;    // index of the initial state in S0
  float* sf;       // array the final state goes to (S_final or M_out), or null
  long long sf_i;  // index in it
};

// Resolves problem p to its token range and state slots. Returns false (and records the
// error) for inconsistent packed offsets.
__device__ __forceinline__ bool resolve_problem(const SeqParams& P, int p, Problem& pr) {
  int q = p;
  pr.ident = false;
  if (P.n_ident > 0) {
    pr.ident = p < P.n_ident;
    if (!pr.ident) q = p - P.n_ident;
  }
  const int s = q / P.H;
  pr.h = q % P.H;
  pr.s0 = q;
  pr.sf = pr.ident ? P.M_out : P.S_final;
  pr.sf_i = q;
  pr.pos0 = 0;
  if (P.seg_len > 0) {
    const int b = s % P.n_seq, sigma = s / P.n_seq;
    const long long a = (long long)sigma * P.seg_len;
    pr.row0 = (size_t)b * P.T + (size_t)a;
    pr.len = (int)max(0ll, min((long long)P.seg_len, (long long)P.T - a));
    pr.pos0 = (int)a;
    if (P.sf_last_only) {
      pr.sf = sigma == P.n_seg - 1 ? P.S_final : nullptr;
      pr.sf_i = (long long)b * P.H + pr.h;
    }
    return true;
  }
  if (P.cu_seqlens == nullptr) {
    pr.row0 = (size_t)s * P.T;
    pr.len = P.T;
    return true;
  }
  const int a = P.cu_seqlens[s], b = P.cu_seqlens[s + 1];
  const int first = P.cu_seqlens[0], last = P.cu_seqlens[P.n_seq];
  if (first != 0 || last != P.T || a < 0 || b < a || b > P.T) {
    record_status(1u /* KDA_ERR_INVALID_ARG */);
    return false;
  }
  pr.row0 = (size_t)a;
  pr.len = b - a;
  return true;
}

template <int DK, int DV, int L>
struct SimtSmem {
  static constexpr int KP = DK + 1;  // padded row stride of the key-side tiles
  static constexpr int LP = L + 1;
  static constexpr size_t floats =
      (size_t)DK * DV + 3 * (size_t)L * KP + (size_t)L * DV + 3 * (size_t)L * LP +
      (size_t)L * DK + (size_t)L * DV + L;
  static constexpr size_t bytes = floats * sizeof(float);
};

template <typename TIn, int DK, int DV, int L, int THREADS>
__global__ void __launch_bounds__(THREADS) chunk_simt_kernel(SeqParams P) {
  using SM = SimtSmem<DK, DV, L>;
  constexpr int KP = SM::KP, LP = SM::LP;
  extern __shared__ float smem[];
  float* S = smem;            // [DK][DV] running state
  float* Kc = S + DK * DV;    // [L][KP]  k, later Khat
  float* Qc = Kc + L * KP;    // [L][KP]  q, later q * exp(Gamma)
  float* Gc = Qc + L * KP;    // [L][KP]  g, then Gamma
  float* Vc = Gc + L * KP;    // [L][DV]  v, then U~
  float* Am = Vc + L * DV;    // [L][LP]  A
  float* Pm = Am + L * LP;    // [L][LP]  P
  float* Tm = Pm + L * LP;    // [L][LP]  T = (I + A)^-1
  float* Wm = Tm + L * LP;    // [L][DK]  beta K exp(Gamma), then W
  float* Um = Wm + L * DK;    // [L][DV]  U
  float* bt = Um + L * DV;    // [L]      beta

  const TIn* __restrict__ q = static_cast<const TIn*>(P.q);
  const TIn* __restrict__ k = static_cast<const TIn*>(P.k);
  const TIn* __restrict__ v = static_cast<const TIn*>(P.v);
  const TIn* __restrict__ g = static_cast<const TIn*>(P.g);
  const TIn* __restrict__ beta = static_cast<const TIn*>(P.beta);
  TIn* __restrict__ out = static_cast<TIn*>(P.out);

  const int p = blockIdx.x;
  const int tid = threadIdx.x;
  Problem pr;
  if (!resolve_problem(P, p, pr)) return;
  const int H = P.H, h = pr.h, len = pr.len;
  const size_t row0 = pr.row0;

  for (int i = tid; i < DK * DV; i += THREADS) {
    if (pr.ident)
      S[i] = (i / DV == i % DV) ? 1.f : 0.f;
    else
      S[i] = P.S0 ? P.S0[(size_t)pr.s0 * DK * DV + i] : 0.f;
  }

  for (int t0 = 0; t0 < len; t0 += L) {
    const int n = min(L, len - t0);
    __syncthreads();  // previous block's users of the tiles are done
    // ---- stage the block; rows past the end are zero (g = 0 keeps Gamma flat there)
    for (int i = tid; i < L * DK; i += THREADS) {
      const int r = i / DK, c = i % DK;
      float kk = 0.f, qq = 0.f, gg = 0.f;
      if (r < n) {
        const size_t e = ((row0 + t0 + r) * H + h) * DK + c;
        kk = to_f32(k[e]);
        qq = to_f32(q[e]);
        gg = to_f32(g[e]);
      }
      Kc[r * KP + c] = kk;
      Qc[r * KP + c] = qq;
      Gc[r * KP + c] = gg;
    }
    for (int i = tid; i < L * DV; i += THREADS) {
      const int r = i / DV, c = i % DV;
      Vc[r * DV + c] = (r < n && !pr.ident) ? to_f32(v[((row0 + t0 + r) * H + h) * DV + c]) : 0.f;
    }
    for (int r = tid; r < L; r += THREADS) bt[r] = r < n ? to_f32(beta[(row0 + t0 + r) * H + h]) : 0.f;
    __syncthreads();
    // ---- Gamma: inclusive cumulative sum along the block
    for (int c = tid; c < DK; c += THREADS) {
      float acc = 0.f;
      for (int r = 0; r < L; ++r) {
        acc += Gc[r * KP + c];
        Gc[r * KP + c] = acc;
      }
    }
    __syncthreads();
    // ---- A (strictly lower, scaled by beta_r) and P (lower incl. diagonal)
    for (int i = tid; i < L * L; i += THREADS) {
      const int r = i / L, j = i % L;
      float a = 0.f, pq = 0.f;
      if (j <= r) {
        const float* kr = Kc + r * KP;
        const float* qr = Qc + r * KP;
        const float* kj = Kc + j * KP;
        const float* gr = Gc + r * KP;
        const float* gj = Gc + j * KP;
        for (int c = 0; c < DK; ++c) {
          const float kd = kj[c] * expf(gr[c] - gj[c]);
          a = fmaf(kr[c], kd, a);
          pq = fmaf(qr[c], kd, pq);
        }
      }
      Am[r * LP + j] = (j < r) ? bt[r] * a : 0.f;
      Pm[r * LP + j] = pq;
    }
    __syncthreads();
    // ---- T = (I + A)^-1: each thread owns one column and substitutes down the rows
    if (tid < L) {
      const int j = tid;
      float col[L];
#pragma unroll
      for (int r = 0; r < L; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) acc = fmaf(Am[r * LP + i], col[i], acc);
        col[r] = (r == j) ? 1.f : (r > j ? -acc : 0.f);
      }
#pragma unroll
      for (int r = 0; r < L; ++r) Tm[r * LP + j] = col[r];
    }
    // beta K exp(Gamma) (operand of W); Q exp(Gamma) for the state read-out
    for (int i = tid; i < L * DK; i += THREADS) {
      const int r = i / DK, c = i % DK;
      const float e = expf(Gc[r * KP + c]);
      Wm[r * DK + c] = bt[r] * Kc[r * KP + c] * e;
    }
    __syncthreads();
    // ---- W = T (beta K exp Gamma) in place (rows bottom-up); U~ = T (beta V) in place
    for (int c = tid; c < DK + DV; c += THREADS) {
      float* col = c < DK ? Wm + c : Vc + (c - DK);
      const int ld = c < DK ? DK : DV;
      const bool scale_beta = c >= DK;
      for (int r = L - 1; r >= 0; --r) {
        float acc = 0.f;
        for (int j = 0; j <= r; ++j) {
          const float x = scale_beta ? bt[j] * col[j * ld] : col[j * ld];
          acc = fmaf(Tm[r * LP + j], x, acc);
        }
        col[r * ld] = acc;
      }
    }
    __syncthreads();
    // ---- U = U~ - W S
    for (int i = tid; i < L * DV; i += THREADS) {
      const int r = i / DV, c = i % DV;
      float acc = Vc[r * DV + c];
      const float* w = Wm + r * DK;
      for (int kk = 0; kk < DK; ++kk) acc = fmaf(-w[kk], S[kk * DV + c], acc);
      Um[r * DV + c] = acc;
    }
    // q exp(Gamma) in place (A and P are done with q)
    for (int i = tid; i < L * DK; i += THREADS) {
      const int r = i / DK, c = i % DK;
      Qc[r * KP + c] *= expf(Gc[r * KP + c]);
    }
    __syncthreads();
    // ---- O = (Q exp Gamma) S + P U, written straight out
    for (int i = tid; out != nullptr && i < n * DV; i += THREADS) {
      const int r = i / DV, c = i % DV;
      float acc = 0.f;
      const float* qr = Qc + r * KP;
      for (int kk = 0; kk < DK; ++kk) acc = fmaf(qr[kk], S[kk * DV + c], acc);
      for (int j = 0; j <= r; ++j) acc = fmaf(Pm[r * LP + j], Um[j * DV + c], acc);
      out[((row0 + t0 + r) * H + h) * DV + c] = from_f32<TIn>(acc);
    }
    // Khat = K exp(Gamma_L - Gamma) in place (W was formed from its own copy)
    for (int i = tid; i < L * DK; i += THREADS) {
      const int r = i / DK, c = i % DK;
      Kc[r * KP + c] *= expf(Gc[(L - 1) * KP + c] - Gc[r * KP + c]);
    }
    __syncthreads();
    // ---- S' = Diag(exp Gamma_L) S + Khat^T U
    for (int i = tid; i < DK * DV; i += THREADS) {
      const int r = i / DV, c = i % DV;
      float acc = expf(Gc[(L - 1) * KP + r]) * S[i];
      for (int j = 0; j < L; ++j) acc = fmaf(Kc[j * KP + r], Um[j * DV + c], acc);
      S[i] = acc;
    }
  }
  __syncthreads();
  if (pr.sf)
    for (int i = tid; i < DK * DV; i += THREADS) pr.sf[(size_t)pr.sf_i * DK * DV + i] = S[i];
}

}  // namespace kda
