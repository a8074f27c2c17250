// Tensor-core chunkwise KDA prefill for bf16 inputs (d_k = d_v = 128, C = 64), sm_103a.
//
// Mathematics (Kimi K3 wiki: "Notations mathématiques", table "Attention et KDA" for the
// recurrence; "Glossaire", entries "Chunkwise", "UT" and "Décroissance bornée"). For one block
// of C tokens, with Gamma the inclusive cumulative sum of g inside the block:
//   A_rj = beta_r sum_c k_rc k_jc e^{Gamma_rc - Gamma_jc} (j < r),  T = (I + A)^{-1}
//   W = T Diag(beta) (K e^Gamma),  U~ = T Diag(beta) V,  U = U~ - W S
//   P_rj = sum_c q_rc k_jc e^{Gamma_rc - Gamma_jc} (j <= r),  O = (Q e^Gamma) S + P U
//   S' = Diag(e^{Gamma_L}) S + Khat^T U,  Khat_j = k_j e^{Gamma_L - Gamma_j}
//
// Bounded decay. Over a block of 64 tokens Gamma can fall to -320, so e^{-Gamma} overflows any
// floating type and A, P cannot be formed as one product (K e^Gamma)(K e^{-Gamma})^T. With
// g >= g_min = -5 every 16-token sub-block spans at most e^80, inside the bf16/fp32 range, so
// A and P are built from four tensor-core products, one per 16-row block R with reference
// B_R = Gamma at the row before the block (0 for the first block):
//   rows r in block R:  X[r] = [k_r ; q_r] * e^{Gamma_r - B_R}          (factor in [e^-80, 1])
//   columns j < 16(R+1): Y_R[j] = k_j * e^{B_R - Gamma_j}               (<= 1 before the block,
//                                                                        <= e^80 inside it)
//   D_R = X Y_R^T gives A (rows 0..63 of X, the k side) and P (rows 64..127, the q side) for
// the rows of block R; the other rows of D_R are not used. Every factor is formed from one
// exponential per element: e^{Gamma_r - B_R} and its inverse, times per-channel boundary
// factors e^{B_R' - B_R} <= 1.
//
// Layout and pipeline. One CTA (256 threads) owns one (sequence, head) problem. Per block:
//   TMA (4 tensors x two 64-column, 128-byte-swizzled boxes) -> shared memory
//   SIMT:   Gamma (registers), boundary factors, X and Y_R operands (bf16, swizzled)
//   tcgen05: D_R = X Y_R^T                                 (M=128, N=16(R+1), K=128) x4
//   SIMT:   A, P out of TMEM; T = (I + A)^{-1} by 16x16 block forward substitution;
//           T Diag(beta), K e^Gamma, Q e^Gamma, Khat operands
//   tcgen05: W^T = (K e^Gamma)^T (T Diag beta)^T,  U~^T = V^T (T Diag beta)^T   (M=128,N=64,K=64)
//   (next block's TMA is issued here: its inputs are no longer read)
//   tcgen05: U^T = U~^T - S^T W^T,  O^T = S^T (Q e^Gamma)^T                   (M=128,N=64,K=128)
//   tcgen05: dS = Khat^T U (M=128,N=128,K=64),  O^T += U^T P^T                (M=128,N=64,K=64)
//   SIMT:   O -> global (bf16); S <- e^{Gamma_L} S + dS kept in fp32 registers, bf16 copy to
//           shared memory as the next block's operand.
// The transposed forms keep every product at M = 128 (TMEM lane = row). The fp32 state lives
// in registers for the whole sequence (64 values per thread); only its bf16 copy feeds the
// tensor cores, so rounding does not accumulate in S itself.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <string>

#include "../../include/kda.h"
#include "kda_chunk_simt.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace tc {

constexpr int C = 64;
constexpr int D = 128;
constexpr int THREADS = 256;

// ---- shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t IN_K = 0, IN_Q = 16384, IN_V = 32768, IN_G = 49152;  // TMA tiles, 16 KB each
constexpr uint32_t RX = 65536;                 // 72 KB region, two uses per block:
constexpr uint32_t XA = RX;                    //   [k e^(G-B); q e^(G-B)]  128 x 128, K-major
constexpr uint32_t YB = RX + 32768;            //   Y_0..Y_3 (16,32,48,64 rows), K-major
constexpr uint32_t KG = RX;                    //   K e^Gamma  (A of W^T, MN-major)
constexpr uint32_t QG = RX + 16384;            //   Q e^Gamma  (B of O^T, K-major)
constexpr uint32_t KH = RX + 32768;            //   Khat       (A of dS, MN-major)
constexpr uint32_t WT = RX + 49152;            //   W^T        (B of U^T, MN-major)
constexpr uint32_t TB = RX + 65536;            //   T Diag(beta) (B of W^T and U~^T, K-major)
constexpr uint32_t SS = RX + 73728;            // bf16 S (A of U^T and O^T, MN-major), 32 KB
constexpr uint32_t US = SS + 32768;            // bf16 U (B of dS / A of O^T, K-major), 16 KB
constexpr uint32_t PS = US + 16384;            // bf16 P (B of O^T, K-major), 8 KB
constexpr uint32_t AM = PS + 8192;             // fp32 A, then T in place: [64][65]
constexpr uint32_t AM_LD = 65;
constexpr uint32_t SMEM_BYTES = AM + 64 * AM_LD * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for aligning the base
// Inside the G tile once Gamma is in registers (the tile is dead until the next TMA):
constexpr uint32_t TAB = IN_G;                 // float [14][128] boundary factors
constexpr uint32_t XM = IN_G + 14 * 128 * 4;   // float [16][48] block-solve scratch
constexpr uint32_t TX_BYTES = 4 * 16384;       // bytes landed by one block's TMA

__host__ __device__ constexpr uint32_t y_base(int R) { return YB + 4096u * (uint32_t)(R * (R + 1) / 2); }
__host__ __device__ constexpr uint32_t y_panel(int R) { return 2048u * (uint32_t)(R + 1); }

// ---- TMEM columns (512 allocated)
constexpr uint32_t TM_DS = 0, TM_U = 128, TM_O = 192, TM_WT = 256, TM_AP = 320;
__host__ __device__ constexpr uint32_t ap_off(int R) { return 8u * (uint32_t)(R * (R + 1)); }  // 0,16,48,96

// table rows inside TAB
constexpr int TAB_EXPB = 0;   // e^{B_R}, R = 0..3
constexpr int TAB_EXPL = 4;   // e^{B_4 - B_R}, R = 0..3   (B_4 = Gamma_L)
constexpr int TAB_E = 8;      // e^{B_R' - B_R}, pairs (R, R') with R < R' <= 3
__host__ __device__ constexpr int pair_index(int R, int Rp) {
  return R == 0 ? Rp - 1 : (R == 1 ? Rp + 1 : 5);  // (0,1)0 (0,2)1 (0,3)2 (1,2)3 (1,3)4 (2,3)5
}

struct TmaMaps {
  CUtensorMap q, k, v, g;
};

using namespace sm100;

__device__ __forceinline__ void st_bf16(uint8_t* base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float ld_bf16(const uint8_t* base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + off));
}

// Packs 8 floats into 8 bf16 (round to nearest even) and stores them as one 16-byte chunk.
__device__ __forceinline__ void st_chunk8(uint8_t* p, const float* x) {
  __nv_bfloat162 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = *reinterpret_cast<const uint4*>(h);
}

// Writes 32 consecutive values (columns col0..col0+31 of a 64-column swizzled panel row).
__device__ __forceinline__ void st_row32(uint8_t* panel, uint32_t row, uint32_t col0,
                                         const float* x) {
#pragma unroll
  for (int c = 0; c < 4; ++c) st_chunk8(panel + sw128_off(row, col0 + 8 * c), x + 8 * c);
}

__global__ void __launch_bounds__(THREADS, 1)
    chunk_tc_kernel(const __grid_constant__ TmaMaps maps, SeqParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_base_s;
  __shared__ float beta_s[C];
  __shared__ float xch[D];
  __shared__ float bnd[5][D];  // B_0..B_4 per channel (B_4 = Gamma_L)

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3;   // TMEM lane quarter this warp may address
  const int colhalf = warp >> 2;  // which half of the columns this warp handles
  const int c = tid & (D - 1);    // channel owned in the elementwise phases (= TMEM lane)
  const int rhalf = tid >> 7;     // rows 32*rhalf .. +31 in the elementwise phases

  int h, len;
  size_t row0;
  const int p = blockIdx.x;
  if (!resolve_problem(P, p, h, row0, len)) return;
  const int H = P.H;
  const __nv_bfloat16* __restrict__ beta_g = static_cast<const __nv_bfloat16*>(P.beta);
  __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(P.out);

  if (tid == 0) {
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    prefetch_tensormap(&maps.q);
    prefetch_tensormap(&maps.k);
    prefetch_tensormap(&maps.v);
    prefetch_tensormap(&maps.g);
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tlane = (uint32_t)(32 * quarter) << 16;

  auto issue_tma = [&](int t0) {
    mbar_arrive_expect_tx(&bar_tma, TX_BYTES);
    const int row = (int)(row0 + t0);
#pragma unroll
    for (int pnl = 0; pnl < 2; ++pnl) {
      tma_load_3d(sm + IN_K + pnl * 8192, &maps.k, 64 * pnl, h, row, &bar_tma);
      tma_load_3d(sm + IN_Q + pnl * 8192, &maps.q, 64 * pnl, h, row, &bar_tma);
      tma_load_3d(sm + IN_V + pnl * 8192, &maps.v, 64 * pnl, h, row, &bar_tma);
      tma_load_3d(sm + IN_G + pnl * 8192, &maps.g, 64 * pnl, h, row, &bar_tma);
    }
  };

  // ---- initial state: fp32 in registers (lane c, columns 64*colhalf + j), bf16 copy in SS
  float S[64];
  {
    const float* s0 = P.S0 ? P.S0 + ((size_t)p * D + c) * D + 64 * colhalf : nullptr;
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      float4 x = s0 ? *reinterpret_cast<const float4*>(s0 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
    }
    uint8_t* panel = sm + SS + 16384u * colhalf;
    st_row32(panel, c, 0, S);
    st_row32(panel, c, 32, S + 32);
  }
  if (tid == 0 && len > 0) issue_tma(0);

  uint32_t tma_phase = 0, mma_phase = 0;
  bool tma_pending = len > 0;
  bool aborted = false;

  auto mma_done = [&]() -> bool {
    const bool ok = mbar_wait(&bar_mma, mma_phase);
    mma_phase ^= 1u;
    tc_fence_after();
    return ok;
  };

  for (int t0 = 0; t0 < len && !aborted; t0 += C) {
    const int n = min(C, len - t0);
    // ---------------- stage: beta, wait for the tiles
    if (tid < C) beta_s[tid] = tid < n ? __bfloat162float(beta_g[(row0 + t0 + tid) * H + h]) : 0.f;
    {
      const bool ok = mbar_wait(&bar_tma, tma_phase);
      tma_phase ^= 1u;
      if (__syncthreads_or(!ok)) { aborted = true; break; }
      tma_pending = false;
    }
    // ---------------- Gamma (registers): thread owns channel c, rows 32*rhalf .. +31
    float Gm[32];
    {
      const uint8_t* gp = sm + IN_G + (c >> 6) * 8192;
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * rhalf + i;
        acc += r < n ? ld_bf16(gp, sw128_off(r, c & 63)) : 0.f;
        Gm[i] = acc;
      }
      if (rhalf == 0) xch[c] = acc;
    }
    __syncthreads();
    if (rhalf == 1) {
      const float base = xch[c];
#pragma unroll
      for (int i = 0; i < 32; ++i) Gm[i] += base;
      bnd[3][c] = Gm[15];
      bnd[4][c] = Gm[31];
    } else {
      bnd[0][c] = 0.f;
      bnd[1][c] = Gm[15];
      bnd[2][c] = Gm[31];
    }
    __syncthreads();
    float* tab = reinterpret_cast<float*>(sm + TAB);
    if (tid < D) {
      float b[5];
#pragma unroll
      for (int R = 0; R < 5; ++R) b[R] = bnd[R][c];
#pragma unroll
      for (int R = 0; R < 4; ++R) {
        tab[(TAB_EXPB + R) * D + c] = __expf(b[R]);
        tab[(TAB_EXPL + R) * D + c] = __expf(b[4] - b[R]);
      }
#pragma unroll
      for (int R = 0; R < 3; ++R)
#pragma unroll
        for (int Rp = R + 1; Rp < 4; ++Rp) tab[(TAB_E + pair_index(R, Rp)) * D + c] = __expf(b[Rp] - b[R]);
    }
    // F = e^{Gamma_r - B_R} and its inverse, kept for the second operand pass
    float F[32], Fi[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int R = (32 * rhalf + i) >> 4;
      const float L = Gm[i] - bnd[R][c];
      F[i] = __expf(L);
      Fi[i] = __expf(-L);
    }
    __syncthreads();
    // ---------------- X = [k F ; q F] and Y_R' = k Fi e^{B_R - B_R'}... (R' >= R)
    {
      const uint8_t* kp = sm + IN_K + (c >> 6) * 8192;
      const uint8_t* qp = sm + IN_Q + (c >> 6) * 8192;
      uint8_t* xa = sm + XA + (c >> 6) * 16384;
      const int cc = c & 63;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * rhalf + i;
        const int R = r >> 4;
        const uint32_t o = sw128_off(r, cc);
        const float kk = r < n ? ld_bf16(kp, o) : 0.f;
        const float qq = r < n ? ld_bf16(qp, o) : 0.f;
        st_bf16(xa, o, kk * F[i]);
        st_bf16(xa, sw128_off(64 + r, cc), qq * F[i]);
        const float kf = kk * Fi[i];
#pragma unroll
        for (int Rp = 0; Rp < 4; ++Rp) {
          if (Rp < R) continue;
          const float e = Rp == R ? 1.f : tab[(TAB_E + pair_index(R, Rp)) * D + c];
          st_bf16(sm + y_base(Rp) + (c >> 6) * y_panel(Rp), o, kf * e);
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    // ---------------- tcgen05: D_R = X Y_R^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int R = 0; R < 4; ++R) {
        const uint32_t idesc = idesc_bf16(128, 16 * (R + 1), 0, 0, 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t a = desc_sw128(smem_u32(sm + XA + (kk >> 2) * 16384 + (kk & 3) * 32), 16, 1024);
          const uint64_t b = desc_sw128(
              smem_u32(sm + y_base(R) + (kk >> 2) * y_panel(R) + (kk & 3) * 32), 16, 1024);
          umma_bf16(tmem + TM_AP + ap_off(R), a, b, idesc, kk > 0);
        }
      }
      umma_commit(&bar_mma);
    }
    if (__syncthreads_or(!mma_done())) { aborted = true; break; }
    // ---------------- A and P out of TMEM
    {
      float* Am = reinterpret_cast<float*>(sm + AM);
      const bool pside = quarter >= 2;
      const int r = (quarter & 1) * 32 + lane;     // block row index of this lane
      const int R = ((quarter & 1) << 1) + colhalf;  // block this warp reads
      const bool valid = (r >> 4) == R;
      const int NR = 16 * (R + 1);
      for (int c0 = 0; c0 < NR; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + tlane + TM_AP + ap_off(R) + c0, v);
        tmem_ld_wait();
        if (valid) {
          if (!pside) {
            const float b = beta_s[r];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int jj = c0 + j;
              Am[r * AM_LD + jj] = (jj < r) ? b * __uint_as_float(v[j]) : 0.f;
            }
          } else {
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = (c0 + j <= r) ? __uint_as_float(v[j]) : 0.f;
            st_row32(sm + PS, r, c0, x);
          }
        }
      }
      if (valid) {  // the rest of the row is the (zero) upper triangle
        if (!pside) {
          for (int jj = NR; jj < C; ++jj) Am[r * AM_LD + jj] = 0.f;
        } else if (NR < C) {
          float z[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) z[j] = 0.f;
          for (int c0 = NR; c0 < C; c0 += 32) {
            // NR is a multiple of 16; write whole 8-element chunks up to 64
            for (int cc8 = c0; cc8 < c0 + 32 && cc8 < C; cc8 += 8)
              st_chunk8(sm + PS + sw128_off(r, cc8), z);
          }
        }
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    // ---------------- T = (I + A)^{-1}, in place in Am (16x16 block forward substitution)
    {
      float* Am = reinterpret_cast<float*>(sm + AM);
      float* Xm = reinterpret_cast<float*>(sm + XM);
      float col[16];
      const int Rd = tid >> 4, jj = tid & 15;
      if (tid < 64) {
#pragma unroll
        for (int r2 = 0; r2 < 16; ++r2) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < r2; ++i) acc = fmaf(Am[(16 * Rd + r2) * AM_LD + 16 * Rd + i], col[i], acc);
          col[r2] = (r2 == jj) ? 1.f : (r2 > jj ? -acc : 0.f);
        }
      }
      __syncthreads();
      if (tid < 64) {
#pragma unroll
        for (int r2 = 0; r2 < 16; ++r2) Am[(16 * Rd + r2) * AM_LD + 16 * Rd + jj] = col[r2];
      }
      __syncthreads();
      for (int R = 1; R < 4; ++R) {
        const int nJ = 16 * R;
        for (int idx = tid; idx < 16 * nJ; idx += THREADS) {
          const int rr = idx / nJ, j = idx % nJ;
          const float* arow = Am + (16 * R + rr) * AM_LD;
          float acc = 0.f;
          for (int i = j; i < nJ; ++i) acc = fmaf(arow[i], Am[i * AM_LD + j], acc);
          Xm[rr * 48 + j] = -acc;
        }
        __syncthreads();
        for (int idx = tid; idx < 16 * nJ; idx += THREADS) {
          const int rr = idx / nJ, j = idx % nJ;
          const float* trow = Am + (16 * R + rr) * AM_LD + 16 * R;
          float acc = 0.f;
          for (int i = 0; i <= rr; ++i) acc = fmaf(trow[i], Xm[i * 48 + j], acc);
          Am[(16 * R + rr) * AM_LD + j] = acc;
        }
        __syncthreads();
      }
      // T Diag(beta) -> bf16, K-major (row r, column j)
      {
        const int r = tid >> 2, j0 = (tid & 3) * 16;
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = (j0 + j <= r) ? Am[r * AM_LD + j0 + j] * beta_s[j0 + j] : 0.f;
        st_chunk8(sm + TB + sw128_off(r, j0), x);
        st_chunk8(sm + TB + sw128_off(r, j0 + 8), x + 8);
      }
    }
    // K e^Gamma, Q e^Gamma, Khat (same swizzled [row][channel] layout as the input tiles)
    {
      const uint8_t* kp = sm + IN_K + (c >> 6) * 8192;
      const uint8_t* qp = sm + IN_Q + (c >> 6) * 8192;
      const float* tab2 = reinterpret_cast<const float*>(sm + TAB);
      const int cc = c & 63;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * rhalf + i;
        const int R = r >> 4;
        const uint32_t o = sw128_off(r, cc);
        const float kk = r < n ? ld_bf16(kp, o) : 0.f;
        const float qq = r < n ? ld_bf16(qp, o) : 0.f;
        const float eg = F[i] * tab2[(TAB_EXPB + R) * D + c];
        st_bf16(sm + KG + (c >> 6) * 8192, o, kk * eg);
        st_bf16(sm + QG + (c >> 6) * 8192, o, qq * eg);
        st_bf16(sm + KH + (c >> 6) * 8192, o, kk * Fi[i] * tab2[(TAB_EXPL + R) * D + c]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    // ---------------- tcgen05: W^T and U~^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, 1, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t b = desc_sw128(smem_u32(sm + TB + kk * 32), 16, 1024);
        umma_bf16(tmem + TM_WT, desc_sw128(smem_u32(sm + KG + kk * 2048), 8192, 1024), b, idesc, kk > 0);
        umma_bf16(tmem + TM_U, desc_sw128(smem_u32(sm + IN_V + kk * 2048), 8192, 1024), b, idesc, kk > 0);
      }
      umma_commit(&bar_mma);
    }
    if (__syncthreads_or(!mma_done())) { aborted = true; break; }
    // the input tiles are free: fetch the next block while the serial part runs
    if (tid == 0 && t0 + C < len) {
      issue_tma(t0 + C);
      tma_pending = true;
    }
    // W^T -> bf16 (MN-major B: row = channel c, columns = r)
    {
      uint32_t v[32];
      tmem_ld32(tmem + tlane + TM_WT + 32 * colhalf, v);
      tmem_ld_wait();
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
      st_row32(sm + WT, 32 * quarter + lane, 32 * colhalf, x);
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    // ---------------- tcgen05: U^T = U~^T - S^T W^T ; O^T = S^T (Q e^Gamma)^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_u = idesc_bf16(128, 64, 1, 1, 1);
      const uint32_t id_o = idesc_bf16(128, 64, 1, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t a = desc_sw128(smem_u32(sm + SS + kk * 2048), 16384, 1024);
        umma_bf16(tmem + TM_U, a, desc_sw128(smem_u32(sm + WT + kk * 2048), 16384, 1024), id_u, 1);
        umma_bf16(tmem + TM_O, a,
                  desc_sw128(smem_u32(sm + QG + (kk >> 2) * 8192 + (kk & 3) * 32), 16, 1024), id_o,
                  kk > 0);
      }
      umma_commit(&bar_mma);
    }
    if (__syncthreads_or(!mma_done())) { aborted = true; break; }
    // U -> bf16, K-major (row = v, column = r)
    {
      uint32_t v[32];
      tmem_ld32(tmem + tlane + TM_U + 32 * colhalf, v);
      tmem_ld_wait();
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
      st_row32(sm + US, 32 * quarter + lane, 32 * colhalf, x);
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    // ---------------- tcgen05: dS = Khat^T U ; O^T += U^T P^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_s = idesc_bf16(128, 128, 1, 0, 0);
      const uint32_t id_o = idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t u = desc_sw128(smem_u32(sm + US + kk * 32), 16, 1024);
        umma_bf16(tmem + TM_DS, desc_sw128(smem_u32(sm + KH + kk * 2048), 8192, 1024), u, id_s, kk > 0);
        umma_bf16(tmem + TM_O, u, desc_sw128(smem_u32(sm + PS + kk * 32), 16, 1024), id_o, 1);
      }
      umma_commit(&bar_mma);
    }
    if (__syncthreads_or(!mma_done())) { aborted = true; break; }
    // ---------------- outputs and the state update
    {
      uint32_t v[32];
      tmem_ld32(tmem + tlane + TM_O + 32 * colhalf, v);
      tmem_ld_wait();
      const int vcol = 32 * quarter + lane;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int r = 32 * colhalf + j;
        if (r < n) out[((row0 + t0 + r) * H + h) * D + vcol] = __float2bfloat16_rn(__uint_as_float(v[j]));
      }
      const float gl = __expf(bnd[4][c]);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        tmem_ld32(tmem + tlane + TM_DS + 64 * colhalf + 32 * half, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) S[32 * half + j] = fmaf(gl, S[32 * half + j], __uint_as_float(v[j]));
      }
      uint8_t* panel = sm + SS + 16384u * colhalf;
      st_row32(panel, c, 0, S);
      st_row32(panel, c, 32, S + 32);
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
  }

  if (aborted) {
    record_status(4u /* KDA_ERR_TIMEOUT */);
    if (tma_pending) (void)mbar_wait(&bar_tma, tma_phase);  // let an issued copy land
  } else if (P.S_final) {
    float* sf = P.S_final + ((size_t)p * D + c) * D + 64 * colhalf;
#pragma unroll
    for (int j = 0; j < 64; j += 4) *reinterpret_cast<float4*>(sf + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side

inline bool tc_supports(int C_) { return C_ == C; }

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [rows, H, 128] bf16 token tensor viewed as a 3-D map with 64 x 1 x 64 boxes, 128-byte swizzle.
inline bool encode_token_map(CUtensorMap* m, const void* base, long long rows, int H) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

inline bool tc_supports(int C) { return tc::tc_supports(C); }

inline kda_status_t launch_chunk_tc(const SeqParams& P, int n_problems, int C, cudaStream_t st,
                                    std::string& err) {
  (void)C;
  tc::TmaMaps maps;
  const long long rows = P.cu_seqlens ? (long long)P.T : (long long)P.n_seq * P.T;
  if (!tc::encode_token_map(&maps.q, P.q, rows, P.H) || !tc::encode_token_map(&maps.k, P.k, rows, P.H) ||
      !tc::encode_token_map(&maps.v, P.v, rows, P.H) || !tc::encode_token_map(&maps.g, P.g, rows, P.H)) {
    err = "cuTensorMapEncodeTiled failed";
    return KDA_ERR_CUDA;
  }
  cudaError_t e = cudaFuncSetAttribute(tc::chunk_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc::SMEM_ALLOC);
  if (e != cudaSuccess) {
    err = std::string("cudaFuncSetAttribute(chunk_tc): ") + cudaGetErrorString(e);
    return KDA_ERR_CUDA;
  }
  tc::chunk_tc_kernel<<<n_problems, tc::THREADS, tc::SMEM_ALLOC, st>>>(maps, P);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("chunk_tc launch: ") + cudaGetErrorString(e);
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

}  // namespace kda
