// Composition of segment transitions: the incoming state of every T-segment of a sequence.
//
// Kimi K3 wiki, "Notations mathématiques", table "Attention et KDA": M_t is the transition
// (I - beta_t k_t k_t^T) Diag(alpha_t) and S~ the state reached from S = 0; "Glossaire", entry
// "KCP": the pair (cumulative M, local S~) of a stretch of tokens composes associatively. For
// segments sigma = 0, 1, ... of one (sequence, head) with pairs (M_sigma, S~_sigma):
//   S_in(0) = S0,   S_in(sigma + 1) = M_sigma S_in(sigma) + S~_sigma.
// Columns of S are independent, so one CTA owns (sequence, head, 1024 / d_k value columns) and walks
// the segments in order. M_sigma (fp32, d_k x d_k) is staged in shared memory by asynchronous
// copies one segment ahead, S~ one segment ahead in registers; the NC columns of S_in stay in
// shared memory; fp32 FMAs throughout.
//
// Layouts (fp32, row-major): M [n_seg - 1, BH, DK, DK]; St [n_seg - 1, BH, DK, DV];
// S0 [BH, DK, DV] or null (zeros); S_in [n_seg, BH, DK, DV].
#pragma once

#include "kda_common.cuh"

namespace kda {
namespace scan {

constexpr int THREADS = 256;

template <int DK>
struct ScanSmem {
  static constexpr int NC = 1024 / DK;  // value columns per CTA: 4 per thread
  static constexpr int LDM = DK + 4;  // padded row stride of M (16-byte aligned rows)
  static constexpr size_t m_floats = (size_t)DK * LDM;
  static constexpr size_t bytes = (2 * m_floats + (size_t)DK * NC) * sizeof(float);
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int DK, int DV>
__global__ void __launch_bounds__(THREADS)
    segment_scan_kernel(const float* __restrict__ M, const float* __restrict__ St,
                        const float* __restrict__ S0, float* __restrict__ S_in, int n_seg, int BH) {
  using SM = ScanSmem<DK>;
  constexpr int LDM = SM::LDM;
  constexpr int NC = SM::NC;
  constexpr int CPT = DK * NC / THREADS;  // columns per thread
  constexpr int TPR = NC / CPT;           // threads per row
  static_assert(CPT % 4 == 0 && NC % CPT == 0, "bad scan tiling");
  extern __shared__ __align__(16) float sm[];
  float* Sc = sm + 2 * SM::m_floats;  // [DK][NC]; M double-buffered before it

  const int bh = blockIdx.x;
  const int c_base = blockIdx.y * NC;
  const int tid = threadIdx.x;
  const int i = tid / TPR;           // row of S owned in the products
  const int c0 = (tid % TPR) * CPT;  // first of its columns inside the tile
  const size_t mat = (size_t)DK * DK, st = (size_t)DK * DV;

  auto load_m = [&](int sigma, float* dst) {
    const float* src = M + ((size_t)sigma * BH + bh) * mat;
    for (int e = tid; e < DK * DK / 4; e += THREADS) {
      const int r = e / (DK / 4), c4 = e % (DK / 4);
      cp_async16(dst + r * LDM + 4 * c4, src + (size_t)r * DK + 4 * c4);
    }
    cp_async_commit();
  };

  // S_in(0) = S0 (or zeros), into the tile and out to S_in[0]
  float acc[CPT];
  {
    const float* s0 = S0 ? S0 + (size_t)bh * st + (size_t)i * DV + c_base + c0 : nullptr;
#pragma unroll
    for (int j = 0; j < CPT; j += 4) {
      float4 x = s0 ? *reinterpret_cast<const float4*>(s0 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      acc[j] = x.x; acc[j + 1] = x.y; acc[j + 2] = x.z; acc[j + 3] = x.w;
    }
  }
  // S~ of the step in flight, loaded one step ahead so that its latency overlaps a step's products
  float4 stn[CPT / 4];
  auto load_st = [&](int sigma) {
    const float* st_row = St + ((size_t)sigma * BH + bh) * st + (size_t)i * DV + c_base + c0;
#pragma unroll
    for (int j = 0; j < CPT; j += 4) stn[j / 4] = *reinterpret_cast<const float4*>(st_row + j);
  };
  if (n_seg > 1) {
    load_m(0, sm);
    load_st(0);
  }
  for (int sigma = 0;; ++sigma) {
    float* out = S_in + ((size_t)sigma * BH + bh) * st + (size_t)i * DV + c_base + c0;
#pragma unroll
    for (int j = 0; j < CPT; j += 4) {
      *reinterpret_cast<float4*>(out + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
      *reinterpret_cast<float4*>(Sc + i * NC + c0 + j) =
          make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
    }
    if (sigma + 1 >= n_seg) break;
    // the next segment's M one step ahead, then wait for this one's
    if (sigma + 2 < n_seg) {
      load_m(sigma + 1, sm + ((sigma + 1) & 1) * SM::m_floats);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // M_sigma and the tile are in place
#pragma unroll
    for (int j = 0; j < CPT; j += 4) {
      const float4 x = stn[j / 4];
      acc[j] = x.x; acc[j + 1] = x.y; acc[j + 2] = x.z; acc[j + 3] = x.w;
    }
    if (sigma + 2 < n_seg) load_st(sigma + 1);
    const float* mrow = sm + (sigma & 1) * SM::m_floats + i * LDM;
#pragma unroll 4
    for (int k = 0; k < DK; k += 4) {
      const float4 m = *reinterpret_cast<const float4*>(mrow + k);
      const float mk[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float* srow = Sc + (k + kk) * NC + c0;
#pragma unroll
        for (int j = 0; j < CPT; j += 4) {
          const float4 s = *reinterpret_cast<const float4*>(srow + j);
          acc[j] = fmaf(mk[kk], s.x, acc[j]);
          acc[j + 1] = fmaf(mk[kk], s.y, acc[j + 1]);
          acc[j + 2] = fmaf(mk[kk], s.z, acc[j + 2]);
          acc[j + 3] = fmaf(mk[kk], s.w, acc[j + 3]);
        }
      }
    }
    __syncthreads();  // every thread has read the tile and M_sigma
  }
}

}  // namespace scan
}  // namespace kda
