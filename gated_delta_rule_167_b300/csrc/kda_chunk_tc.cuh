// Tensor-core chunkwise KDA prefill for bf16 inputs in 64-token blocks, sm_103a: d_k = d_v = 128
// (64-channel heads run in the same tiles, zero-padded in shared memory), with the input side
// (short convolution, L2 norm, gate) and the output side (RMSNorm, output gate) optionally fused.
//
// Mathematics (Kimi K3 wiki: "Notations mathématiques", table "Attention et KDA" for the
// recurrence; "Glossaire", entries "Chunkwise", "UT" and "Décroissance bornée"). For one block
// of C tokens with incoming state S, Gamma the inclusive cumulative sum of g inside the block:
//   A_rj = beta_r sum_c k_rc k_jc e^{Gamma_rc - Gamma_jc} (j < r)
//   (I + A) U = Diag(beta) (V - (K e^Gamma) S)     (the UT transform of the residual)
//   P_rj = sum_c q_rc k_jc e^{Gamma_rc - Gamma_jc} (j <= r),  O = (Q e^Gamma) S + P U
//   S' = Diag(e^{Gamma_L}) S + Khat^T U,  Khat_j = k_j e^{Gamma_L - Gamma_j}
// U equals U~ - W S with U~ = T Diag(beta) V, W = T Diag(beta) K e^Gamma and T = (I + A)^{-1};
// forming the residual V - (K e^Gamma) S first needs no W. T is formed explicitly: the four
// 16 x 16 diagonal inverses by forward substitution, then the block-inverse identity
//   [[P, 0], [C, Q]]^{-1} = [[P^{-1}, 0], [-Q^{-1} C P^{-1}, Q^{-1}]]
// inside each 32-token half and for the two halves, and U = T Diag(beta) (V - Z) is one
// tensor-core product with Z = (K e^Gamma) S.
//
// Bounded decay. Over a block of 64 tokens Gamma can fall to -320, so e^{-Gamma} overflows any
// floating type and A, P cannot be one product (K e^Gamma)(K e^{-Gamma})^T. With
// g >= g_min = -5 every 16-token sub-block spans at most e^80, inside the bf16/fp32 range. The
// block is split into two 32-token halves, each with its own reference point rho placed on the
// boundary between its two 16-token sub-blocks (rho_A = Gamma_15, rho_B = Gamma_47):
//   X[r]   = [k_r ; q_r] e^{Gamma_r - rho(r)}     for every row r        (factor in [e^-80, e^75])
//   Y_A[j] = k_j e^{rho_A - Gamma_j}              for j < 32             (in [e^-75, e^80])
//   Y_B[j] = k_j e^{rho_B - Gamma_j}              for j < 64             (<= e^80)
// so that one tensor-core product X [Y_B ; Y_A]^T (N = 96) holds every A_rj and P_rj with
// j <= r: rows of the first half read the Y_A columns, rows of the second half the Y_B columns.
// Entries above the diagonal may overflow in that product; they are discarded by selection.
//
// Layout. One CTA (512 threads) owns one (sequence, head) problem and walks its blocks in
// order. The state is kept transposed in TMEM: S^T in fp32 (lane = value channel v, column =
// key channel c) and its bf16 copy, which is the A operand of the products with S. Every
// intermediate of the state update (the residual Z = (K e^Gamma) S, U, the bf16 copies) goes
// TMEM -> registers -> TMEM, so only operands built from the inputs pass through shared memory.
//
// Two warp groups work on consecutive blocks at the same time:
//   group P (warps 0-7), block n + 1: X, Y, (K e^Gamma)^T, (Q e^Gamma)^T, Khat^T from transposed
//     8 x 8 matrix loads of the inputs (running sums of g by warp MMAs), written back by matrix
//     stores as [channel][token] rows; the A/P product D = X [Y_B | Y_A]^T; A (fp32) and P (bf16)
//     out of TMEM; the diagonal inverses T_RR; then, once S has finished block n, Khat^T of
//     block n + 1 and block n's O out of TMEM.
//   group S (warps 8-15), block n:
//     tcgen05: Z^T = S^T (K e^Gamma)^T, O^T = S^T (Q e^Gamma)^T; while it runs, the off-diagonal
//       blocks of T (tf32 warp MMAs) and G = T Diag(beta) (bf16); then Z^T -> bf16
//     tcgen05: U^T = V^T G^T - Z^T G^T; while it runs, S^T <- S^T e^{Gamma_L}; U^T -> bf16
//     tcgen05: O^T += U^T P^T;  S^T += U^T Khat;  SIMT: bf16 copy of S^T
// Shared buffers pass between the groups through mbarriers: P may rewrite X and Y once its
// A/P product of the previous block has completed, (K/Q e^Gamma)^T once S's first product has,
// A (WS) once S has finished its solve, and Khat^T (held in registers until then) once S's last
// product has; S starts a block once P has written that block's operands and the O of two
// blocks ago (O^T and P are double-buffered by block parity). Transposed products keep every
// tcgen05 product at M = 128 (TMEM lane = row). Only the bf16 copy of the state feeds the tensor
// cores; the fp32 state accumulates in TMEM, so rounding does not accumulate in S itself. Every
// wait ends by a per-CTA deadline; after a wait gives up the later ones end at once, the groups
// run through their remaining blocks, and the kernel latches KDA_ERR_TIMEOUT, lets issued copies
// and products land, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <string>

#include "../../include/kda.h"
#include "kda_chunk_simt.cuh"
#include "kda_post.cuh"
#include "kda_pre.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace tc {

constexpr int C = 64;
constexpr int D = 128;
constexpr int THREADS = 512;  // two groups of 256
constexpr int GROUP = 256;
constexpr int BAR_P = 1, BAR_S = 2;  // hardware barrier ids of the groups
constexpr int BAR_PAIR0 = 3;        // ids 3..6: pairs of warps of the state group in its solve
constexpr int BAR_TILE0 = 7;        // ids 7, 8: the two warps of a diagonal tile in the solve
constexpr int kLongestFirstMax = 256;  // packed batches of up to this many sequences run longest first
constexpr float LOG2E = 1.4426950408889634f;

// Row stride (floats) of the fp32 64 x 64 solve workspace: 76 puts the eight 16-byte rows of a
// matrix load, and the rows of a warp's 16-byte stores, in distinct banks.
constexpr int WLD = 76;

// ---- shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t IN_K = 0;           // k tile (two 64-channel boxes of [64 tokens][64])
constexpr uint32_t IN_Q = 16384;       // q tile
constexpr uint32_t IN_G = 32768;       // g tile
constexpr uint32_t IN_V = 49152;       // v tile: MN-major A operand V^T of U^T = V^T G^T - Z^T G^T
constexpr uint32_t XK = 65536;         // X rows 0..63 (k side), MN-major A panel 0
constexpr uint32_t XQ = XK + 16384;    // X rows 64..127 (q side), MN-major A panel 1
constexpr uint32_t YP = XQ + 16384;    // [Y_B | Y_A], N = 96 columns in 2 MN-major B panels
// (K e^Gamma)^T and (Q e^Gamma)^T [c][r]: the two MN-major B panels of the product with S, in
// the order of its TMEM output: even blocks [(Q e^Gamma)^T | (K e^Gamma)^T] -> [O^T | Z^T],
// odd blocks [(K e^Gamma)^T | (Q e^Gamma)^T] -> [Z^T | O^T]
constexpr uint32_t KQ = YP + 32768;    // 2 x 16 KB
constexpr uint32_t KH = KQ + 32768;    // Khat^T [c][r]: K-major B of S^T += U^T Khat
constexpr uint32_t WS = KH + 16384;    // fp32 A, then T ([64][WLD], 19 KB)
constexpr uint32_t PT = WS + 64 * WLD * 4;  // P [r][j], K-major B of O^T += U^T P^T, 2 x 8 KB by parity
constexpr uint32_t GB = PT + 16384;    // G = T Diag(beta) [r][j] bf16, K-major B of U^T (8 KB)
constexpr uint32_t SMEM_BYTES = GB + 8192;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for aligning the base
constexpr uint32_t BOX_BYTES = 8192;                // one 64-channel x 64-token TMA box

// ---- TMEM columns (512 allocated)
constexpr uint32_t T_ST = 0;    // S^T fp32 [v][c], 128
constexpr uint32_t T_SB = 128;  // S^T bf16 (A operand), 64
constexpr uint32_t T_D = 192;   // X [Y_B | Y_A]^T, 96
// O^T fp32 by block parity at 288 (even) and 416 (odd), Z^T fp32 between them at 352, so that
// [O^T | Z^T] (even) and [Z^T | O^T] (odd) are one 128-column product; group P writes one O^T
// out while group S accumulates the other
constexpr uint32_t T_ZT = 352;  // Z^T fp32, 64; after its bf16 copy: U^T fp32
__host__ __device__ constexpr uint32_t t_ot_of(int b) { return (b & 1) ? 416u : 288u; }
constexpr uint32_t T_ZB = 480;  // Z^T bf16 (A operand), 32
constexpr uint32_t T_UT = T_ZT;  // U^T fp32 once Z^T has its bf16 copy
constexpr uint32_t T_UB = T_ZB;  // U^T bf16 (A operand), over Z^T bf16 once the U product read it

// Columns of the A/P product: Y_B (reference rho_B) at 0..63, Y_A (rho_A) at 64..95.
constexpr int Y_A = 64;

constexpr int TLD = 20;  // row stride (floats) of the diagonal inverses
struct TmaMaps {
  CUtensorMap q, k, v, g;
  CUtensorMap u;  // output gate rows (output side fused only)
};

using namespace sm100;

// 16 x 8 tile of acc += A B over K = 8 nk (nk <= 4) with tf32 warp MMAs on fp32 values already
// rounded to tf32: A as four 8 x 8 b16 matrix loads (8 rows x 4 fp32 each: rows 0-7 / 8-15 x
// columns 0-3 / 4-7, which is the tf32 A fragment; Ab has 16-byte aligned rows), B as two
// 32-bit loads per k step.
__device__ __forceinline__ void tile_mma(float (&acc)[4], const float* Ab, int lda, const float* Bb,
                                         int ldb, int nk) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const uint32_t ar = smem_u32(Ab) + 4u * (uint32_t)(((lane & 7) + 8 * ((lane >> 3) & 1)) * lda + 4 * (lane >> 4));
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    if (ks < nk) {
      uint32_t a[4];
      ldsm_x4(ar + 32u * (uint32_t)ks, a);
      const uint32_t b[2] = {__float_as_uint(Bb[(8 * ks + t) * ldb + g]),
                             __float_as_uint(Bb[(8 * ks + t + 4) * ldb + g])};
      mma_tf32(acc, a, b);
    }
  }
}

// Input side, fused. Thread (cg, rg) of a group handles channels [8 cg, 8 cg + 8) of rows
// 4 rg .. 4 rg + 3 of a staged [64 tokens][128] bf16 tile (two 128-byte-swizzled 64-channel
// boxes); the 16 threads of a row are the lanes of a half-warp. Chunk address of row r:
__device__ __forceinline__ uint32_t tile_chunk(int cg, int r) {
  return (uint32_t)((cg >> 3) * BOX_BYTES + r * 128 + 16 * ((cg & 7) ^ (r & 7)));
}

// The causal 4-tap convolution of this thread's 4 rows (tap-major weights w[h][j][c], all 32 of
// this thread's taps loaded in one batch before they are needed, so that their latency is paid
// once). Taps before row 0 come from the previous block's last three raw rows, which that block's
// pass left in a stash (halo(hr) = address of this thread's chunk of raw row 61 + hr);
// `first_pos` is the position of row 0 inside its sequence, so that no tap reaches before a
// sequence start. The 7 input rows stay packed (bf16 pairs) until used.
template <typename Halo>
__device__ __forceinline__ void conv_rows4(const uint8_t* tile, const float* w, int h, int cg, int rg,
                                           int first_pos, Halo halo, float (&y)[4][8]) {
  float t[4][8];
  pre::load_taps<D>(w, h, 8 * cg, t);
  uint32_t xr[7][4];
#pragma unroll
  for (int m = 0; m < 7; ++m) {
    const int r = 4 * rg + m - 3;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r >= 0) v = *reinterpret_cast<const uint4*>(tile + tile_chunk(cg, r));
    else if (first_pos > 0) v = *reinterpret_cast<const uint4*>(halo(r + 3));
    xr[m][0] = v.x; xr[m][1] = v.y; xr[m][2] = v.z; xr[m][3] = v.w;
  }
  // channels in pairs (e, e + 1), one packed fma per tap: each lane rounds as fmaf does, in the
  // same tap order
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float2 x[7];
#pragma unroll
    for (int m = 0; m < 7; ++m)
      x[m] = make_float2(__uint_as_float(xr[m][e >> 1] << 16), __uint_as_float(xr[m][e >> 1] & 0xFFFF0000u));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 a = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j <= first_pos + 4 * rg + i) a = fma2(make_float2(t[j][e], t[j][e + 1]), x[i + 3 - j], a);
      y[i][e] = a.x;
      y[i][e + 1] = a.y;
    }
  }
}

// Copies this thread's chunks of raw rows 61..63 (threads of rows 60..63) into the stash.
template <typename Halo>
__device__ __forceinline__ void stash_rows(const uint8_t* tile, int cg, Halo halo) {
#pragma unroll
  for (int r = 61; r < 64; ++r)
    *reinterpret_cast<uint4*>(halo(r - 61)) = *reinterpret_cast<const uint4*>(tile + tile_chunk(cg, r));
}

// Writes this thread's 4 rows (packed bf16) back into a staged tile.
__device__ __forceinline__ void put_rows4(uint8_t* tile, int cg, int rg, const uint4 (&pk)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(tile + tile_chunk(cg, 4 * rg + i)) = pk[i];
}

__device__ __forceinline__ void st_pack8(uint32_t saddr, const float (&x)[8]) {
  st_shared_v4(saddr, pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
               pack_bf16(x[6], x[7]));
}

// PRE: the inputs are the raw projections and the input side is computed in the kernel; POST: the
// output side is applied in the output epilogue. The plain kernel (both false) carries neither.
// DH is the head size of the tensors in memory, d_k = d_v = 128 or 64. At 64 (the plain kernel
// only) the problem runs in the same 128-channel tiles: the TMA loads only the first 64-channel
// box of each tile and the second box stays zero, so k, q, v and g are zero-padded (g = 0 is a
// decay factor of 1). Padded key channels of S are never written (k = 0 there) and padded value
// channels stay zero (v = 0 and Z = 0 there), so the first 64 x 64 block of S and the first 64
// channels of O are those of the unpadded problem; only they are read in and written out.
template <bool PRE, bool POST, int DH = 128>
__global__ void __launch_bounds__(THREADS, 1)
    chunk_tc_kernel(const __grid_constant__ TmaMaps maps, SeqParams P) {
  static_assert(DH == 128 || (DH == 64 && !PRE && !POST), "head size 64: plain kernel only");
  constexpr int NBOX = DH / 64;  // 64-channel boxes loaded per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  // bar_in: k, q, g tiles landed          bar_v: v tile landed
  // bar_prep: P finished a block's operands (release / acquire for its generic stores)
  // bar_ext: P has taken A (into WS) and P (into PT) out of the A/P product, made the diagonal
  //          inverses T_RR (trr) and rounded the A blocks that S multiplies to tf32
  // bar_wsfree: S has read a block's A out of WS (P may put the next one there)
  // bar_khr: P has stored a block's Khat^T and read the previous block's O out of TMEM
  // bar_D, bar_ZO, bar_G2, bar_G3: tcgen05 products complete
  __shared__ uint64_t bar_in, bar_v, bar_prep, bar_ext, bar_wsfree, bar_khr, bar_D, bar_ZO, bar_G2,
      bar_G3;
  // bar_qg (input side fused): group S has formed a block's q and g in place in the staged tiles
  // bar_u (output side fused): a block's gate rows u have landed in XQ
  __shared__ uint64_t bar_qg, bar_u;
  __shared__ uint32_t tmem_base_s;
  __shared__ int cta_abort;  // this CTA ran past its deadline (a wait gave up)
  __shared__ __align__(16) float beta_s[2][C];  // by block parity
  __shared__ __align__(16) float gl_s[2][D];    // e^{Gamma_L} per key channel, by block parity
  // diagonal blocks T_RR of the solve (written by group P, read by group S); rows of 20 floats:
  // 16-byte aligned, and the eight row addresses of a matrix load fall in distinct banks
  __shared__ __align__(16) float trr[4][16][TLD];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int quarter = warp & 3;   // TMEM lane quarter this warp may address
  const bool isP = tid < GROUP;
  const int lt = tid & (GROUP - 1);  // index inside the group
  const int c = lt & (D - 1);        // channel (= TMEM lane) owned in the elementwise phases
  const int hh = lt >> 7;            // which half this thread handles inside its group
  const int lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;  // mma fragment coordinates

  // A packed batch is launched longest sequences first: CTAs start in blockIdx order, so giving
  // the (sequence, head) problems of the longest sequences the lowest indices evens out the end
  // of the launch. Thread s < n_seq ranks sequence s (length descending, index ascending on
  // ties, a permutation whatever the offsets hold); CTA p takes the sequence of rank p / H.
  int p = blockIdx.x;
  if (P.cu_seqlens != nullptr && P.seg_len == 0 && P.n_ident == 0 && P.n_seq <= kLongestFirstMax) {
    __shared__ int seq_of_rank;
    const int r = p / P.H;
    if (tid < P.n_seq) {
      const int li = P.cu_seqlens[tid + 1] - P.cu_seqlens[tid];
      int rank = 0;
      for (int j = 0; j < P.n_seq; ++j) {
        const int lj = P.cu_seqlens[j + 1] - P.cu_seqlens[j];
        rank += (lj > li) || (lj == li && j < tid);
      }
      if (rank == r) seq_of_rank = tid;
    }
    __syncthreads();
    p = seq_of_rank * P.H + p % P.H;
  }
  Problem pr;
  if (!resolve_problem(P, p, pr)) return;
  const int H = P.H, h = pr.h, len = pr.len;
  const size_t row0 = pr.row0;
  const bool vzero = pr.ident;              // v = 0: no v tile, U^T = -Z^T G^T
  const bool write_out = P.out != nullptr;  // outputs wanted
  constexpr bool pre = PRE;
  // input side fused: group P forms k; group S forms q, and g as well when the output side is
  // fused too (group P then also runs the output epilogue), so that the two groups' chains per
  // block come out closest
  constexpr bool s_takes_q = true;
  constexpr bool s_takes_g = POST;
  const int nblocks = (len + C - 1) / C;

  if (tid == 0) {
    cta_abort = 0;
    mbar_init(&bar_in, 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_prep, 1);
    mbar_init(&bar_ext, GROUP / 32);  // one arrive per warp of group P
    mbar_init(&bar_wsfree, 1);
    mbar_init(&bar_khr, 1);
    mbar_init(&bar_D, 1);
    mbar_init(&bar_ZO, 1);
    mbar_init(&bar_G2, 1);
    mbar_init(&bar_G3, 2);  // the two issuers of the last product commit to it
    mbar_init(&bar_qg, 1);
    mbar_init(&bar_u, 1);
    fence_mbar_init();
    prefetch_tensormap(&maps.q);
    prefetch_tensormap(&maps.k);
    prefetch_tensormap(&maps.v);
    prefetch_tensormap(&maps.g);
    if constexpr (POST) prefetch_tensormap(&maps.u);
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, 512);
  if constexpr (DH == 64) {  // the second box of every input tile is the zero padding
#pragma unroll
    for (uint32_t base : {IN_K, IN_Q, IN_G, IN_V})
      for (int i = tid; i < (int)BOX_BYTES / 16; i += THREADS)
        st_shared_v4(sb + base + BOX_BYTES + 16u * (uint32_t)i, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // v is a tensor-core operand
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);  // this warp's lane quarter

  auto load2 = [&](uint32_t dst, const CUtensorMap* m, int row, uint64_t* bar) {
    tma_load_3d(sm + dst, m, 0, h, row, bar);
    if constexpr (NBOX == 2) tma_load_3d(sm + dst + BOX_BYTES, m, 64, h, row, bar);
  };
  // Waits of a whole group: the group's first warp polls the mbarrier (all its lanes, so that
  // the warp does not diverge) while the other warps sleep in the group's hardware barrier (no
  // issue slots spent spinning). Every wait of the CTA ends by one deadline, 2 s plus 50 us per
  // block (about ten times a block's normal time). Nothing branches on a wait's outcome (a
  // branch, or any use of the outcome, at the waits cost 4-8 % of the kernel's time): after a
  // wait gives up, every later wait ends at once, the groups run through their remaining blocks
  // on whatever the buffers hold (every address stays valid), and at the end a CTA that is past
  // its deadline latches KDA_ERR_TIMEOUT.
  volatile int* const abort_flag = &cta_abort;
  const uint64_t deadline = globaltimer_ns() + kWaitLimitNs + 50000ull * (uint64_t)nblocks;
  auto group_wait2 = [&](uint64_t* b1, uint32_t p1, uint64_t* b2, uint32_t p2, int id) {
    if (lt < 32) {
      mbar_wait_until(b1, p1, deadline);
      if (b2 != nullptr) mbar_wait_until(b2, p2, deadline);
    }
    named_sync(id, GROUP);
  };
  // up to three hand-offs under one group barrier (each group barrier costs the chain ~0.1 K cycles)
  auto group_wait3 = [&](uint64_t* b1, uint32_t p1, uint64_t* b2, uint32_t p2, uint64_t* b3, uint32_t p3, int id) {
    if (lt < 32) {
      if (b1 != nullptr) mbar_wait_until(b1, p1, deadline);
      if (b2 != nullptr) mbar_wait_until(b2, p2, deadline);
      mbar_wait_until(b3, p3, deadline);
    }
    named_sync(id, GROUP);
  };

  // input side fused: g = g_min sigma(e^A z + b) on thread (cg, rg)'s chunks of the staged z tile
  auto gate_rows4 = [&](int cg, int rg) {
    const float eA = expf(P.A_log[h]);
    float b8[8];
    post::load_w8(P.b_decay + (size_t)h * D + 8 * cg, b8);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4* p4 = reinterpret_cast<uint4*>(sm + IN_G + tile_chunk(cg, 4 * rg + i));
      float z[8];
      post::unpack8(*p4, z);
#pragma unroll
      for (int e = 0; e < 8; ++e) z[e] = pre::decay_gate<__nv_bfloat16>(z[e], eA, b8[e]);
      *p4 = post::pack8(z);
    }
  };

  if (isP) {
    // =====================================================================  group P
    const unsigned short* __restrict__ beta_u = static_cast<const unsigned short*>(P.beta);
    auto issue_in = [&](int b) {
      const int row = (int)(row0 + (size_t)b * C);
      mbar_arrive_expect_tx(&bar_in, 3 * NBOX * BOX_BYTES);
      load2(IN_K, &maps.k, row, &bar_in);
      load2(IN_Q, &maps.q, row, &bar_in);
      load2(IN_G, &maps.g, row, &bar_in);
      if (b + 1 < nblocks) {  // the block after it into L2, so that its load finds it there
        const CUtensorMap* mp[3] = {&maps.k, &maps.q, &maps.g};
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          tma_prefetch_3d(mp[i], 0, h, row + C);
          if constexpr (NBOX == 2) tma_prefetch_3d(mp[i], 64, h, row + C);
        }
      }
    };
    if (nblocks > 0 && lt == 0) issue_in(0);
    // beta of the next block is loaded one block ahead, kept as raw bits so that nothing waits
    // on the load until the block that needs it
    unsigned short beta_next = 0;
    if (lt < C && lt < len) beta_next = beta_u[(row0 + lt) * H + h];
    __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(P.out);
    // O of block b: TMEM -> bf16 rows [token][128] staged in XK (free: this group's A/P product
    // of the block after b has completed, and the next operands are written after the group's
    // next barrier), then, after a group barrier, 16-byte global stores, each warp writing two
    // whole 256-byte rows. The 16-byte chunks of a staged row are permuted by chunk ^ (token % 8)
    // so that the eight rows of a matrix store fall in distinct banks.
    // Warp w reads lanes (value channels) 32 (w % 4) .. + 31, columns (tokens) 32 hh .. + 31 in the
    // 16 x 256 b shape, whose registers are the m16n8 fragment that a transposed matrix store
    // writes as [token][channel] rows.
    uint8_t* stg = sm + XK;
    const uint32_t stg_s = sb + XK;
    auto stage_o = [&](int b) {
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {  // lanes 32 q + 16 sl .. + 15
        uint32_t v[16];
        const int cb = 32 * quarter + 16 * sl;  // first channel of the slab
        tmem_ld_16x256b_x4(tmem + ((uint32_t)cb << 16) + t_ot_of(b) + 32 * hh, v);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          // matrix i: channels cb + 8 (i & 1) .., tokens 32 hh + 8 (2u + (i >> 1)) ..
          const int li = lane >> 3, lj = lane & 7;
          const int tok = 32 * hh + 8 * (2 * u + (li >> 1)) + lj;
          const int chunk = ((cb + 8 * (li & 1)) >> 3) ^ (tok & 7);
          const int k0 = 2 * u, k1 = 2 * u + 1;
          stsm_x4_trans(stg_s + (uint32_t)(tok * 256 + 16 * chunk),
                        pack_bf16(__uint_as_float(v[4 * k0]), __uint_as_float(v[4 * k0 + 1])),
                        pack_bf16(__uint_as_float(v[4 * k0 + 2]), __uint_as_float(v[4 * k0 + 3])),
                        pack_bf16(__uint_as_float(v[4 * k1]), __uint_as_float(v[4 * k1 + 1])),
                        pack_bf16(__uint_as_float(v[4 * k1 + 2]), __uint_as_float(v[4 * k1 + 3])));
        }
      }
      tc_fence_before();
    };
    // after a group barrier that follows stage_o(b). With an output gate, each row of 128
    // channels (16 lanes of a half-warp, 8 channels each) is normalised and gated on its way out:
    // y = o~ / sqrt(mean(o~^2) + eps) * w * sigma(u), the mean by a 16-lane reduction.
    constexpr bool gated = POST;
    // The gate rows u of block b come by TMA into XQ (the q-side X panel, free from the completion
    // of the A/P product that read it until the next block's operands are written), issued as
    // soon as that product completes; the rows of the block after it go into L2 meanwhile.
    auto issue_u = [&](int b, uint32_t dst) {
      const int row = (int)(row0 + (size_t)b * C);
      mbar_arrive_expect_tx(&bar_u, NBOX * BOX_BYTES);
      load2(dst, &maps.u, row, &bar_u);
      if (b + 1 < nblocks) {
        tma_prefetch_3d(&maps.u, 0, h, row + C);
        tma_prefetch_3d(&maps.u, 64, h, row + C);
      }
    };
    auto store_o = [&](int b, uint32_t ubase) {
      const int tb = b * C;
      const int nb = min(C, len - tb);
      const int q = lt & 15;  // 16-byte chunk of a row; rows lt / 16 + 16 i
      const size_t off = ((row0 + tb + (lt >> 4)) * H + h) * D + 8 * q;
      __nv_bfloat16* ob = out + off;
      if constexpr (DH == 64) {  // the first 8 chunks of each row: chunk lt % 8 of rows lt / 8 + 32 i
        const int q8 = lt & 7;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = (lt >> 3) + 32 * i;
          if (r < nb)
            *reinterpret_cast<uint4*>(out + ((row0 + tb + r) * H + h) * DH + 8 * q8) =
                *reinterpret_cast<const uint4*>(stg + r * 256 + 16 * (q8 ^ (r & 7)));
        }
      } else if constexpr (gated) {  // u from the tile at ubase, after bar_u
        float w8[8];
        post::load_w8(P.norm_w + 8 * q, w8);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = (lt >> 4) + 16 * i;
          float x[8], u8[8];
          post::unpack8(*reinterpret_cast<const uint4*>(stg + r * 256 + 16 * (q ^ (r & 7))), x);
          post::unpack8(*reinterpret_cast<const uint4*>(sm + ubase + tile_chunk(q, r)), u8);
          post::gate_chunk(x, u8, w8, P.norm_eps, D);
          if (r < nb) *reinterpret_cast<uint4*>(ob + (size_t)(16 * i) * H * D) = post::pack8(x);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = (lt >> 4) + 16 * i;
          if (r < nb)
            *reinterpret_cast<uint4*>(ob + (size_t)(16 * i) * H * D) =
                *reinterpret_cast<const uint4*>(stg + r * 256 + 16 * (q ^ (r & 7)));
        }
      }
    };

    for (int blk = 0; blk < nblocks; ++blk) {
      const int t0 = blk * C;
      const int n = min(C, len - t0);
      const int par = blk & 1;
      // S has started the previous block (its first product read (K/Q e^Gamma)^T and the
      // per-parity arrays of two blocks ago are no longer read), the previous A/P product has
      // released X and Y, and this block's k, q, g tiles have landed: one wait for the three.
      // (beta of this block is first read after the operand phase's group barrier.)
      group_wait3(blk > 0 ? &bar_ZO : nullptr, (blk - 1) & 1, blk > 0 ? &bar_D : nullptr, (blk - 1) & 1,
                  &bar_in, blk & 1, BAR_P);
      if (lt < C) {
        beta_s[par][lt] = __uint_as_float((uint32_t)beta_next << 16);  // zero past the end
        beta_next = 0;
        if (lt < len - t0 - C) beta_next = beta_u[(row0 + t0 + C + lt) * H + h];
      }
      if constexpr (pre) {
        // ---------------- input side: k = L2Norm(ShortConv(k~)) in place in the staged tile (and
        // g = g_min sigma(e^A z + b) unless group S forms it), thread (cg, rg): channels 8 cg .. + 7
        // of rows 4 rg .. + 3; group S forms q meanwhile (bar_qg). Every raw row is read before any
        // is written. The last three raw rows of k~ (and
        // of q~, group S) wait for the next block in the padding columns 64..71 of WS, which no other
        // step touches: 16-byte chunk ((tensor * 3 + row) * 16 + cg) at WS row chunk / 2, byte
        // 256 + 16 (chunk % 2).
        const int cg = lt & 15, rg = lt >> 4;
        const int first_pos = pr.pos0 + t0;
#pragma unroll
        for (int ts = 0; ts < (s_takes_q ? 1 : 2); ++ts) {  // k (and q), one tensor at a time
          auto halo = [&](int hr) {
            const int chunk = (ts * 3 + hr) * 16 + cg;
            return sm + WS + (chunk >> 1) * (WLD * 4) + 64 * 4 + (chunk & 1) * 16;
          };
          uint8_t* tile = sm + (ts ? IN_Q : IN_K);
          uint4 pk[4];
          {
            float y[4][8];
            conv_rows4(tile, ts ? P.conv_q : P.conv_k, h, cg, rg, first_pos, halo, y);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              pre::l2norm8<D, false>(y[i]);
              pk[i] = post::pack8(y[i]);
            }
          }
          if (!s_takes_g && ts == 0) gate_rows4(cg, rg);
          named_sync(BAR_P, GROUP);  // every raw row of this tile (and its stash) has been read
          if (rg == 15 && blk + 1 < nblocks) stash_rows(tile, cg, halo);
          put_rows4(tile, cg, rg, pk);
        }
        // q and g of this block from group S (the wait's group barrier also orders the k rows)
        group_wait2(&bar_qg, blk & 1, nullptr, 0, BAR_P);
      }
      // ---------------- operands: X, Y, (K e^Gamma)^T, (Q e^Gamma)^T; Khat^T kept packed
      // Warp w covers channels 16 w .. 16 w + 15 (channel group cg = 0, 1 of 8) over all 64 tokens:
      // lane (g, t) holds, for each 8-token block m, the tokens 8 m + 2 t, 8 m + 2 t + 1 of
      // channels 16 w + 8 cg + g as bf16 pairs (transposed 8 x 8 loads of the [token][channel]
      // tiles), which is the mma A-fragment layout of g^T and the row layout of the [channel]
      // [token] operands written back with matrix stores. The running sums of g inside each
      // 16-token sub-block R come from warp MMAs with a triangular matrix of ones:
      //   L_r = Gamma_r - Gamma_{16R-1} = sum_{16R <= j <= r} g_j
      // Every factor is e^{+-L} times an anchor, an exponential of a sum of g over whole
      // sub-blocks (two exponentials per element). Where an anchor may underflow it is <= 1 and
      // multiplies a factor <= 1, so a product flushes to zero only when its own value is below
      // the fp32 range.
      uint32_t kh[2][8];  // Khat^T: [channel group][8-token block], bf16 pairs
      {
        // first channel of this warp; with DH = 64 warps w and w + 4 take the same 16 channels,
        // tokens 0..31 and 32..63 (hf = w / 4)
        const int cw = 16 * (DH == 64 ? (warp & 3) : warp);
        const int hf_only = DH == 64 ? (warp >> 2) : -1;
        const uint32_t boxo = (uint32_t)(cw >> 6) * BOX_BYTES, cin = (uint32_t)(cw & 63);
        const int lr = lane & 7, li = lane >> 3;  // row and matrix of this lane's matrix address
        auto live = [&](int m) -> uint32_t {      // keeps the tokens of block m that exist
          const int r = 8 * m + 2 * t;
          return (r < n ? 0x0000FFFFu : 0u) | (r + 1 < n ? 0xFFFF0000u : 0u);
        };
        // g^T as A fragments of k step R: {cg 0 | cg 1} x {tokens 16R .. +7 | 16R + 8 .. +15}
        uint32_t ga[4][4];
#pragma unroll
        for (int R = 0; R < 4; ++R) {
          ldsm_x4_trans(sb + IN_G + boxo + sw128_off(16 * R + 8 * (li >> 1) + lr, cin + 8 * (li & 1)), ga[R]);
#pragma unroll
          for (int i = 0; i < 4; ++i) ga[R][i] &= live(2 * R + (i >> 1));
        }
        // Lr[R][e]: tokens 16 R + 8 e + 2t (+1) of channel groups 0 (regs 0, 1) and 1 (regs 2, 3),
        // from U_e[j][r] = 1 if j <= 8 e + r (j: token in the sub-block, r: token in the 8-block)
        const uint32_t tri = ((2 * t <= g) ? 0x3F80u : 0u) | ((2 * t + 1 <= g) ? 0x3F800000u : 0u);
        float Lr[4][2][4];
#pragma unroll
        for (int R = 0; R < 4; ++R)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t bu[2] = {e ? 0x3F803F80u : tri, e ? tri : 0u};
            Lr[R][e][0] = Lr[R][e][1] = Lr[R][e][2] = Lr[R][e][3] = 0.f;
            mma_bf16_16816(Lr[R][e], ga[R], bu);
          }
        // sub-block sums (log2 units): token 16 R + 15 is held by lane t = 3
        float sg[2][4];
#pragma unroll
        for (int R = 0; R < 4; ++R)
#pragma unroll
          for (int cg = 0; cg < 2; ++cg)
            sg[cg][R] = __shfl_sync(0xffffffffu, Lr[R][1][2 * cg + 1], (lane & ~3) | 3) * LOG2E;
        if (t == 0 && (DH == 128 || warp < 4)) {  // e^{Gamma_L} per key channel for the state decay
#pragma unroll
          for (int cg = 0; cg < 2; ++cg)
            gl_s[par][cw + 8 * cg + g] = ex2(sg[cg][0] + sg[cg][1] + sg[cg][2] + sg[cg][3]);
        }
#pragma unroll
        for (int cg = 0; cg < 2; ++cg) {
          // e^{s_R} (<= 1) per sub-block, and e^{-s_R} where a sub-block ends at its reference;
          // every anchor is a product of these
          const float e0 = ex2(sg[cg][0]), e1 = ex2(sg[cg][1]), e2 = ex2(sg[cg][2]), e3 = ex2(sg[cg][3]);
          const float f0 = ex2(-sg[cg][0]), f2 = ex2(-sg[cg][2]);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {  // tokens 32 hf .. 32 hf + 31: sub-blocks 2 hf, 2 hf + 1
            if (DH == 64 && hf != hf_only) continue;
            uint32_t kw[4], qw[4];
            const uint32_t lo = boxo + sw128_off(32 * hf + 8 * li + lr, cin + 8 * cg);
            ldsm_x4_trans(sb + IN_K + lo, kw);
            ldsm_x4_trans(sb + IN_Q + lo, qw);
            uint32_t oxk[4], oxq[4], oy[4], oyb[4], okg[4], oqg[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int m = 4 * hf + i, R = m >> 1, e = m & 1;
              const bool odd = R & 1;  // sub-block starts right after its reference (else ends at it)
              const uint32_t lv = live(m);
              kw[i] &= lv;
              qw[i] &= lv;
              // anchors e^{Gamma_{16R-1}}, e^{Gamma_L - Gamma_{16R+15}}, e^{rho_B - Gamma_{16R+15}},
              // e^{+-(Gamma_{16R+15} - Gamma_{16R-1})}
              const float eb = R == 0 ? 1.f : (R == 1 ? e0 : (R == 2 ? e0 * e1 : e0 * e1 * e2));
              const float ea = R == 0 ? e1 * e2 * e3 : (R == 1 ? e2 * e3 : (R == 2 ? e3 : 1.f));
              const float es = R == 0 ? e0 : (R == 1 ? e1 : (R == 2 ? e2 : e3));
              const float ef = R == 0 ? f0 : (R == 2 ? f2 : 1.f);
              const float L0 = Lr[R][e][2 * cg] * LOG2E, L1 = Lr[R][e][2 * cg + 1] * LOG2E;
              const float2 u = make_float2(ex2(L0), ex2(L1));
              const float2 wv = make_float2(ex2(-L0), ex2(-L1));
              const float2 sfx = mul2(make_float2(es, es), wv);  // e^{Gamma_{16R+15} - Gamma}
              const float2 F = mul2(make_float2(ef, ef), u);     // e^{Gamma - rho}
              const float2 Fi = odd ? wv : sfx;                  // e^{rho - Gamma}
              const float2 eG = mul2(make_float2(eb, eb), u);    // e^{Gamma}
              const float2 eH = mul2(make_float2(ea, ea), sfx);  // e^{Gamma_L - Gamma}
              // the factors to bf16 pairs, then products with the bf16 k / q pairs as loaded
              const uint32_t Fb = pack_bf16(F.x, F.y), Fib = pack_bf16(Fi.x, Fi.y);
              const uint32_t eGb = pack_bf16(eG.x, eG.y), eHb = pack_bf16(eH.x, eH.y);
              oxk[i] = mul_bf16x2(kw[i], Fb);
              oxq[i] = mul_bf16x2(qw[i], Fb);
              oy[i] = mul_bf16x2(kw[i], Fib);
              okg[i] = mul_bf16x2(kw[i], eGb);
              oqg[i] = mul_bf16x2(qw[i], eGb);
              kh[cg][m] = mul_bf16x2(kw[i], eHb);
              if (hf == 0) {
                const float et = R == 0 ? e1 * e2 : e2;
                const float2 eY = mul2(make_float2(et, et), sfx);  // e^{rho_B - Gamma}
                oyb[i] = mul_bf16x2(kw[i], pack_bf16(eY.x, eY.y));
              }
            }
            // rows: channel cw + 8 cg + lr; 16-byte chunk: 8-token block 4 hf + li
            const uint32_t so = sw128_off((uint32_t)(cw + 8 * cg + lr), (uint32_t)(8 * (4 * hf + li)));
            stsm_x4(sb + XK + so, oxk[0], oxk[1], oxk[2], oxk[3]);
            stsm_x4(sb + XQ + so, oxq[0], oxq[1], oxq[2], oxq[3]);
            stsm_x4(sb + KQ + (par ? 0u : 16384u) + so, okg[0], okg[1], okg[2], okg[3]);
            stsm_x4(sb + KQ + (par ? 16384u : 0u) + so, oqg[0], oqg[1], oqg[2], oqg[3]);
            if (hf == 0) {
              stsm_x4(sb + YP + 16384u + so, oy[0], oy[1], oy[2], oy[3]);  // Y_A (panel 1)
              stsm_x4(sb + YP + so, oyb[0], oyb[1], oyb[2], oyb[3]);       // Y_B (panel 0)
            } else {
              stsm_x4(sb + YP + so, oy[0], oy[1], oy[2], oy[3]);  // Y_B (e^{rho - Gamma} = e^{rho_B - Gamma})
            }
          }
        }
      }
      // X, Y and (K/Q e^Gamma)^T are in place: release them and start the A/P product
      fence_proxy_async_smem();
      named_sync(BAR_P, GROUP);
      if (lt == 0) {
        // ---------------- tcgen05: D = X [Y_B | Y_A]^T (M 128, N 96, K 128); this group read the
        // previous block's D out already. Issued before the operands are released, so that it
        // enters the tensor pipe ahead of the state group's first product.
        tc_fence_after();
        const uint32_t id_d = idesc_bf16(128, 96, 1, 1, 0);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk)  // K = the real key channels
          umma_bf16(tmem + T_D, desc_sw128(sb + XK + 2048u * kk, 16384, 1024),
                    desc_sw128(sb + YP + 2048u * kk, 16384, 1024), id_d, kk > 0);
        umma_commit(&bar_D);
        mbar_arrive(&bar_prep);
        if (blk + 1 < nblocks) issue_in(blk + 1);  // the k, q and g tiles are dead
      }
      // A goes into WS once S has read the previous block's A out of it
      group_wait2(&bar_D, blk & 1, blk > 0 ? &bar_wsfree : nullptr, (blk - 1) & 1, BAR_P);
      tc_fence_after();
      if constexpr (gated) {  // XQ is free now: the previous block's gate rows
        if (lt == 0 && blk > 0 && write_out) issue_u(blk - 1, XQ);
      }
      // ---------------- A (fp32, into WS) and P (bf16, into PT) out of TMEM
      // Lane m: rows 0..63 are the k side (A), 64..127 the q side (P); row r = m & 63 reads the
      // Y_A columns in the first half of the block, the Y_B columns in the second (warp-uniform).
      // This thread covers columns j in [32 hh, +32).
      {
        float* ws = reinterpret_cast<float*>(sm + WS);
        const int r = c & 63;
        const bool pside = c >= 64;
        const bool firsthalf = (quarter & 1) == 0;
        const float b = beta_s[par][r];
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const int j0 = 32 * hh + 16 * part;  // columns j0 .. j0 + 15
          float vals[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) vals[j] = 0.f;
          if (!firsthalf || hh == 0) {  // the first half has columns j < 32 only
            uint32_t v[16];
            tmem_ld16(tl + T_D + (uint32_t)(firsthalf ? Y_A + 16 * part : j0), v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) vals[j] = __uint_as_float(v[j]);
          }
          if (!pside) {
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              float4 x;
              const int j = j0 + 4 * j4;
              x.x = (j < r) ? b * vals[4 * j4] : 0.f;
              x.y = (j + 1 < r) ? b * vals[4 * j4 + 1] : 0.f;
              x.z = (j + 2 < r) ? b * vals[4 * j4 + 2] : 0.f;
              x.w = (j + 3 < r) ? b * vals[4 * j4 + 3] : 0.f;
              *reinterpret_cast<float4*>(ws + r * WLD + j) = x;
            }
          } else {
#pragma unroll
            for (int j8 = 0; j8 < 2; ++j8) {
              float x[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int j = j0 + 8 * j8 + e;
                x[e] = (j <= r) ? vals[8 * j8 + e] : 0.f;
              }
              st_pack8(sb + PT + 8192u * (uint32_t)par + sw128_off(r, j0 + 8 * j8), x);
            }
          }
        }
      }
      fence_proxy_async_smem();  // P is a tensor-core operand of S's last product
      named_sync(BAR_P, GROUP);
      // ---------------- first step of the solve of T = (I + A)^{-1}, which needs A only: the
      // 16 x 16 diagonal inverses T_RR (fp32, rounded to tf32 into trr; the state group reads trr
      // from bar_ext until it releases WS), and the blocks of A that the state group uses as MMA
      // A operands rounded to tf32 in place
      {
        float* ws = reinterpret_cast<float*>(sm + WS);
        if (lt >= GROUP - 64) {
          // thread (Rd, jj) of the last two warps solves (I + A_RR) x = e_jj by column sweeps
          // (x_i -= A_im x_m for i > m), one fma per step on the chain through x
          const int q = lt - (GROUP - 64), Rd = q >> 4, jj = q & 15;
          const float* ab = ws + 16 * Rd * (WLD + 1);
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = i == jj ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < 15; ++m)
#pragma unroll
            for (int i = m + 1; i < 16; ++i) x[i] = fmaf(-ab[i * WLD + m], x[m], x[i]);
#pragma unroll
          for (int i = 0; i < 16; ++i) trr[Rd][i][jj] = tf32r(x[i]);
        } else {
          // A_10, A_32 and rows 32..63 x columns 0..31: 384 float4, two per thread
#pragma unroll
          for (int e = lt; e < 384; e += GROUP - 64) {
            int row, col;
            if (e < 128) {  // e < 64: A_10 (rows 16..31, columns 0..15); else A_32 (48.., 32..)
              row = 16 + 32 * (e >> 6) + ((e & 63) >> 2);
              col = 32 * (e >> 6) + 4 * (e & 3);
            } else {
              row = 32 + ((e - 128) >> 3);
              col = 4 * ((e - 128) & 7);
            }
            float4* pa = reinterpret_cast<float4*>(ws + row * WLD + col);
            float4 v4 = *pa;
            v4.x = tf32r(v4.x); v4.y = tf32r(v4.y); v4.z = tf32r(v4.z); v4.w = tf32r(v4.w);
            *pa = v4;
          }
        }
      }
      // each warp hands its part to group S as it finishes (no group barrier on this chain:
      // nothing below reads WS or trr before the next block's bar_wsfree)
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ext);
      // ---------------- once S's last product of the previous block is complete: Khat^T of this
      // block (that product read the previous one) and the previous block's O
      if (blk > 0) {
        group_wait2(&bar_G3, (blk - 1) & 1, (gated && write_out) ? &bar_u : nullptr, (blk - 1) & 1, BAR_P);
        tc_fence_after();
      }
#pragma unroll
      for (int cg = 0; cg < 2; ++cg)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (DH == 64 && hf != (warp >> 2)) continue;  // the other warp of the pair holds it
          const int cw = 16 * (DH == 64 ? (warp & 3) : warp);
          stsm_x4(sb + KH + sw128_off((uint32_t)(cw + 8 * cg + (lane & 7)), (uint32_t)(8 * (4 * hf + (lane >> 3)))),
                  kh[cg][4 * hf], kh[cg][4 * hf + 1], kh[cg][4 * hf + 2], kh[cg][4 * hf + 3]);
        }
      fence_proxy_async_smem();
      if (blk > 0 && write_out) stage_o(blk - 1);
      named_sync(BAR_P, GROUP);
      // Khat^T is stored and the previous block's O is out of TMEM; its global stores follow (the
      // release of this arrive does not wait for them)
      if (lt == 0) mbar_arrive(&bar_khr);
      if (blk > 0 && write_out) store_o(blk - 1, XQ);
    }
    if (nblocks > 0) {  // the last block's O (its gate rows into the k tile, which no one reads
      // any more, while XQ may still be read for the block before it)
      if (gated && write_out && lt == 0) issue_u(nblocks - 1, IN_K);
      group_wait2(&bar_G3, (nblocks - 1) & 1, (gated && write_out) ? &bar_u : nullptr,
                  (nblocks - 1) & 1, BAR_P);
      tc_fence_after();
      if (write_out) {
        stage_o(nblocks - 1);
        named_sync(BAR_P, GROUP);
        store_o(nblocks - 1, IN_K);
      }
    }
  } else {
    // =====================================================================  group S
    const bool leader = lt == 0;
    auto issue_v = [&](int b) {
      mbar_arrive_expect_tx(&bar_v, NBOX * BOX_BYTES);
      load2(IN_V, &maps.v, (int)(row0 + (size_t)b * C), &bar_v);
      if (b + 1 < nblocks) {  // the next v tile into L2
        tma_prefetch_3d(&maps.v, 0, h, (int)(row0 + (size_t)(b + 1) * C));
        if constexpr (NBOX == 2) tma_prefetch_3d(&maps.v, 64, h, (int)(row0 + (size_t)(b + 1) * C));
      }
    };
    // ---- initial state S^T: lane v = c, key channels 64 hh .. 64 hh + 63 (coalesced over v);
    // with DH = 64 only key and value channels below 64 exist, the rest is the zero padding
    {
      const bool real = DH == 128 || (c < DH && hh == 0);
      const float* s0 = (P.S0 && !pr.ident && real) ? P.S0 + (size_t)pr.s0 * DH * DH + c : nullptr;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[32], sbf[16];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int cc = 64 * hh + 32 * half + j;  // key channel
          sv[j] = s0 ? __float_as_uint(s0[(size_t)cc * DH])
                     : ((pr.ident && real && cc == c) ? 0x3F800000u : 0u);
        }
        tmem_st32(tl + T_ST + 64 * hh + 32 * half, sv);
#pragma unroll
        for (int j = 0; j < 16; ++j) sbf[j] = pack_bf16(__uint_as_float(sv[2 * j]), __uint_as_float(sv[2 * j + 1]));
        tmem_st16(tl + T_SB + 32 * hh + 16 * half, sbf);
      }
      tmem_st_wait();
      tc_fence_before();
    }
    // input side fused: q = L2Norm(ShortConv(q~)) and g = g_min sigma(e^A z + b) of block b in
    // place in the staged tiles, once they have landed (group P forms k meanwhile); thread
    // (cg, rg) as in group P's pass, the last three raw rows of q~ stashed in the WS padding
    auto transform_qg = [&](int b) {
      group_wait2(&bar_in, b & 1, nullptr, 0, BAR_S);
      const int cg = lt & 15, rg = lt >> 4;
      if constexpr (s_takes_q) {
        auto halo = [&](int hr) {
          const int chunk = (3 + hr) * 16 + cg;
          return sm + WS + (chunk >> 1) * (WLD * 4) + 64 * 4 + (chunk & 1) * 16;
        };
        uint8_t* tile = sm + IN_Q;
        uint4 pk[4];
        {
          float y[4][8];
          conv_rows4(tile, P.conv_q, h, cg, rg, pr.pos0 + b * C, halo, y);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pre::l2norm8<D, false>(y[i]);
            pk[i] = post::pack8(y[i]);
          }
        }
        if constexpr (s_takes_g) gate_rows4(cg, rg);
        named_sync(BAR_S, GROUP);  // every raw row of the q tile (and its stash) has been read
        if (rg == 15 && b + 1 < nblocks) stash_rows(tile, cg, halo);
        put_rows4(tile, cg, rg, pk);
      } else {
        gate_rows4(cg, rg);
      }
      named_sync(BAR_S, GROUP);
      if (leader) mbar_arrive(&bar_qg);
    };
    if (nblocks > 0 && !vzero && leader) issue_v(0);
    // G is zero above the diagonal blocks; those entries are never written again
    for (int i = lt; i < 8192 / 16; i += GROUP) st_shared_v4(sb + GB + 16u * (uint32_t)i, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    named_sync(BAR_S, GROUP);
    if constexpr (pre) {
      if (nblocks > 0) transform_qg(0);
    }

    for (int blk = 0; blk < nblocks; ++blk) {
      const int t0 = blk * C;
      const int n = min(C, len - t0);
      const int par = blk & 1;
      const uint32_t ph = (uint32_t)par;
      // P's operands of this block are in place. (P has read the O of two blocks ago out of
      // TMEM, whose columns this block's O takes: bar_khr of the previous block, waited for
      // before the previous block's last product. Waiting for it again here could alias: P may
      // already have completed the next phase of bar_khr, and a parity wait would then look
      // for the phase after it.)
      group_wait2(&bar_prep, ph, nullptr, 0, BAR_S);
      tc_fence_after();
      const uint32_t t_ot = t_ot_of(blk);  // this block's O^T columns
      // ---------------- tcgen05: [O^T | Z^T] (even) or [Z^T | O^T] (odd) =
      // S^T [(Q e^Gamma)^T | (K e^Gamma)^T] (or the other order) (N 128, K 128)
      if (leader) {
        tc_fence_after();
        const uint32_t id_zo = idesc_bf16(128, 128, 0, 1, 0);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk)  // K = the real key channels
          umma_bf16_tmem_a(tmem + (par ? T_ZT : t_ot), tmem + T_SB + 8u * kk,
                           desc_sw128(sb + KQ + 2048u * kk, 16384, 1024), id_zo, kk > 0);
        umma_commit(&bar_ZO);
      }
      // ---------------- while that product runs: the solve of this block, once group P has
      // written A, P and the diagonal inverses (bar_ext)
      group_wait2(&bar_ext, ph, nullptr, 0, BAR_S);
      // ---------------- T = (I + A)^{-1} (unit lower triangular) and G = T Diag(beta) (bf16)
      // From the 16 x 16 diagonal inverses T_RR (group P, in trr) and the block-inverse identity
      // [[P, 0], [C, Q]]^{-1} = [[P^{-1}, 0], [-Q^{-1} C P^{-1}, Q^{-1}]]: the off-diagonal
      // 16 x 16 block of each 32 x 32 half and then the off-diagonal 32 x 32 block, as tf32 warp
      // MMAs on fp32 blocks in WS (T overwrites A where A is no longer read).
      {
        float* ws = reinterpret_cast<float*>(sm + WS);
        // scratch: rows 0..31, columns 32..63 of WS, where A is zero and no block of T is kept
        float* qs = ws + 32;
        const int sw = warp - GROUP / 32;  // warp index inside the group
        const float* bt = beta_s[par];
        // two adjacent entries of G = T Diag(beta): row r, columns j and j + 1 (j even)
        auto g_store = [&](int r, int j, float x0, float x1) {
          *reinterpret_cast<uint32_t*>(sm + GB + sw128_off((uint32_t)r, (uint32_t)j)) =
              pack_bf16(x0 * bt[j], x1 * bt[j + 1]);
        };
        // (2) warp (h, n) of warps 0-3, h = 32-row half, n = 8-column half: columns 8n .. 8n + 7
        //     of Y = A_10 T_00 (into qs), then of T_10 = -T_11 Y (into WS), which need no other
        //     columns of Y (h = 1: A_32, T_22, T_33, T_32); warps 4-7: the T_RR into the diagonal
        //     blocks of WS, where A_RR is no longer read, and G of the diagonal blocks
        if (sw < 4) {
          const int tile = sw >> 1, nh = sw & 1;
          float* y = qs + 16 * tile + 8 * nh;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          tile_mma(acc, ws + (16 + 32 * tile) * WLD + 32 * tile, WLD, &trr[2 * tile][0][8 * nh], TLD, 2);
          float* yo = y + 2 * t;
          yo[g * WLD] = tf32r(acc[0]);
          yo[g * WLD + 1] = tf32r(acc[1]);
          yo[(g + 8) * WLD] = tf32r(acc[2]);
          yo[(g + 8) * WLD + 1] = tf32r(acc[3]);
          __syncwarp();
          float acc2[4] = {0.f, 0.f, 0.f, 0.f};
          tile_mma(acc2, &trr[2 * tile + 1][0][0], TLD, y, WLD, 2);
          // T_10 goes over A_10, which the other warp of the tile reads whole (all 16 columns)
          named_sync(BAR_TILE0 + tile, 64);
          float* o = ws + (16 + 32 * tile) * WLD + 32 * tile + 8 * nh + 2 * t;
          o[g * WLD] = tf32r(-acc2[0]);
          o[g * WLD + 1] = tf32r(-acc2[1]);
          o[(g + 8) * WLD] = tf32r(-acc2[2]);
          o[(g + 8) * WLD + 1] = tf32r(-acc2[3]);
        } else {
          for (int e = lt - 128; e < 1024; e += 128) {
            const int R = e >> 8, i = (e >> 4) & 15, j = e & 15;
            ws[(16 * R + i) * WLD + 16 * R + j] = trr[R][i][j];
          }
          for (int e = lt - 128; e < 512; e += 128) {
            const int R = e >> 7, i = (e >> 3) & 15, jp = 2 * (e & 7);
            g_store(16 * R + i, 16 * R + jp, trr[R][i][jp], trr[R][i][jp + 1]);
          }
        }
        named_sync(BAR_S, GROUP);
        // (3) warp (n, m), n = sw & 3, m = sw >> 2: tile (m, n) of Q = A_(32)10 T_(32)00 (rows
        //     32 + 16 m .., columns 8 n .., K 32; into qs); the two warps of column block n meet
        //     at their own barrier; then tile (m, n) of G rows 32..63: T_(32)10 = -T_(32)11 Q.
        //     Every thread also writes one pair of G of T_10 and T_32.
        {
          const int nt = sw & 3, mt = sw >> 2;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          tile_mma(acc, ws + (32 + 16 * mt) * WLD, WLD, ws + 8 * nt, WLD, 4);
          float* o = qs + 16 * mt * WLD + 8 * nt + 2 * t;
          o[g * WLD] = tf32r(acc[0]);
          o[g * WLD + 1] = tf32r(acc[1]);
          o[(g + 8) * WLD] = tf32r(acc[2]);
          o[(g + 8) * WLD + 1] = tf32r(acc[3]);
          {
            const int tile = lt >> 7, i = (lt >> 3) & 15, jp = 2 * (lt & 7);
            const int r = 16 + 32 * tile + i, j = 32 * tile + jp;
            g_store(r, j, ws[r * WLD + j], ws[r * WLD + j + 1]);
          }
          named_sync(BAR_PAIR0 + nt, 64);
          float acc2[4] = {0.f, 0.f, 0.f, 0.f};
          tile_mma(acc2, ws + (32 + 16 * mt) * WLD + 32, WLD, qs + 8 * nt, WLD, 4);
          const int r = 32 + 16 * mt + g, j = 8 * nt + 2 * t;
          g_store(r, j, -acc2[0], -acc2[1]);
          g_store(r + 8, j, -acc2[2], -acc2[3]);
        }
      }
      fence_proxy_async_smem();  // G is a tensor-core operand
      if constexpr (pre) {  // the next block's q and g, which group P's operand phase waits for
        if (blk + 1 < nblocks) transform_qg(blk + 1);
      }
      // ---------------- Z^T (lane v = c, tokens 32 hh ..) -> bf16 A operand, once the product is
      // complete; the wait's group barrier also says that every thread is done with WS. The v tile
      // (issued a block ago) is waited for here too, one group barrier for both.
      group_wait2(&bar_ZO, ph, vzero ? nullptr : &bar_v, ph, BAR_S);
      if (leader) mbar_arrive(&bar_wsfree);
      tc_fence_after();
      {
        uint32_t v[32], zb[16];
        tmem_ld32(tl + T_ZT + 32 * hh, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) zb[j] = pack_bf16(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        tmem_st16(tl + T_ZB + 16 * hh, zb);
      }
      tmem_st_wait();
      tc_fence_before();
      // a group barrier orders the bf16 Z^T before the U product (the v tile has landed)
      if (!vzero) {
        named_sync(BAR_S, GROUP);
        if constexpr (pre) {  // input side: v = ShortConv(v~) in place in the staged tile (as for k above);
          // the last three raw rows wait for the next block in the padding columns 16..19 of trr
          // (16-byte chunk row * 16 + cg), which no other step touches
          const int cg = lt & 15, rg = lt >> 4;
          auto halo = [&](int hr) {
            const int chunk = hr * 16 + cg;
            return reinterpret_cast<uint8_t*>(&trr[chunk >> 4][chunk & 15][16]);
          };
          float y[4][8];
          conv_rows4(sm + IN_V, P.conv_v, h, cg, rg, pr.pos0 + t0, halo, y);
          uint4 pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) pk[i] = post::pack8(y[i]);
          named_sync(BAR_S, GROUP);  // every raw row (and the stash) has been read
          if (rg == 15 && blk + 1 < nblocks) stash_rows(sm + IN_V, cg, halo);
          put_rows4(sm + IN_V, cg, rg, pk);
          fence_proxy_async_smem();  // v is a tensor-core operand
          named_sync(BAR_S, GROUP);
        }
      } else {
        named_sync(BAR_S, GROUP);
      }
      // ---------------- tcgen05: U^T = V^T G^T - Z^T G^T (M 128, N 64, K 64), which is
      // U = T Diag(beta) (V - Z), the solution of (I + A) U = Diag(beta) (V - Z)
      if (leader) {
        tc_fence_after();
        const uint32_t id_v = idesc_bf16(128, 64, 1, 0, 0);
        const uint32_t id_z = idesc_bf16(128, 64, 0, 0, 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bg = desc_sw128(sb + GB + 32u * kk, 16, 1024);
          if (!vzero)
            umma_bf16(tmem + T_UT, desc_sw128(sb + IN_V + 2048u * kk, BOX_BYTES, 1024), bg, id_v, kk > 0);
          umma_bf16_tmem_a(tmem + T_UT, tmem + T_ZB + 8u * kk, bg, id_z, (kk > 0 || !vzero) ? 1u : 0u);
        }
        umma_commit(&bar_G2);
      }
      // ---------------- while U runs: S^T <- S^T Diag(e^{Gamma_L}) (the first product read the
      // bf16 copy; Khat^T U accumulates onto this one, after the barrier that follows U^T -> bf16).
      // The issuing thread's warp waits while its products enter the tensor pipe, so the warp of
      // the same lane quarter in the other half scales all 128 columns of those lanes.
      if (lt >= 32) {
        const bool both = lt >= 128 && lt < 160;  // lane quarter 0, second half
        // 16-column parts; with DH = 64 only key channels below 64 (and value lanes below 64) exist
        constexpr int NC = DH;  // key channels to scale
        const int np = (DH == 64 && c >= 64) ? 0 : (both ? NC / 16 : NC / 32);
        const int cb = both ? 0 : (NC / 2) * hh;
        uint32_t v[16];
#pragma unroll 1
        for (int part = 0; part < np; ++part) {
          const int c0 = cb + 16 * part;
          tmem_ld16(tl + T_ST + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 gv = *reinterpret_cast<const float4*>(&gl_s[par][c0 + j]);
            const float2 a0 = mul2(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])),
                                   make_float2(gv.x, gv.y));
            const float2 a1 = mul2(make_float2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])),
                                   make_float2(gv.z, gv.w));
            v[j] = __float_as_uint(a0.x); v[j + 1] = __float_as_uint(a0.y);
            v[j + 2] = __float_as_uint(a1.x); v[j + 3] = __float_as_uint(a1.y);
          }
          tmem_st16(tl + T_ST + c0, v);
        }
      }
      group_wait2(&bar_G2, ph, nullptr, 0, BAR_S);
      tc_fence_after();
      {  // U^T (lane v, tokens 32 hh ..) -> bf16 A operand, over Z^T bf16 (read by the product)
        uint32_t v[32], ub[16];
        tmem_ld32(tl + T_UT + 32 * hh, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) ub[j] = pack_bf16(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        tmem_st16(tl + T_UB + 16 * hh, ub);
        tmem_st_wait();
      }
      tc_fence_before();
      // ---------------- tcgen05: O^T += U^T P^T (N 64) ; S^T += U^T Khat (N 128), K 64; P has
      // stored this block's Khat^T by bar_khr. The two products have their own accumulators and
      // are issued by two threads in different warps; both commit to bar_G3.
      // (the wait's group barrier also orders every thread's U^T bf16 stores before the products)
      group_wait2(&bar_khr, ph, nullptr, 0, BAR_S);
      if (leader) {
        tc_fence_after();
        const uint32_t id_s = idesc_bf16(128, DH, 0, 0, 0);  // N = the real key channels
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a(tmem + T_ST, tmem + T_UB + 8u * kk,
                           desc_sw128(sb + KH + 32u * kk, 16, 1024), id_s, 1);
        umma_commit(&bar_G3);
      } else if (lt == 128) {
        tc_fence_after();
        const uint32_t id_o = idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a(tmem + t_ot, tmem + T_UB + 8u * kk,
                           desc_sw128(sb + PT + 8192u * (uint32_t)par + 32u * kk, 16, 1024), id_o, 1);
        umma_commit(&bar_G3);
      }
      if (blk + 1 < nblocks && !vzero && leader) issue_v(blk + 1);  // the v tile is dead (U is complete)
      group_wait2(&bar_G3, ph, nullptr, 0, BAR_S);
      tc_fence_after();
      // ---------------- bf16 copy of the new state for the next block (group P writes O)
      {
        // with DH = 64 only value lanes and key columns below 64 exist: each half copies 32
        // columns of them (the rest of the copy keeps the zeros it started with)
        constexpr int CPH = DH / 2;  // columns per half
        const int nparts = (DH == 64 && c >= 64) ? 0 : CPH / 16;
#pragma unroll 1
        for (int part = 0; part < nparts; ++part) {
          uint32_t v[16], sbf[8];
          tmem_ld16(tl + T_ST + CPH * hh + 16 * part, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j) sbf[j] = pack_bf16(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          tmem_st8(tl + T_SB + CPH / 2 * hh + 8 * part, sbf);
        }
        tmem_st_wait();
      }
      tc_fence_before();  // the next block's operand wait is the group barrier after the copy
    }
    if (pr.sf && (DH == 128 || (c < DH && hh == 0))) {  // S_final[c'][v] from S^T (lane
      // v): coalesced over v
      float* sf = pr.sf + (size_t)pr.sf_i * DH * DH + c;
      uint32_t v[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        tmem_ld32(tl + T_ST + 64 * hh + 32 * half, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) sf[(size_t)(64 * hh + 32 * half + j) * DH] = __uint_as_float(v[j]);
      }
    }
  }
  // a CTA that ran past its deadline had a wait give up: its results are not to be trusted
  if (tid == 0 && globaltimer_ns() > deadline) *abort_flag = 1;
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // the copies and products already issued land before TMEM and the CTA's memory go away:
    // each completes within microseconds
    if (tid == 0) {
      record_status(4u /* KDA_ERR_TIMEOUT */);
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
    }
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side

// The kernel works in 64-token blocks. A request for 128-token chunks is served by the same
// kernel: each chunk is two consecutive 64-token blocks, which is the same mathematics (the
// block form is exact for any block size) with fewer intra-block products.
inline bool tc_supports(int C_) { return C_ == C || C_ == 2 * C; }

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

// [rows, H, dh] bf16 token tensor (dh = 128 or 64) viewed as a 3-D map with 64 x 1 x 64 boxes,
// 128-byte swizzle.
inline bool encode_token_map(CUtensorMap* m, const void* base, long long rows, int H, int dh) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)dh, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)dh * 2, (cuuint64_t)H * dh * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

// Shapes the tensor-core kernel takes: bf16 with C = 64 or 128, and head size 128 (every mode)
// or 64 (without the input and output sides).
inline bool tc_supports(int C, int d, const SeqParams& P) {
  return tc::tc_supports(C) &&
         (d == 128 || (d == 64 && P.conv_q == nullptr && P.gate_u == nullptr));
}

inline kda_status_t launch_chunk_tc(const SeqParams& P, int n_problems, int d, cudaStream_t st,
                                    std::string& err) {
  tc::TmaMaps maps;
  memset(&maps, 0, sizeof(maps));
  const long long rows = P.cu_seqlens ? (long long)P.T : (long long)P.n_seq * P.T;
  if (!tc::encode_token_map(&maps.q, P.q, rows, P.H, d) ||
      !tc::encode_token_map(&maps.k, P.k, rows, P.H, d) ||
      !tc::encode_token_map(&maps.v, P.v, rows, P.H, d) ||
      !tc::encode_token_map(&maps.g, P.g, rows, P.H, d) ||
      (P.gate_u != nullptr && !tc::encode_token_map(&maps.u, P.gate_u, rows, P.H, d))) {
    err = "cuTensorMapEncodeTiled failed";
    return KDA_ERR_CUDA;
  }
  const bool pre = P.conv_q != nullptr, post = P.gate_u != nullptr;
  auto kern = d == 64 ? tc::chunk_tc_kernel<false, false, 64>
              : pre   ? (post ? tc::chunk_tc_kernel<true, true> : tc::chunk_tc_kernel<true, false>)
                      : (post ? tc::chunk_tc_kernel<false, true> : tc::chunk_tc_kernel<false, false>);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)tc::SMEM_ALLOC);
  if (e != cudaSuccess) {
    err = std::string("cudaFuncSetAttribute(chunk_tc): ") + cudaGetErrorString(e);
    return KDA_ERR_CUDA;
  }
  kern<<<n_problems, tc::THREADS, tc::SMEM_ALLOC, st>>>(maps, P);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("chunk_tc launch: ") + cudaGetErrorString(e);
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

}  // namespace kda
