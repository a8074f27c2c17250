// C ABI of the KDA forward library: argument validation, kernel selection and launches.
// Declarations and the full contract are in include/kda.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/kda.h"
#include "kda_chunk_simt.cuh"
#include "kda_chunk_tc.cuh"
#include "kda_common.cuh"
#include "kda_decode.cuh"
#include "kda_post.cuh"
#include "kda_pre.cuh"
#include "kda_scan.cuh"
#include "kda_selftest.cuh"

namespace {

thread_local std::string t_last_error;

kda_status_t fail(kda_status_t st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kda_status_t fail(kda_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

kda_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(KDA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status_t check_ptr(const void* p, const char* name, bool required) {
  if (p == nullptr) {
    if (required) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", name);
    return KDA_OK;
  }
  if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return KDA_OK;
}

kda_status_t check_common(int H, int d_k, int d_v, kda_dtype_t dtype) {
  if (H < 1) return fail(KDA_ERR_INVALID_ARG, "H must be >= 1 (got %d)", H);
  if (d_k < 1 || d_v < 1) return fail(KDA_ERR_INVALID_ARG, "d_k, d_v must be >= 1");
  if (dtype != KDA_DTYPE_F32 && dtype != KDA_DTYPE_BF16)
    return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (!(d_k == d_v && (d_k == 64 || d_k == 128)))
    return fail(KDA_ERR_UNSUPPORTED, "supported head sizes: d_k = d_v in {64, 128} (got %d, %d)",
                d_k, d_v);
  return KDA_OK;
}

template <typename TIn, int D>
kda_status_t launch_simt(const kda::SeqParams& P, int n_problems, int C, cudaStream_t st) {
  constexpr int THREADS = 256;
  cudaError_t e;
  if (C == 16) {
    using SM = kda::SimtSmem<D, D, 16>;
    auto kern = kda::chunk_simt_kernel<TIn, D, D, 16, THREADS>;
    e = kda::ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)SM::bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(chunk_simt)");
    kern<<<n_problems, THREADS, SM::bytes, st>>>(P);
  } else {
    using SM = kda::SimtSmem<D, D, 32>;
    auto kern = kda::chunk_simt_kernel<TIn, D, D, 32, THREADS>;
    e = kda::ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)SM::bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(chunk_simt)");
    kern<<<n_problems, THREADS, SM::bytes, st>>>(P);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "chunk_simt launch");
  return KDA_OK;
}

kda_status_t run_chunk(const kda::SeqParams& P, int n_problems, int d, int C, kda_dtype_t dtype,
                       cudaStream_t st) {
  if (n_problems == 0) return KDA_OK;
  if (dtype == KDA_DTYPE_BF16 && kda::tc_supports(C, d, P))
    return kda::launch_chunk_tc(P, n_problems, d, st, t_last_error);
  if (dtype == KDA_DTYPE_F32)
    return d == 128 ? launch_simt<float, 128>(P, n_problems, C, st)
                    : launch_simt<float, 64>(P, n_problems, C, st);
  return d == 128 ? launch_simt<__nv_bfloat16, 128>(P, n_problems, C, st)
                  : launch_simt<__nv_bfloat16, 64>(P, n_problems, C, st);
}

// Launches the scan of segment transitions (see kda_scan.cuh).
kda_status_t launch_scan(const float* M, const float* St, const float* S0, float* S_in, int n_seg,
                         int BH, int d, int d_v, cudaStream_t st) {
  (void)d_v;
  dim3 grid(BH, d / (d == 128 ? kda::scan::ScanSmem<128>::NC : kda::scan::ScanSmem<64>::NC));
  cudaError_t e;
  if (d == 128) {
    auto kern = kda::scan::segment_scan_kernel<128, 128>;
    const int bytes = (int)kda::scan::ScanSmem<128>::bytes;
    e = kda::ensure_smem_limit(reinterpret_cast<const void*>(kern), bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(segment_scan)");
    kern<<<grid, kda::scan::THREADS, bytes, st>>>(M, St, S0, S_in, n_seg, BH);
  } else {
    auto kern = kda::scan::segment_scan_kernel<64, 64>;
    const int bytes = (int)kda::scan::ScanSmem<64>::bytes;
    e = kda::ensure_smem_limit(reinterpret_cast<const void*>(kern), bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(segment_scan)");
    kern<<<grid, kda::scan::THREADS, bytes, st>>>(M, St, S0, S_in, n_seg, BH);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "segment_scan launch");
  return KDA_OK;
}

// Launches the standalone output gate over n_rows rows of d_v channels (y may alias o).
kda_status_t launch_output_gate(const void* o, const void* u, const float* w, float eps, void* y,
                                long long n_rows, int d_v, kda_dtype_t dtype, cudaStream_t st) {
  if (n_rows == 0) return KDA_OK;
  using bf = __nv_bfloat16;
  if (d_v == 128) {
    const unsigned grid = (unsigned)((n_rows + 15) / 16);
    if (dtype == KDA_DTYPE_BF16)
      kda::post::output_gate_kernel<bf><<<grid, 256, 0, st>>>((const bf*)o, (const bf*)u, w, eps,
                                                              (bf*)y, n_rows);
    else
      kda::post::output_gate_kernel<float><<<grid, 256, 0, st>>>((const float*)o, (const float*)u,
                                                                 w, eps, (float*)y, n_rows);
  } else {
    const unsigned grid = (unsigned)((n_rows + 31) / 32);
    if (dtype == KDA_DTYPE_BF16)
      kda::post::output_gate64_kernel<bf><<<grid, 256, 0, st>>>((const bf*)o, (const bf*)u, w, eps,
                                                                (bf*)y, n_rows);
    else
      kda::post::output_gate64_kernel<float><<<grid, 256, 0, st>>>(
          (const float*)o, (const float*)u, w, eps, (float*)y, n_rows);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "output_gate launch");
  return KDA_OK;
}

// Tokens per segment when T is split into (at most) n_seg segments of whole 64-token blocks.
long long segment_tokens(int T, int n_seg) {
  const long long blocks = ((long long)T + 63) / 64;
  return ((blocks + n_seg - 1) / n_seg) * 64;
}

}  // namespace

extern "C" {

kda_status_t kda_chunk_fwd(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, const float* S0, void* out, float* S_final, int B,
                           int H, int T, int d_k, int d_v, int C, kda_dtype_t dtype,
                           void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d_k, d_v, dtype);
  if (s != KDA_OK) return s;
  if (B < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "B and T must be >= 0 (got %d, %d)", B, T);
  if (!(C == 16 || C == 32 || C == 64 || C == 128))
    return fail(KDA_ERR_UNSUPPORTED, "C must be 16, 32, 64 or 128 (got %d)", C);
  if ((long long)B * T * H * d_k >= (1ll << 40) || (long long)B * H >= (1ll << 31) ||
      (long long)B * T >= (1ll << 31))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  const bool tokens = (long long)B * T > 0;
  if ((s = check_ptr(q, "q", tokens)) || (s = check_ptr(k, "k", tokens)) ||
      (s = check_ptr(v, "v", tokens)) || (s = check_ptr(g, "g", tokens)) ||
      (s = check_ptr(beta, "beta", false)) || (s = check_ptr(out, "out", tokens)) ||
      (s = check_ptr(S0, "S0", false)) || (s = check_ptr(S_final, "S_final", false)))
    return s;
  if (tokens && beta == nullptr) return fail(KDA_ERR_INVALID_ARG, "beta is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  kda::SeqParams P{q, k, v, g, beta, S0, out, S_final, nullptr, B, H, T};
  return run_chunk(P, B * H, d_k, C, dtype, st);
}

kda_status_t kda_chunk_fwd_varlen(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* S0, void* out, float* S_final,
                                  const int32_t* cu_seqlens, int N, int H, int T_total, int d_k,
                                  int d_v, int C, kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d_k, d_v, dtype);
  if (s != KDA_OK) return s;
  if (N < 0 || T_total < 0)
    return fail(KDA_ERR_INVALID_ARG, "N and T_total must be >= 0 (got %d, %d)", N, T_total);
  if (!(C == 16 || C == 32 || C == 64 || C == 128))
    return fail(KDA_ERR_UNSUPPORTED, "C must be 16, 32, 64 or 128 (got %d)", C);
  if ((long long)T_total * H * d_k >= (1ll << 40) || (long long)N * H >= (1ll << 31) ||
      N >= (1 << 30))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if (cu_seqlens == nullptr) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is not 4-byte aligned");
  const bool tokens = T_total > 0;
  if ((s = check_ptr(q, "q", tokens)) || (s = check_ptr(k, "k", tokens)) ||
      (s = check_ptr(v, "v", tokens)) || (s = check_ptr(g, "g", tokens)) ||
      (s = check_ptr(beta, "beta", false)) || (s = check_ptr(out, "out", tokens)) ||
      (s = check_ptr(S0, "S0", false)) || (s = check_ptr(S_final, "S_final", false)))
    return s;
  if (tokens && beta == nullptr) return fail(KDA_ERR_INVALID_ARG, "beta is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  kda::SeqParams P{q, k, v, g, beta, S0, out, S_final, cu_seqlens, N, H, T_total};
  return run_chunk(P, N * H, d_k, C, dtype, st);
}

kda_status_t kda_recurrent_step(const void* q, const void* k, const void* v, const void* g,
                                const void* beta, float* S, void* out, int N, int H, int d_k,
                                int d_v, kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d_k, d_v, dtype);
  if (s != KDA_OK) return s;
  if (N < 0) return fail(KDA_ERR_INVALID_ARG, "N must be >= 0 (got %d)", N);
  if (N == 0) return KDA_OK;
  if ((long long)N * H >= (1ll << 31)) return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if ((s = check_ptr(q, "q", true)) || (s = check_ptr(k, "k", true)) ||
      (s = check_ptr(v, "v", true)) || (s = check_ptr(g, "g", true)) ||
      (s = check_ptr(beta, "beta", false)) || (s = check_ptr(S, "S", true)) ||
      (s = check_ptr(out, "out", true)))
    return s;
  if (beta == nullptr) return fail(KDA_ERR_INVALID_ARG, "beta is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = N * H;
  if (dtype == KDA_DTYPE_F32) {
    const float *qq = (const float*)q, *kk = (const float*)k, *vv = (const float*)v,
                *gg = (const float*)g, *bb = (const float*)beta;
    if (d_k == 128)
      kda::decode_step_kernel<float, 128, 128, 256><<<grid, 256, 0, st>>>(qq, kk, vv, gg, bb, S,
                                                                          (float*)out);
    else
      kda::decode_step_kernel<float, 64, 64, 128><<<grid, 128, 0, st>>>(qq, kk, vv, gg, bb, S,
                                                                        (float*)out);
  } else {
    using bf = __nv_bfloat16;
    const bf *qq = (const bf*)q, *kk = (const bf*)k, *vv = (const bf*)v, *gg = (const bf*)g,
             *bb = (const bf*)beta;
    if (d_k == 128)
      kda::decode_step_kernel<bf, 128, 128, 256><<<grid, 256, 0, st>>>(qq, kk, vv, gg, bb, S,
                                                                       (bf*)out);
    else
      kda::decode_step_kernel<bf, 64, 64, 128><<<grid, 128, 0, st>>>(qq, kk, vv, gg, bb, S,
                                                                     (bf*)out);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_step launch");
  return KDA_OK;
}

kda_status_t kda_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* g,
                                 const void* beta, const float* S0, const void* gate_u,
                                 const float* norm_w, float norm_eps, void* out, float* S_final,
                                 const int32_t* cu_seqlens, int n_seq, int H, int T, int d_k,
                                 int d_v, int C, kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d_k, d_v, dtype);
  if (s != KDA_OK) return s;
  if (n_seq < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "n_seq and T must be >= 0 (got %d, %d)", n_seq, T);
  if (!(C == 16 || C == 32 || C == 64 || C == 128))
    return fail(KDA_ERR_UNSUPPORTED, "C must be 16, 32, 64 or 128 (got %d)", C);
  if (!(norm_eps >= 0.f) || !(norm_eps < 1e30f))
    return fail(KDA_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
  const bool packed = cu_seqlens != nullptr;
  const long long rows = packed ? (long long)T : (long long)n_seq * T;
  if (rows * H * d_k >= (1ll << 40) || (long long)n_seq * H >= (1ll << 31) || rows >= (1ll << 31) ||
      n_seq >= (1 << 30))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if (packed && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is not 4-byte aligned");
  const bool tokens = rows > 0;
  if ((s = check_ptr(q, "q", tokens)) || (s = check_ptr(k, "k", tokens)) ||
      (s = check_ptr(v, "v", tokens)) || (s = check_ptr(g, "g", tokens)) ||
      (s = check_ptr(beta, "beta", tokens)) || (s = check_ptr(out, "out", tokens)) ||
      (s = check_ptr(gate_u, "gate_u", tokens)) || (s = check_ptr(norm_w, "norm_w", tokens)) ||
      (s = check_ptr(S0, "S0", false)) || (s = check_ptr(S_final, "S_final", false)))
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  kda::SeqParams P{q, k, v, g, beta, S0, out, S_final, cu_seqlens, n_seq, H, T};
  const int n_problems = n_seq * H;
  if (dtype == KDA_DTYPE_BF16 && d_k == 128 && kda::tc::tc_supports(C)) {
    // the tensor-core kernel gates each block's output on its way out
    P.gate_u = gate_u;
    P.norm_w = norm_w;
    P.norm_eps = norm_eps;
    return run_chunk(P, n_problems, d_k, C, dtype, st);
  }
  // other shapes: the raw output, then the standalone gate over it in place
  if ((s = run_chunk(P, n_problems, d_k, C, dtype, st)) != KDA_OK) return s;
  return launch_output_gate(out, gate_u, norm_w, norm_eps, out, rows * H, d_v, dtype, st);
}

kda_status_t kda_output_gate(const void* o, const void* gate_u, const float* norm_w,
                             float norm_eps, void* y, long long n_rows, int d_v,
                             kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(1, d_v, d_v, dtype);
  if (s != KDA_OK) return s;
  if (n_rows < 0) return fail(KDA_ERR_INVALID_ARG, "n_rows must be >= 0");
  if (n_rows >= (1ll << 36)) return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if (!(norm_eps >= 0.f) || !(norm_eps < 1e30f))
    return fail(KDA_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
  const bool any = n_rows > 0;
  if ((s = check_ptr(o, "o", any)) || (s = check_ptr(gate_u, "gate_u", any)) ||
      (s = check_ptr(norm_w, "norm_w", any)) || (s = check_ptr(y, "y", any)))
    return s;
  return launch_output_gate(o, gate_u, norm_w, norm_eps, y, n_rows, d_v, dtype,
                            static_cast<cudaStream_t>(stream));
}

kda_status_t kda_pre_core(const void* q_raw, const void* k_raw, const void* v_raw,
                          const void* z, const float* conv_q, const float* conv_k,
                          const float* conv_v, const float* A_log, const float* b_decay, void* q,
                          void* k, void* v, void* g, const int32_t* cu_seqlens, int n_seq, int H,
                          int T, int d, kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d, d, dtype);
  if (s != KDA_OK) return s;
  if (n_seq < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "n_seq and T must be >= 0 (got %d, %d)", n_seq, T);
  const bool packed = cu_seqlens != nullptr;
  const long long rows = packed ? (long long)T : (long long)n_seq * T;
  if (rows * H * d >= (1ll << 40) || rows >= (1ll << 31) || n_seq >= (1 << 30))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if (packed && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is not 4-byte aligned");
  const bool any = rows > 0;
  if ((s = check_ptr(q_raw, "q_raw", any)) || (s = check_ptr(k_raw, "k_raw", any)) ||
      (s = check_ptr(v_raw, "v_raw", any)) || (s = check_ptr(z, "z", any)) ||
      (s = check_ptr(conv_q, "conv_q", any)) || (s = check_ptr(conv_k, "conv_k", any)) ||
      (s = check_ptr(conv_v, "conv_v", any)) || (s = check_ptr(A_log, "A_log", any)) ||
      (s = check_ptr(b_decay, "b_decay", any)) || (s = check_ptr(q, "q", any)) ||
      (s = check_ptr(k, "k", any)) || (s = check_ptr(v, "v", any)) || (s = check_ptr(g, "g", any)))
    return s;
  if (!any) return KDA_OK;
  kda::pre::PreParams P{q_raw, k_raw, v_raw, z, conv_q, conv_k, conv_v, A_log, b_decay,
                        q, k, v, g, cu_seqlens, n_seq, H, T};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int tok_per_cta = 4 * (256 / (d / 8));
  const long long tiles = (rows + tok_per_cta - 1) / tok_per_cta;
  // (head, tile, output tensor); the kernel strides over tiles
  const dim3 grid((unsigned)H, (unsigned)(tiles < 65535 ? tiles : 65535), 4);
  using bf = __nv_bfloat16;
  if (d == 128) {
    if (dtype == KDA_DTYPE_BF16) kda::pre::pre_core_kernel<bf, 128><<<grid, 256, 0, st>>>(P, rows);
    else kda::pre::pre_core_kernel<float, 128><<<grid, 256, 0, st>>>(P, rows);
  } else {
    if (dtype == KDA_DTYPE_BF16) kda::pre::pre_core_kernel<bf, 64><<<grid, 256, 0, st>>>(P, rows);
    else kda::pre::pre_core_kernel<float, 64><<<grid, 256, 0, st>>>(P, rows);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pre_core launch");
  return KDA_OK;
}

kda_status_t kda_chunk_fwd_fused(const void* q_raw, const void* k_raw, const void* v_raw,
                                 const void* z, const void* beta, const float* conv_q,
                                 const float* conv_k, const float* conv_v, const float* A_log,
                                 const float* b_decay, const float* S0, const void* gate_u,
                                 const float* norm_w, float norm_eps, void* out, float* S_final,
                                 const int32_t* cu_seqlens, int n_seq, int H, int T, int d_k,
                                 int d_v, int C, kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d_k, d_v, dtype);
  if (s != KDA_OK) return s;
  if (!(dtype == KDA_DTYPE_BF16 && d_k == 128 && (C == 64 || C == 128)))
    return fail(KDA_ERR_UNSUPPORTED,
                "the fused input side runs on the bf16 tensor-core path (d = 128, C = 64 or 128); "
                "for other shapes use kda_pre_core, then kda_chunk_fwd or kda_chunk_fwd_gated");
  if (n_seq < 0 || T < 0) return fail(KDA_ERR_INVALID_ARG, "n_seq and T must be >= 0 (got %d, %d)", n_seq, T);
  if (gate_u != nullptr && (!(norm_eps >= 0.f) || !(norm_eps < 1e30f)))
    return fail(KDA_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
  const bool packed = cu_seqlens != nullptr;
  const long long rows = packed ? (long long)T : (long long)n_seq * T;
  if (rows * H * d_k >= (1ll << 40) || (long long)n_seq * H >= (1ll << 31) || rows >= (1ll << 31) ||
      n_seq >= (1 << 30))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if (packed && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is not 4-byte aligned");
  const bool tokens = rows > 0;
  if ((s = check_ptr(q_raw, "q_raw", tokens)) || (s = check_ptr(k_raw, "k_raw", tokens)) ||
      (s = check_ptr(v_raw, "v_raw", tokens)) || (s = check_ptr(z, "z", tokens)) ||
      (s = check_ptr(beta, "beta", tokens)) || (s = check_ptr(out, "out", tokens)) ||
      (s = check_ptr(conv_q, "conv_q", tokens)) || (s = check_ptr(conv_k, "conv_k", tokens)) ||
      (s = check_ptr(conv_v, "conv_v", tokens)) || (s = check_ptr(A_log, "A_log", tokens)) ||
      (s = check_ptr(b_decay, "b_decay", tokens)) || (s = check_ptr(gate_u, "gate_u", false)) ||
      (s = check_ptr(norm_w, "norm_w", gate_u != nullptr && tokens)) ||
      (s = check_ptr(S0, "S0", false)) || (s = check_ptr(S_final, "S_final", false)))
    return s;
  kda::SeqParams P{q_raw, k_raw, v_raw, z, beta, S0, out, S_final, cu_seqlens, n_seq, H, T};
  P.conv_q = conv_q;
  P.conv_k = conv_k;
  P.conv_v = conv_v;
  P.A_log = A_log;
  P.b_decay = b_decay;
  P.gate_u = gate_u;
  P.norm_w = norm_w;
  P.norm_eps = norm_eps;
  return run_chunk(P, n_seq * H, d_k, C, dtype, static_cast<cudaStream_t>(stream));
}

kda_status_t kda_segment_transitions(const void* k, const void* v, const void* g,
                                     const void* beta, float* M, float* S_tilde, int B, int H,
                                     int T, int seg_len, int n_seg, int d_k, int d_v, int C,
                                     kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d_k, d_v, dtype);
  if (s != KDA_OK) return s;
  if (B < 0 || T < 0 || n_seg < 0)
    return fail(KDA_ERR_INVALID_ARG, "B, T and n_seg must be >= 0 (got %d, %d, %d)", B, T, n_seg);
  if (seg_len < 1) return fail(KDA_ERR_INVALID_ARG, "seg_len must be >= 1 (got %d)", seg_len);
  if (!(C == 16 || C == 32 || C == 64 || C == 128))
    return fail(KDA_ERR_UNSUPPORTED, "C must be 16, 32, 64 or 128 (got %d)", C);
  if ((long long)B * T * H * d_k >= (1ll << 40) || 2ll * n_seg * B * H >= (1ll << 31) ||
      (long long)B * T >= (1ll << 31))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  const long long work = (long long)n_seg * B * H;
  if (work == 0) return KDA_OK;
  const bool tokens = (long long)B * T > 0;
  if ((s = check_ptr(k, "k", tokens)) || (s = check_ptr(v, "v", tokens)) ||
      (s = check_ptr(g, "g", tokens)) || (s = check_ptr(beta, "beta", tokens)) ||
      (s = check_ptr(M, "M", true)) || (s = check_ptr(S_tilde, "S_tilde", true)))
    return s;
  // q is never read for its outputs here (none are written); k stands in for it
  kda::SeqParams P{k, k, v, g, beta, nullptr, nullptr, S_tilde, nullptr, B, H, T};
  P.seg_len = seg_len;
  P.n_seg = n_seg;
  P.n_ident = (int)work;
  P.M_out = M;
  return run_chunk(P, (int)(2 * work), d_k, C, dtype, static_cast<cudaStream_t>(stream));
}

kda_status_t kda_segment_scan(const float* M, const float* S_tilde, const float* S0, float* S_in,
                              int n_seg, int B, int H, int d_k, int d_v, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d_k, d_v, KDA_DTYPE_F32);
  if (s != KDA_OK) return s;
  if (n_seg < 1 || B < 0)
    return fail(KDA_ERR_INVALID_ARG, "n_seg must be >= 1 and B >= 0 (got %d, %d)", n_seg, B);
  if ((long long)B * H >= (1ll << 31) || (long long)n_seg * B * H * d_k * d_v >= (1ll << 40))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if (B == 0) return KDA_OK;
  if ((s = check_ptr(M, "M", n_seg > 1)) || (s = check_ptr(S_tilde, "S_tilde", n_seg > 1)) ||
      (s = check_ptr(S0, "S0", false)) || (s = check_ptr(S_in, "S_in", true)))
    return s;
  return launch_scan(M, S_tilde, S0, S_in, n_seg, B * H, d_k, d_v,
                     static_cast<cudaStream_t>(stream));
}

size_t kda_chunk_fwd_segmented_workspace(int B, int H, int T, int d_k, int d_v, int n_seg) {
  if (B < 0 || H < 1 || T < 1 || n_seg < 1 || d_k < 1 || d_v < 1) return 0;
  if (n_seg == 1) return 0;
  const long long n = ((long long)T + segment_tokens(T, n_seg) - 1) / segment_tokens(T, n_seg);
  const long long segs = n < 1 ? 1 : n;
  // M and S~ of the first segs - 1 segments, then S_in of every segment
  return (size_t)4 * (size_t)B * H * ((size_t)(segs - 1) * ((size_t)d_k * d_k + (size_t)d_k * d_v) +
                                      (size_t)segs * d_k * d_v);
}

kda_status_t kda_chunk_fwd_segmented(const void* q, const void* k, const void* v, const void* g,
                                     const void* beta, const float* S0, void* out,
                                     float* S_final, int B, int H, int T, int d_k, int d_v, int C,
                                     int n_seg, void* workspace, size_t workspace_bytes,
                                     kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  if (n_seg < 1) return fail(KDA_ERR_INVALID_ARG, "n_seg must be >= 1 (got %d)", n_seg);
  const long long seg = segment_tokens(T, n_seg);
  const int segs = T > 0 ? (int)(((long long)T + seg - 1) / seg) : 1;
  if (segs <= 1)
    return kda_chunk_fwd(q, k, v, g, beta, S0, out, S_final, B, H, T, d_k, d_v, C, dtype, stream);
  kda_status_t s = check_common(H, d_k, d_v, dtype);
  if (s != KDA_OK) return s;
  if (B < 0) return fail(KDA_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
  if (!(C == 16 || C == 32 || C == 64 || C == 128))
    return fail(KDA_ERR_UNSUPPORTED, "C must be 16, 32, 64 or 128 (got %d)", C);
  if ((long long)B * T * H * d_k >= (1ll << 40) || 2ll * segs * B * H >= (1ll << 31) ||
      (long long)B * T >= (1ll << 31))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if (B == 0) return KDA_OK;
  const size_t need = kda_chunk_fwd_segmented_workspace(B, H, T, d_k, d_v, n_seg);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(KDA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu%s)", need,
                workspace_bytes, workspace ? "" : ", NULL");
  if ((s = check_ptr(q, "q", true)) || (s = check_ptr(k, "k", true)) ||
      (s = check_ptr(v, "v", true)) || (s = check_ptr(g, "g", true)) ||
      (s = check_ptr(beta, "beta", true)) || (s = check_ptr(out, "out", true)) ||
      (s = check_ptr(S0, "S0", false)) || (s = check_ptr(S_final, "S_final", false)) ||
      (s = check_ptr(workspace, "workspace", true)))
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t BH = (size_t)B * H;
  float* M = static_cast<float*>(workspace);
  float* St = M + (size_t)(segs - 1) * BH * d_k * d_k;
  float* S_in = St + (size_t)(segs - 1) * BH * d_k * d_v;
  // 1. (M, S~) of every segment but the last
  kda::SeqParams P1{k, k, v, g, beta, nullptr, nullptr, St, nullptr, B, H, T};
  P1.seg_len = (int)seg;
  P1.n_seg = segs - 1;
  P1.n_ident = (int)((segs - 1) * BH);
  P1.M_out = M;
  if ((s = run_chunk(P1, 2 * P1.n_ident, d_k, C, dtype, st)) != KDA_OK) return s;
  // 2. incoming state of every segment
  if ((s = launch_scan(M, St, S0, S_in, segs, (int)BH, d_k, d_v, st)) != KDA_OK) return s;
  // 3. every segment from its incoming state: outputs, and the final state of the last one
  kda::SeqParams P2{q, k, v, g, beta, S_in, out, S_final, nullptr, B, H, T};
  P2.seg_len = (int)seg;
  P2.n_seg = segs;
  P2.sf_last_only = 1;
  return run_chunk(P2, (int)(segs * BH), d_k, C, dtype, st);
}

}  // extern "C"

// Scratch of kda_chunk_fwd_segmented_noalloc: a fixed array in the library's device image, so
// that the call needs no allocation. Every device that loads the library holds it until the
// process exits. In host code the name stands for a host-side shadow, not a device address; the
// device address comes from cudaGetSymbolAddress, once per device, in noalloc_scratch().
static __device__ __align__(256) unsigned char kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device (looked up on the first call there).
kda_status_t noalloc_scratch(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(KDA_ERR_UNSUPPORTED, "device ordinal %d is beyond the %d devices tracked", dev,
                kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, kda_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(kda_noalloc_scratch)");
    g_noalloc_addr[dev] = p;
  }
  *addr = g_noalloc_addr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_chunk_fwd_segmented_noalloc(const void* q, const void* k, const void* v,
                                             const void* g, const void* beta, const float* S0,
                                             void* out, float* S_final, int B, int H, int T,
                                             int d_k, int d_v, int C, int n_seg,
                                             kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  if (n_seg < 1) return fail(KDA_ERR_INVALID_ARG, "n_seg must be >= 1 (got %d)", n_seg);
  const size_t need = kda_chunk_fwd_segmented_workspace(B, H, T, d_k, d_v, n_seg);
  if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES)
    return fail(KDA_ERR_UNSUPPORTED,
                "this request needs %zu bytes of scratch; the library's fixed scratch holds %zu "
                "(use fewer segments, or kda_chunk_fwd_segmented with a caller workspace)",
                need, (size_t)KDA_NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  if (need > 0) {
    kda_status_t s = noalloc_scratch(&ws);
    if (s != KDA_OK) return s;
  }
  // The segmented path writes every byte of scratch it reads (transitions, then the scan), so
  // nothing in the array has to start at zero.
  return kda_chunk_fwd_segmented(q, k, v, g, beta, S0, out, S_final, B, H, T, d_k, d_v, C, n_seg,
                                 ws, need, dtype, stream);
}

int kda_segments_auto(int B, int H, int T) {
  if (B < 1 || H < 1 || T < 1) return 1;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long P = (long long)B * H;
  const long long nb = ((long long)T + 63) / 64;
  // cost in 64-token block times: transitions (two problems per segment but the last), the
  // scan (about a quarter block per segment) and the outputs pass; two extra launches
  auto waves = [&](long long n) { return (n + sms - 1) / sms; };
  double best = (double)waves(P) * nb;
  int best_n = 1;
  for (int n = 2; n <= 64 && n <= nb; ++n) {
    const long long L = (nb + n - 1) / n;
    const int segs = (int)((nb + L - 1) / L);
    const double cost = (double)waves(2 * P * (segs - 1)) * L + 0.25 * (segs - 1) +
                        (double)waves(P * segs) * L + 1.0;
    if (cost < best * 0.97) {
      best = cost;
      best_n = segs;
    }
  }
  return best_n;
}

kda_status_t kda_recurrent_steps(const void* q, const void* k, const void* v, const void* g,
                                 const void* beta, float* S, void* out, int N, int K, int H,
                                 int d_k, int d_v, kda_dtype_t dtype, void* stream) {
  t_last_error.clear();
  kda_status_t s = check_common(H, d_k, d_v, dtype);
  if (s != KDA_OK) return s;
  if (N < 0 || K < 0) return fail(KDA_ERR_INVALID_ARG, "N and K must be >= 0 (got %d, %d)", N, K);
  if (N == 0 || K == 0) return KDA_OK;
  // two CTAs per (sequence, head) at d = 128: N * H * 2 must stay a valid grid size
  if ((long long)N * H >= (1ll << 30) || (long long)N * K * H * d_k >= (1ll << 40))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if ((s = check_ptr(q, "q", true)) || (s = check_ptr(k, "k", true)) ||
      (s = check_ptr(v, "v", true)) || (s = check_ptr(g, "g", true)) ||
      (s = check_ptr(beta, "beta", true)) || (s = check_ptr(S, "S", true)) ||
      (s = check_ptr(out, "out", true)))
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = N * H;
  using bf = __nv_bfloat16;
  if (dtype == KDA_DTYPE_F32) {
    const float *qq = (const float*)q, *kk = (const float*)k, *vv = (const float*)v,
                *gg = (const float*)g, *bb = (const float*)beta;
    if (d_k == 128)
      kda::decode_tokens_kernel<float, 128, 128, 128><<<grid * 2, 128, 0, st>>>(qq, kk, vv, gg, bb, S, (float*)out, K, H);
    else
      kda::decode_tokens_kernel<float, 64, 64, 128><<<grid, 128, 0, st>>>(qq, kk, vv, gg, bb, S, (float*)out, K, H);
  } else {
    const bf *qq = (const bf*)q, *kk = (const bf*)k, *vv = (const bf*)v, *gg = (const bf*)g,
             *bb = (const bf*)beta;
    if (d_k == 128)
      kda::decode_tokens_kernel<bf, 128, 128, 128><<<grid * 2, 128, 0, st>>>(qq, kk, vv, gg, bb, S, (bf*)out, K, H);
    else
      kda::decode_tokens_kernel<bf, 64, 64, 128><<<grid, 128, 0, st>>>(qq, kk, vv, gg, bb, S, (bf*)out, K, H);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_tokens launch");
  return KDA_OK;
}

kda_status_t kda_wait_selftest(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(KDA_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10] (got %llu)", limit_ns);
  kda::selftest::unanswered_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
  return KDA_OK;
}

kda_status_t kda_sync_status(void* stream) {
  static std::atomic<unsigned int> next_slot{0};
  t_last_error.clear();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Everything queued on `stream` before this call finishes first; then one thread takes the
  // word and clears it in a single atomic exchange, so a code latched by a kernel on another
  // stream is either taken here or left for the next call, never lost.
  const int slot = (int)(next_slot.fetch_add(1u) % (unsigned)kda::kStatusSlots);
  kda::take_status_kernel<<<1, 1, 0, st>>>(slot);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "status read launch");
  unsigned int word = 0;
  e = cudaMemcpyFromSymbolAsync(&word, kda::g_status_taken, sizeof(word),
                                sizeof(word) * (size_t)slot, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (word != 0)
    return fail((kda_status_t)word, "device reported %s", kda_status_string((kda_status_t)word));
  return KDA_OK;
}

const char* kda_status_string(kda_status_t status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
  }
  return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error(void) { return t_last_error.c_str(); }

int kda_version(void) { return 100; }

}  // extern "C"
