// C ABI of the KDA forward library: argument validation, kernel selection and launches.
// Declarations and the full contract are in include/kda.h.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/kda.h"
#include "kda_chunk_simt.cuh"
#include "kda_chunk_tc.cuh"
#include "kda_common.cuh"
#include "kda_decode.cuh"
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
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(chunk_simt)");
    kern<<<n_problems, THREADS, SM::bytes, st>>>(P);
  } else {
    using SM = kda::SimtSmem<D, D, 32>;
    auto kern = kda::chunk_simt_kernel<TIn, D, D, 32, THREADS>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::bytes);
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
  if (dtype == KDA_DTYPE_BF16 && d == 128 && kda::tc_supports(C)) {
    kda_status_t s = kda::launch_chunk_tc(P, n_problems, C, st, t_last_error);
    return s;
  }
  if (dtype == KDA_DTYPE_F32)
    return d == 128 ? launch_simt<float, 128>(P, n_problems, C, st)
                    : launch_simt<float, 64>(P, n_problems, C, st);
  return d == 128 ? launch_simt<__nv_bfloat16, 128>(P, n_problems, C, st)
                  : launch_simt<__nv_bfloat16, 64>(P, n_problems, C, st);
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
  if ((long long)B * T * H * d_k >= (1ll << 40))
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
  if ((long long)T_total * H * d_k >= (1ll << 40))
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

kda_status_t kda_wait_selftest(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(KDA_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10] (got %llu)", limit_ns);
  kda::selftest::unanswered_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
  return KDA_OK;
}

kda_status_t kda_sync_status(void* stream) {
  t_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&word, kda::g_status, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (word != 0) {
    e = cudaMemcpyToSymbol(kda::g_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
    return fail((kda_status_t)word, "device reported %s", kda_status_string((kda_status_t)word));
  }
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
