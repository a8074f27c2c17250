/*
 * kda.h -- C ABI of the KDA (Kimi Delta Attention) forward library for NVIDIA B300 (sm_103a).
 *
 * What is computed (Kimi K3 wiki, "Notations mathématiques", table "Attention et KDA"):
 *   alpha_t = exp(g_t)                      per key channel, g_t in (g_min = -5, 0)^{d_k}
 *   S_t     = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t     = S_t^T q_t                     raw output, read from the updated state
 * Prefill uses the exact chunkwise (block) form: serial across blocks of C tokens, parallel
 * inside a block (Glossaire, entries "Chunkwise" and "UT"); decode applies one token of the
 * recurrence to a resident state (Glossaire, entry "Decode").
 *
 * Conventions shared by every entry point
 *  - Every tensor pointer is a DEVICE pointer on the current CUDA device, 16-byte aligned,
 *    contiguous row-major, in the layout given below. The caller owns every buffer; the
 *    library allocates no device memory.
 *  - Sequence tensors use [B, T, H, d]: q, k, g are [B, T, H, d_k]; v and out are
 *    [B, T, H, d_v]; beta is [B, T, H]. Their element type is `dtype` (all the same).
 *  - States S0, S_final, S are fp32 [B (or N), H, d_k, d_v] with d_v fastest.
 *  - q and k are expected to be L2-normalised per token (a precondition of the method, not
 *    re-checked). No 1/sqrt(d_k) scale is applied. Values of g and beta are not range-checked.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Calls are
 *    asynchronous: a KDA_OK return means the arguments were valid and the work was enqueued.
 *  - Errors: invalid pointers/sizes return KDA_ERR_INVALID_ARG and shapes outside the
 *    supported set return KDA_ERR_UNSUPPORTED, both before anything is launched; a failed
 *    launch returns KDA_ERR_CUDA. Conditions detected on the device (a bounded wait that ran
 *    out, inconsistent cu_seqlens) are latched in a per-device status word that
 *    kda_sync_status() returns and clears. kda_last_error() gives a message for the most
 *    recent failure on the calling thread.
 *  - Supported: d_k = d_v in {64, 128}; C in {16, 32, 64, 128}; T >= 0; B, H >= 1 (B = 0 or
 *    T = 0 is a no-op apart from copying S0 to S_final).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative or inconsistent size        */
  KDA_ERR_UNSUPPORTED = 2, /* valid request outside the supported shapes/dtypes              */
  KDA_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed                            */
  KDA_ERR_TIMEOUT = 4      /* a bounded on-device wait gave up (reported by kda_sync_status) */
} kda_status_t;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype_t;

/*
 * Chunkwise prefill over a dense batch of B sequences of T tokens each.
 *   q, k, g : [B, T, H, d_k]  dtype      v : [B, T, H, d_v]  dtype     beta : [B, T, H] dtype
 *   S0      : [B, H, d_k, d_v] fp32, read only; NULL means a zero initial state
 *   out     : [B, T, H, d_v]  dtype, written (o_t for every token)
 *   S_final : [B, H, d_k, d_v] fp32, written with the state after token T; NULL = not written
 *   C       : chunk size (16, 32, 64 or 128); the result does not depend on it beyond rounding
 * fp32 inputs run on CUDA cores in fp32 throughout, in 16- or 32-token blocks. bf16 inputs run
 * on the tensor cores (bf16 operands, fp32 accumulation, fp32 state) when C is 64 or 128; that
 * kernel works in 64-token blocks, so a 128-token chunk is processed as two consecutive 64-token
 * blocks (the same mathematics), and in 128-channel tiles, so a head of 64 channels runs with
 * the upper half of every tile zero (the results are those of the 64-channel problem).
 */
kda_status_t kda_chunk_fwd(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, const float* S0, void* out, float* S_final,
                           int B, int H, int T, int d_k, int d_v, int C, kda_dtype_t dtype,
                           void* stream);

/*
 * Chunkwise prefill over a packed batch of N variable-length sequences sharing one token
 * axis of length T_total (the leading batch dimension is 1).
 *   q, k, g : [1, T_total, H, d_k]   v, out : [1, T_total, H, d_v]   beta : [1, T_total, H]
 *   cu_seqlens : DEVICE int32 [N + 1]; sequence s owns tokens [cu_seqlens[s], cu_seqlens[s+1]);
 *                must satisfy cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] = T_total.
 *                Violations are caught on the device: the affected sequences are skipped and
 *                kda_sync_status() reports KDA_ERR_INVALID_ARG.
 *   S0, S_final : [N, H, d_k, d_v] fp32 (per sequence; NULL as above). The state is reset at
 *                 every sequence boundary. Blocks start at each sequence's first token; the
 *                 last block of a sequence may be partial.
 */
kda_status_t kda_chunk_fwd_varlen(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* S0, void* out,
                                  float* S_final, const int32_t* cu_seqlens, int N, int H,
                                  int T_total, int d_k, int d_v, int C, kda_dtype_t dtype,
                                  void* stream);

/*
 * One decode token for N sequences x H heads, updating the resident states in place.
 *   q, k, g : [N, H, d_k] dtype   v, out : [N, H, d_v] dtype   beta : [N, H] dtype
 *   S       : [N, H, d_k, d_v] fp32, read and overwritten with the updated state
 * out receives o = S_new^T q. S must not alias any other argument.
 */
kda_status_t kda_recurrent_step(const void* q, const void* k, const void* v, const void* g,
                                const void* beta, float* S, void* out, int N, int H, int d_k,
                                int d_v, kda_dtype_t dtype, void* stream);

/*
 * K decode tokens for each of N sequences x H heads, updating the resident states in place: the
 * recurrence applied K times (Glossaire, entry "Decode"), with each state slice held on chip across
 * the K tokens, so the state crosses HBM once in each direction whatever K is (verification of K
 * speculative draft tokens, or a short run of tokens).
 *   q, k, g : [N, K, H, d_k] dtype   v, out : [N, K, H, d_v] dtype   beta : [N, K, H] dtype
 *   S       : [N, H, d_k, d_v] fp32, read and overwritten with the state after the K tokens
 * out receives o_t = S_t^T q_t for every token. K = 1 computes what kda_recurrent_step computes
 * (to fp32 rounding: the column sums over the key channel are added in another order). N * H
 * must be below 2^30 (KDA_ERR_UNSUPPORTED otherwise).
 */
kda_status_t kda_recurrent_steps(const void* q, const void* k, const void* v, const void* g,
                                 const void* beta, float* S, void* out, int N, int K, int H,
                                 int d_k, int d_v, kda_dtype_t dtype, void* stream);

/*
 * Chunkwise prefill followed by the output side of the layer (Kimi K3 wiki, "Notations
 * mathématiques": o~_t is the raw output before the gate; table "Fonctions": RMSNorm(x) =
 * x / sqrt(mean_i x_i^2 + eps) * w; chapter 03: RMSNorm on KDA's recurrent output; "Tableau des
 * spécifications": RMSNorm epsilon 1e-5 and a full-rank KDA output gate). `out` receives
 *   y_t = RMSNorm(o~_t) * norm_w * sigma(u_t)       per token and head, over the d_v channels
 *   gate_u : the gate pre-activation u, shaped and typed like out (the full-rank gate
 *            projection is the caller's)
 *   norm_w : fp32 [d_v], one RMSNorm weight vector shared by the heads; norm_eps >= 0 (1e-5 in K3)
 * cu_seqlens NULL: a dense batch (n_seq = B sequences of T tokens, the layout of kda_chunk_fwd);
 * otherwise a packed batch (n_seq = N sequences, T = T_total, the layout and rules of
 * kda_chunk_fwd_varlen). S0 / S_final as in those calls. The bf16 tensor-core path (d = 128,
 * C = 64 or 128) normalises and gates each block in its output epilogue, from the bf16-rounded
 * raw output; the other paths write o~ and apply kda_output_gate over it in place. Both give the
 * same bits for the same raw output. Precision: with bf16 tensors 1/sqrt(mean + eps) is the
 * hardware reciprocal square root and sigma the hardware tanh form (errors far below the bf16
 * rounding of y); with fp32 tensors both are computed to fp32 accuracy.
 */
kda_status_t kda_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* g,
                                 const void* beta, const float* S0, const void* gate_u,
                                 const float* norm_w, float norm_eps, void* out, float* S_final,
                                 const int32_t* cu_seqlens, int n_seq, int H, int T, int d_k,
                                 int d_v, int C, kda_dtype_t dtype, void* stream);

/*
 * The output side alone (same definition and references as kda_chunk_fwd_gated), for the raw
 * outputs of decode steps or of any other call: y = RMSNorm(o) * norm_w * sigma(u) over each row
 * of d_v channels. o, gate_u, y: [n_rows, d_v] of `dtype` (y may be o); norm_w fp32 [d_v];
 * d_v in {64, 128}.
 */
kda_status_t kda_output_gate(const void* o, const void* gate_u, const float* norm_w,
                             float norm_eps, void* y, long long n_rows, int d_v,
                             kda_dtype_t dtype, void* stream);

/*
 * The input side of the layer (Kimi K3 wiki, "Notations mathématiques", table "Fonctions":
 * ShortConv = causal convolution with a kernel of size 4, L2Norm(x) = x / ||x||_2; table
 * "Attention et KDA": q, k L2-normalised, per-head log scale A_h, per-head decay bias b_alpha^h,
 * decay logit z_t; "Glossaire", entry "Décroissance bornée": g = g_min sigma(e^A z), g_min = -5):
 *   q = L2Norm(ShortConv(q_raw)), k = L2Norm(ShortConv(k_raw)), v = ShortConv(v_raw),
 *   g = -5 sigma(e^{A_log[h]} z + b_decay[h])
 * ShortConv is depthwise: conv_q / conv_k / conv_v are fp32 [H, 4, d], tap-major, with [h, j, c]
 * the weight of channel c on the token j steps back (a [H * d, 1, 4] convolution weight transposed
 * once); zeros before the first token of each sequence, no activation after it.
 * A_log fp32 [H]; b_decay fp32 [H, d]. q_raw, k_raw, v_raw, z and the outputs q, k, v, g share
 * the token layout of kda_chunk_fwd (cu_seqlens NULL: n_seq = B sequences of T tokens) or of
 * kda_chunk_fwd_varlen (cu_seqlens given: n_seq = N, T = T_total). Any dtype, d in {64, 128}.
 */
kda_status_t kda_pre_core(const void* q_raw, const void* k_raw, const void* v_raw,
                          const void* z, const float* conv_q, const float* conv_k,
                          const float* conv_v, const float* A_log, const float* b_decay, void* q,
                          void* k, void* v, void* g, const int32_t* cu_seqlens, int n_seq, int H,
                          int T, int d, kda_dtype_t dtype, void* stream);

/*
 * The layer from the raw projections in one pass: the input side of kda_pre_core computed inside
 * the prefill kernel (k, q, z and v are convolved, normalised and gated in shared memory as each
 * block lands; they never return to global memory), the chunkwise recurrence, and, if gate_u is
 * given, the output side of kda_chunk_fwd_gated in the output epilogue (gate_u NULL: out is the
 * raw output o~). Arguments as in kda_pre_core and kda_chunk_fwd_gated. bf16, d_k = d_v = 128,
 * C in {64, 128} only (KDA_ERR_UNSUPPORTED otherwise: use kda_pre_core and the other calls).
 */
kda_status_t kda_chunk_fwd_fused(const void* q_raw, const void* k_raw, const void* v_raw,
                                 const void* z, const void* beta, const float* conv_q,
                                 const float* conv_k, const float* conv_v, const float* A_log,
                                 const float* b_decay, const float* S0, const void* gate_u,
                                 const float* norm_w, float norm_eps, void* out, float* S_final,
                                 const int32_t* cu_seqlens, int n_seq, int H, int T, int d_k,
                                 int d_v, int C, kda_dtype_t dtype, void* stream);

/*
 * Segment transitions (Kimi K3 wiki, "Notations mathématiques", table "Attention et KDA": the
 * transition M_t and S~, the state computed from S = 0; "Glossaire", entry "KCP": the pair
 * (cumulative M, local S~) of a stretch of tokens composes associatively and exactly).
 * Segment sigma (0 <= sigma < n_seg) of sequence b covers its tokens
 * [sigma * seg_len, min((sigma + 1) * seg_len, T)); for every (sigma, b, h) this writes
 *   M       [n_seg, B, H, d_k, d_k] fp32 : the product M_{last} ... M_{first} of the segment
 *   S_tilde [n_seg, B, H, d_k, d_v] fp32 : the state the segment reaches from S = 0
 * so that S_after = M S_before + S~ for any incoming state. An empty segment gives (I, 0).
 *   k, g : [B, T, H, d_k] dtype   v : [B, T, H, d_v] dtype   beta : [B, T, H] dtype
 * Requires d_k = d_v (supported head sizes as above); seg_len >= 1. Computed by the prefill
 * kernels themselves (M as the final state of a run from S0 = I with v = 0, S~ as that of a run
 * from S0 = 0), so the precision is that of kda_chunk_fwd for the same dtype.
 */
kda_status_t kda_segment_transitions(const void* k, const void* v, const void* g,
                                     const void* beta, float* M, float* S_tilde, int B, int H,
                                     int T, int seg_len, int n_seg, int d_k, int d_v, int C,
                                     kda_dtype_t dtype, void* stream);

/*
 * Incoming state of every segment from the segments' transitions (same references):
 *   S_in[0] = S0 (zeros if S0 is NULL),  S_in[s + 1] = M[s] S_in[s] + S_tilde[s]
 *   M [n_seg - 1, B, H, d_k, d_k], S_tilde [n_seg - 1, B, H, d_k, d_v] (both unused and
 *   may be NULL when n_seg = 1), S0 [B, H, d_k, d_v] or NULL, S_in [n_seg, B, H, d_k, d_v]:
 * all fp32 device arrays. fp32 arithmetic; the segments of one (b, h) are composed in order,
 * different (b, h) and value columns in parallel. n_seg >= 1.
 */
kda_status_t kda_segment_scan(const float* M, const float* S_tilde, const float* S0, float* S_in,
                              int n_seg, int B, int H, int d_k, int d_v, void* stream);

/*
 * Chunkwise prefill of a dense batch, parallel along T: the same contract and results (up to
 * rounding) as kda_chunk_fwd, for batches with too few (sequence, head) problems to fill the
 * GPU. T is cut into at most n_seg segments of whole 64-token blocks (seg_len =
 * ceil(ceil(T / 64) / n_seg) * 64 tokens); the call runs kda_segment_transitions over every
 * segment but the last, kda_segment_scan from S0, then every segment from its incoming state
 * (outputs, and S_final from the last segment). With one segment it is kda_chunk_fwd.
 *   workspace : caller-owned DEVICE scratch of at least
 *               kda_chunk_fwd_segmented_workspace(B, H, T, d_k, d_v, n_seg) bytes, 16-byte
 *               aligned; its contents on entry are ignored and on return unspecified. Two calls
 *               in flight at the same time need distinct workspaces.
 * Returns KDA_ERR_INVALID_ARG if the workspace is missing or too small.
 */
kda_status_t kda_chunk_fwd_segmented(const void* q, const void* k, const void* v, const void* g,
                                     const void* beta, const float* S0, void* out,
                                     float* S_final, int B, int H, int T, int d_k, int d_v, int C,
                                     int n_seg, void* workspace, size_t workspace_bytes,
                                     kda_dtype_t dtype, void* stream);

/* Bytes of workspace kda_chunk_fwd_segmented needs (0 when it needs none or the sizes are
 * invalid). Host-only; touches no device. */
size_t kda_chunk_fwd_segmented_workspace(int B, int H, int T, int d_k, int d_v, int n_seg);

/* A segment count for kda_chunk_fwd_segmented on the current device (1 when the (B, H)
 * problems alone fill its SMs), from a cost model of the three passes in 64-token block times.
 * Host-only apart from reading the device's SM count (148 if no device is visible). */
int kda_segments_auto(int B, int H, int T);

/* Bytes of the fixed device scratch behind kda_chunk_fwd_segmented_noalloc (32 MiB). */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * kda_chunk_fwd_segmented without a caller workspace and without any allocation. The pages have
 * no counterpart to this entry point; it exists for callers that cannot allocate device memory
 * at the point of the call: runtimes whose device memory is all owned by a fixed arena or pool,
 * plug-ins whose host hands them tensors but no allocator, and loops that cannot afford the
 * synchronisation and unpredictable latency of cudaMalloc / cudaFree.
 *
 * Same arguments, results and errors as kda_chunk_fwd_segmented, minus the workspace. The scratch
 * is one array of KDA_NOALLOC_SCRATCH_BYTES in the library's device image, held on every device
 * that loads the library until the process exits. A request whose scratch
 * (kda_chunk_fwd_segmented_workspace(B, H, T, d_k, d_v, n_seg)) exceeds that size is rejected with
 * KDA_ERR_UNSUPPORTED before anything is launched. The call makes no cudaMalloc, cudaFree or
 * other allocating call.
 *  - The first call on a device looks up the array's device address there (cudaGetSymbolAddress,
 *    with that device current); make that first call before any stream capture on the device.
 *  - All calls on a device share the one array, and it keeps the contents of the last call.
 *    Every byte a call reads from it is written earlier in the same call, so nothing needs
 *    clearing, but calls whose work overlaps on the GPU (different streams, or host threads
 *    without ordering) race on the array and give wrong results: order them on one stream.
 */
kda_status_t kda_chunk_fwd_segmented_noalloc(const void* q, const void* k, const void* v,
                                             const void* g, const void* beta, const float* S0,
                                             void* out, float* S_final, int B, int H, int T,
                                             int d_k, int d_v, int C, int n_seg,
                                             kda_dtype_t dtype, void* stream);

/*
 * Waits for the work queued on `stream` so far, then takes and clears the device-side status
 * word of the current device in one atomic exchange: returns the code latched there (KDA_OK if
 * nothing was latched), or KDA_ERR_CUDA if the wait failed. The word is one per device and is
 * shared by every stream: a code latched by a kernel on another stream is reported by whichever
 * call takes the word first (it is never lost, but it may be reported on another stream), and a
 * kernel still running on another stream may latch a code after this call returns.
 */
kda_status_t kda_sync_status(void* stream);

/*
 * Self-test of the device-side failure report. Launches one thread that waits, for at most
 * limit_ns nanoseconds of the GPU global timer, on an mbarrier that nothing completes, then
 * latches KDA_ERR_TIMEOUT in the status word the way a kernel does when one of its bounded
 * waits gives up, and returns. The next kda_sync_status(stream) reports KDA_ERR_TIMEOUT and
 * clears it; the context stays usable. Asynchronous on `stream`; returns KDA_ERR_INVALID_ARG
 * unless 0 < limit_ns <= 1e10, KDA_ERR_CUDA if the launch fails.
 */
kda_status_t kda_wait_selftest(unsigned long long limit_ns, void* stream);

/* Static, human-readable name of a status code. */
const char* kda_status_string(kda_status_t status);

/* Message describing the most recent failure on the calling thread ("" if none). */
const char* kda_last_error(void);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
