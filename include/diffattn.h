/*
 * diffattn.h — C ABI of libdiffattn.so, the differential-attention operator
 * for NVIDIA GB300 (sm_103a).
 *
 * Sources for what the operator computes (web pages on the method; title and
 * section as printed there):
 *   [P1] "Differential Transformer | ICLR 2025 Oral" (dainus.ai blog)
 *        - "Differential Attention: 빼기의 힘"  (the V1 formula)
 *        - "λ의 역할과 학습"                    (the lambda_init schedule)
 *        - "V2로의 진화"                         (V2 summary, memory-bound decode)
 *   [P2] "Differential Transformer V2" (pogovet.com summary)
 *        - §1 "DIFF V1에서 V2로 바뀐 핵심 구조" (V1 details; V2 structure)
 *        - §2 "빠른 디코딩과 표준 커널 호환성"  (decode: KV heads not increased)
 *        - §4 "RMS 정규화 제거와 차분 계수의 역할" (sigmoid gate, no RMSNorm)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named in a *_params struct are DEVICE pointers unless stated.
 *   The caller owns every buffer (inputs, outputs, optional saves and the
 *   workspace); the library never allocates, frees or synchronises (except
 *   diffattn_get_device_status, which synchronises the given stream).
 * - 4-D tensors are passed as da_t4: a base pointer plus the element strides
 *   of the batch (sb), sequence (sn) and head (sh) dimensions; the last
 *   (feature) dimension is contiguous.  bf16 tensors need 16-byte aligned
 *   base pointers and strides that are multiples of 8 elements.
 * - Every call returns a da_status and never throws.  Arguments are checked
 *   before anything is launched (null pointers, alignment, shapes the kernels
 *   support).  A failed launch returns DA_ERR_CUDA.  Errors that a kernel
 *   detects while running (a bounded wait that expired, an index check) are
 *   recorded in a device status word read by diffattn_get_device_status.
 * - Work is enqueued on the given CUDA stream (cudaStream_t passed as void*;
 *   NULL = the legacy default stream) and runs asynchronously.
 * - Causal masking means key j is visible to query i iff j <= i (queries and
 *   keys share one position axis).
 */
#ifndef DIFFATTN_H
#define DIFFATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DA_OK = 0,
  DA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment          */
  DA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head dim, dtype)    */
  DA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed           */
  DA_ERR_TIMEOUT = 4,      /* a kernel's bounded wait expired (device word)  */
  DA_ERR_BOUNDS = 5,       /* a kernel's index check failed (device word)    */
  DA_ERR_WORKSPACE = 6     /* workspace missing or smaller than required     */
} da_status;

typedef enum { DA_F32 = 0, DA_BF16 = 1 } da_dtype;

/* A [B, N, H, D] tensor: element (b, n, h, x) lives at
 * ptr + b*sb + n*sn + h*sh + x (in elements). */
typedef struct {
  void* ptr;
  int64_t sb, sn, sh;
} da_t4;

/* ------------------------------------------------------------------------ */
/* lambda_init(l) = 0.8 - 0.6 * exp(-0.3 * (l - 1)), l = 1-based layer index.
 * [P1] "λ의 역할과 학습".  Host function; returns NaN for l < 1. */
float diffattn_lambda_init(int layer);

/* ------------------------------------------------------------------------ */
/* V1 forward.  [P1] "Differential Attention: 빼기의 힘"; [P2] §1.
 *   lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init   (one scalar,
 *            computed on the device from the four vectors; never clamped)
 *   O      = (softmax(s Q1 K1^T) - lambda softmax(s Q2 K2^T)) V
 *   Y      = (1 - lambda_init) * w * O / sqrt(mean_k O_k^2 + rms_eps)
 * per (b, n, h), the mean over the V head dim d_v; w = rms_weight, the fixed
 * per-feature RMSNorm weight (fp32 [d_v], shared by heads; NULL = unit).
 * q1, q2, k1, k2: [B, N, H, d_qk]; v, out: [B, N, H, d_v]; all of `dtype`.
 * lq1, lk1, lq2, lk2: fp32 [d_qk].
 * Supported: dtype DA_BF16 with (d_qk, d_v) = (128, 256) or (64, 128);
 *            dtype DA_F32 with d_qk <= 128, d_v <= 256 (d_v % 32 == 0);
 *            causal (key j <= query i) or not.
 * Optional saves for the backward (NULL pointer = not written):
 *   lse1, lse2 (log-sum-exp of the scaled scores per row), rstd
 *   (1/sqrt(mean O^2 + eps)): fp32 [B, H, N] contiguous;
 *   o2 = softmax(s Q2 K2^T) V: [B, N, H, d_v] of `dtype`;
 *   lambda_out: fp32 [1].
 * workspace: diffattn_v1_fwd_workspace_size(...) bytes (for the bf16 path:
 * the work counter of its dynamic schedule, cleared by the call on the
 * stream, and one 64 KB slot per SM through which the two CTAs of a pair
 * exchange half of their outputs, about 10 MB on a 152-SM GPU; 0 for
 * DA_F32), 256-byte aligned, contents on entry irrelevant.  Calls that run
 * at the same time need workspaces of their own. */
typedef struct {
  int B, N, H, d_qk, d_v;
  da_dtype dtype;
  int causal;
  float softmax_scale;   /* <= 0 selects 1/sqrt(d_qk) */
  float lambda_init;
  float rms_eps;
  da_t4 q1, q2, k1, k2, v;
  const float *lq1, *lk1, *lq2, *lk2;
  da_t4 out;
  float *lse1, *lse2, *rstd;
  da_t4 o2;
  float* lambda_out;
  void* workspace;
  size_t workspace_bytes;
  const float* rms_weight;  /* fp32 [d_v]: the RMSNorm weight w (NULL = unit) */
} da_v1_fwd_params;

/* Workspace bytes diffattn_v1_fwd needs on the current device. */
size_t diffattn_v1_fwd_workspace_size(int B, int N, int H, int d_qk, int d_v, da_dtype dtype);
da_status diffattn_v1_fwd(const da_v1_fwd_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* V1 backward: gradients of the V1 forward with respect to q1, q2, k1, k2,
 * v and the four lambda vectors, given dY.  The pages state no backward; it
 * is the chain rule applied to the forward above ([P1] formula, [P2] §1):
 *   dO  = (c dY - Yhat mean(c dY * Yhat)) * rstd,   Yhat = Y / c, c = 1 - lambda_init
 *   dP  = dO V^T;  D1 = <dO, A1 V>;  D2 = <dO, A2 V>
 *   dS1 = A1 (dP - D1);  dS2 = -lambda A2 (dP - D2)
 *   dQt = s dSt Kt;  dKt = s dSt^T Qt;  dV = (A1 - lambda A2)^T dO
 *   dlambda = -sum <dO, A2 V>;  dlq1 = dlambda e^(lq1.lk1) lk1, ... .
 * Inputs: the forward's inputs, its output `out` (Y), `dout` (dY), and the
 * saves lse1, lse2, rstd, o2 written by diffattn_v1_fwd.  Outputs: dq1, dq2,
 * dk1, dk2 [B,N,H,d_qk], dv [B,N,H,d_v] (dtype), dlq1, dlk1, dlq2, dlk2 fp32
 * [d_qk] (overwritten).  rms_weight: the forward's RMSNorm weight (NULL =
 * unit); its entries must be nonzero, since the backward recovers the
 * normalised output as Y / ((1 - lambda_init) w).  Supported: DA_BF16,
 * (d_qk, d_v) = (128, 256) or
 * (64, 128), causal or not, either mode.
 * workspace: at least diffattn_v1_bwd_workspace_size(..., deterministic)
 * bytes, 256-byte aligned; its contents on entry do not matter.  (With
 * deterministic set, that size covers the slots of every tile pair, as a call
 * without the causal mask needs; a causal call uses about half of them.)
 * deterministic = 0: each key tile adds its dQ tile into an fp32 accumulator
 * (TMA reduce-add), so dQ1 / dQ2 may differ in the last bits between runs;
 * every other output is reproducible.  deterministic != 0: each key tile
 * stores its dQ tile into its own slot of the workspace and the finalize sums
 * the slots in ascending key-tile order, so every output is bitwise
 * reproducible; the workspace grows by about B*H*N^2/64 * 4 bytes per stream
 * (B*H*N^2/128 * 4 of them written by a causal call) and the call takes
 * longer. */
typedef struct {
  int B, N, H, d_qk, d_v;
  da_dtype dtype;
  int causal;
  float softmax_scale;
  float lambda_init;
  float rms_eps;
  da_t4 q1, q2, k1, k2, v;
  const float *lq1, *lk1, *lq2, *lk2;
  da_t4 out, dout;
  const float *lse1, *lse2, *rstd;
  da_t4 o2;
  da_t4 dq1, dq2, dk1, dk2, dv;
  float *dlq1, *dlk1, *dlq2, *dlk2;
  void* workspace;
  size_t workspace_bytes;
  int deterministic;
  const float* rms_weight;  /* fp32 [d_v], as given to the forward (NULL = unit) */
} da_v1_bwd_params;

size_t diffattn_v1_bwd_workspace_size(int B, int N, int H, int d_qk, int d_v, int deterministic);
da_status diffattn_v1_bwd(const da_v1_bwd_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* V1 decode.  [P1] "Differential Attention: 빼기의 힘" (the V1 formula) and
 * "V2로의 진화" (LLM decoding, memory-bound); [P2] §1 (per-head RMSNorm and
 * the (1 - lambda_init) scale).  One new token per sequence: for sequence b
 * the new token's K1, K2 and V rows are already stored at position
 * seqlens[b] - 1, and its queries q1, q2 attend to positions
 * 0 .. seqlens[b] - 1 of the two K caches and the shared V cache:
 *   O = (softmax(s q1 K1^T) - lambda softmax(s q2 K2^T)) V
 *   Y = (1 - lambda_init) w O / sqrt(mean_k O_k^2 + rms_eps)  (w: rms_weight)
 * with lambda from the four vectors as in diffattn_v1_fwd.
 * q1, q2: bf16 [B, H, d_qk] contiguous; k1_cache, k2_cache: bf16
 * [B, L_max, H, d_qk], v_cache: bf16 [B, L_max, H, d_v] (da_t4 strides);
 * seqlens: int32 [B] device, each in [1, L_max] (NULL = all L_max);
 * lq1, lk1, lq2, lk2: fp32 [d_qk]; out: bf16 [B, H, d_v] contiguous.
 * num_splits: key-range splits per (b, head); 0 = chosen by the library
 * (diffattn_v1_decode_num_splits).  Workspace: split partials,
 * diffattn_v1_decode_workspace_size bytes, 256-byte aligned.
 * Supported: (d_qk, d_v) = (128, 256) or (64, 128).  A sequence length
 * outside [1, L_max] is recorded as DA_ERR_BOUNDS in the device status word
 * and that row of out is written as zeros. */
typedef struct {
  int B, H, d_qk, d_v, L_max;
  float softmax_scale;   /* <= 0 selects 1/sqrt(d_qk) */
  float lambda_init;
  float rms_eps;
  const void* q1;
  const void* q2;
  da_t4 k1_cache, k2_cache, v_cache;
  const int* seqlens;
  const float *lq1, *lk1, *lq2, *lk2;
  void* out;
  int num_splits;
  void* workspace;
  size_t workspace_bytes;
  const float* rms_weight;  /* fp32 [d_v]: the RMSNorm weight w (NULL = unit) */
} da_v1_decode_params;

int diffattn_v1_decode_num_splits(int B, int H, int L_max);
size_t diffattn_v1_decode_workspace_size(int B, int H, int d_v, int L_max, int num_splits);
da_status diffattn_v1_decode(const da_v1_decode_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* V2 gate.  [P2] §1 and §4: a per-token, per-head coefficient projected from
 * the input X and passed through a sigmoid (no bias):
 *   gate[t, p] = sigmoid(sum_k x[t, k] * w_lambda[k, p])
 * x: bf16 [T, d_model], row stride x_stride (elements, multiple of 8);
 * w_lambda: bf16 [d_model, h] row-major contiguous; gate: fp32 [T, h]
 * contiguous.  Supported: d_model % 64 == 0, h <= 64. */
typedef struct {
  int T, d_model, h;
  const void* x;
  int64_t x_stride;
  const void* w_lambda;
  float* gate;
} da_v2_gate_params;

da_status diffattn_v2_gate(const da_v2_gate_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* V2 forward.  [P2] §1 and the one-line summary: one causal GQA attention
 * over 2h query heads with h_kv K/V heads; q head j reads K/V head
 * j / (2h / h_kv) (contiguous groups, so pair p = heads 2p and 2p+1 always
 * shares one K/V head); then per token t and pair p
 *   out[t, p] = O[t, 2p] - gate[t, p] * O[t, 2p + 1]
 * which brings the width back to h * d.  No normalisation ([P2] §4).
 * q: [B, N, 2h, d]; k, v: [B, N, h_kv, d]; out: [B, N, h, d]; all bf16.
 * Gate source: either `gate` (fp32 [B, N, h] contiguous, already through the
 * sigmoid) or, when gate == NULL, x (bf16 [B, N, d_model] contiguous) and
 * w_lambda (bf16 [d_model, h]); the gate is then computed into the workspace
 * (diffattn_v2_fwd_workspace_size bytes).
 * Optional saves for diffattn_v2_bwd (NULL pointer = not written): lse, fp32
 * [B, 2h, N] contiguous (natural-log log-sum-exp of each head's scaled scores
 * per query); o_heads, bf16 [B, N, 2h, d] (each head's normalised output
 * O[t, j] before the even/odd combination).
 * Supported: d = 64 or 128, causal or not, (2h / h_kv) even. */
typedef struct {
  int B, N, h, h_kv, d, d_model;
  int causal;
  float softmax_scale;   /* <= 0 selects 1/sqrt(d) */
  da_t4 q, k, v;
  const float* gate;
  const void* x;
  const void* w_lambda;
  da_t4 out;
  float* lse;
  da_t4 o_heads;
  void* workspace;
  size_t workspace_bytes;
} da_v2_fwd_params;

size_t diffattn_v2_fwd_workspace_size(int B, int N, int h, int gate_given);
da_status diffattn_v2_fwd(const da_v2_fwd_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* Grouped differential attention, forward.  [P1] "같은 문제, 다른 접근" names
 * the follow-up that gives signal heads and noise heads an uneven share (3:1
 * or 4:1) and says nothing more; the reading implemented here is the V2 form
 * ([P2] §1): one causal GQA attention over Hq = h (ratio + 1) / ratio query
 * heads that come in groups of `ratio` signal heads followed by one noise
 * head, every group inside one K/V group, and per token t and output head p
 * of group g = p / ratio, i = p mod ratio:
 *   out[t, p] = O[t, g (ratio+1) + i] - gate[t, p] * O[t, g (ratio+1) + ratio]
 * With ratio 1 this is diffattn_v2_fwd's result.
 * q: [B, N, Hq, d]; k, v: [B, N, h_kv, d]; out: [B, N, h, d]; all bf16.
 * Gate source as in diffattn_v2_fwd (fp32 [B, N, h], or x + w_lambda with
 * w_lambda [d_model, h]).  Optional saves: lse fp32 [B, Hq, N]; o_heads bf16
 * [B, N, Hq, d] (each head's normalised output; when NULL the per-head
 * outputs go to the workspace).  Supported: d = 64 or 128, causal or not,
 * h divisible by ratio, Hq / h_kv a multiple of ratio + 1 and even.
 * workspace: diffattn_grouped_fwd_workspace_size bytes, 256-byte aligned. */
typedef struct {
  int B, N, h, ratio, h_kv, d, d_model;
  int causal;
  float softmax_scale;   /* <= 0 selects 1/sqrt(d) */
  da_t4 q, k, v;
  const float* gate;
  const void* x;
  const void* w_lambda;
  da_t4 out;
  float* lse;
  da_t4 o_heads;
  void* workspace;
  size_t workspace_bytes;
} da_grouped_fwd_params;

size_t diffattn_grouped_fwd_workspace_size(int B, int N, int h, int ratio, int d, int gate_given,
                                           int heads_given);
da_status diffattn_grouped_fwd(const da_grouped_fwd_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* V2 backward: gradients of diffattn_v2_fwd (and of the gate projection)
 * given dOut.  The pages state no backward; it is the chain rule of the V2
 * forward ([P2] §1, §4).  With g = sigmoid(z), z[t, p] = x[t] . w_lambda[:, p],
 * G = dOut[t, p] and O_j the normalised output of query head j:
 *   dO_2p = G,  dO_2p+1 = -g G,  dz = -<G, O_2p+1> g (1 - g)
 *   dW_lambda = X^T dz,  dX (the part through the gate) = dz W_lambda^T
 *   per query head j reading K/V head c:  A = softmax(s Q_j K_c^T) (causal),
 *   dP = dO_j V_c^T,  dS = A (dP - <dO_j, O_j>),
 *   dQ_j = s dS K_c,  dK_c += s dS^T Q_j,  dV_c += A^T dO_j
 * (dK and dV sum over every query head of the K/V group).
 * Inputs: the forward's q, k, v (as in diffattn_v2_fwd), the gate source
 * (`gate`, or x and w_lambda when gate == NULL), the forward's saves
 * `o_heads` and `lse`, and dout: bf16 [B, N, h, d].
 * Outputs (overwritten): dq [B, N, 2h, d], dk, dv [B, N, h_kv, d], bf16.
 * Optional outputs (NULL = not computed): dgate_logit fp32 [B, N, h]
 * contiguous (dz); dx bf16 [B, N, d_model] contiguous and dw_lambda fp32
 * [d_model, h] row-major, both of which need x and w_lambda.
 * Supported: d = 64 or 128, causal or not, (2h / h_kv) even;
 * d_model % 64 == 0 and h <= 64 where x / w_lambda are used.
 * workspace: diffattn_v2_bwd_workspace_size(B, N, h, d_model) bytes (with
 * d_model = 0 it covers calls that do not request dw_lambda), 256-byte
 * aligned, contents on entry irrelevant. */
typedef struct {
  int B, N, h, h_kv, d, d_model;
  int causal;
  float softmax_scale;   /* <= 0 selects 1/sqrt(d) */
  da_t4 q, k, v;
  const float* gate;
  const void* x;
  const void* w_lambda;
  da_t4 o_heads;
  const float* lse;
  da_t4 dout;
  da_t4 dq, dk, dv;
  float* dgate_logit;
  void* dx;
  float* dw_lambda;
  void* workspace;
  size_t workspace_bytes;
} da_v2_bwd_params;

size_t diffattn_v2_bwd_workspace_size(int B, int N, int h, int d_model);
da_status diffattn_v2_bwd(const da_v2_bwd_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* Grouped differential attention, backward: gradients of diffattn_grouped_fwd
 * (and of the gate projection) given dOut.  The pages state no backward; it
 * is the chain rule of the grouped forward above.  With r = ratio, output
 * head p = g r + i reading signal query head g (r+1) + i and noise query head
 * g (r+1) + r, gate[t, p] = sigmoid(z), G = dOut[t, p]:
 *   dO_signal(p) = G_p,  dO_noise(g) = -sum_i gate[t, g r + i] G_{g r + i}
 *   dz_p = -<G_p, O_noise(g)> gate (1 - gate),  dW_lambda = X^T dz,  dX = dz W_lambda^T
 *   per query head j reading K/V head c: as in diffattn_v2_bwd.
 * With ratio 1 this is diffattn_v2_bwd's result.
 * Inputs: the forward's q, k, v, the gate source (gate fp32 [B, N, h], or x
 * and w_lambda [d_model, h] when gate == NULL), the forward's saves o_heads
 * (bf16 [B, N, Hq, d], required here) and lse (fp32 [B, Hq, N]), and dout
 * (bf16 [B, N, h, d]).  Outputs (overwritten): dq [B, N, Hq, d], dk, dv
 * [B, N, h_kv, d], bf16.  Optional outputs (NULL = not computed):
 * dgate_logit fp32 [B, N, h] (dz); dx bf16 [B, N, d_model] and dw_lambda fp32
 * [d_model, h] (these need x and w_lambda).  Supported: the shapes of
 * diffattn_grouped_fwd; d_model % 64 == 0 and h <= 64 where x / w_lambda are
 * used.  workspace: diffattn_grouped_bwd_workspace_size(B, N, h, ratio,
 * d_model) bytes (d_model = 0 covers calls without dw_lambda), 256-byte
 * aligned, contents on entry irrelevant.  dQ is accumulated with fp32
 * reduce-adds (not bitwise reproducible); every other output is. */
typedef struct {
  int B, N, h, ratio, h_kv, d, d_model;
  int causal;
  float softmax_scale;   /* <= 0 selects 1/sqrt(d) */
  da_t4 q, k, v;
  const float* gate;
  const void* x;
  const void* w_lambda;
  da_t4 o_heads;
  const float* lse;
  da_t4 dout;
  da_t4 dq, dk, dv;
  float* dgate_logit;
  void* dx;
  float* dw_lambda;
  void* workspace;
  size_t workspace_bytes;
} da_grouped_bwd_params;

size_t diffattn_grouped_bwd_workspace_size(int B, int N, int h, int ratio, int d_model);
da_status diffattn_grouped_bwd(const da_grouped_bwd_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* V2 decode.  [P1] "V2로의 진화" and [P2] §2: one new token per sequence
 * attends over its KV cache; the KV heads and cache are those of a standard
 * GQA model (only the query heads double), so the step is bound by reading
 * the cache.  For sequence b the new token is already stored at position
 * seqlens[b] - 1 and attends to positions 0 .. seqlens[b] - 1; then the
 * even/odd combination with the gate as in diffattn_v2_fwd.
 * q: bf16 [B, 2h, d] contiguous; k_cache, v_cache: bf16 [B, L_max, h_kv, d]
 * (da_t4 strides; position stride sn); seqlens: int32 [B] device, each in
 * [1, L_max] (NULL = all L_max); gate fp32 [B, h] or x bf16 [B, d_model] +
 * w_lambda as in diffattn_v2_fwd; out: bf16 [B, h, d] contiguous.
 * num_splits: key-range splits per (b, kv head); 0 = chosen by the library
 * (diffattn_v2_decode_num_splits).  Workspace: split partials,
 * diffattn_v2_decode_workspace_size bytes.  Supported: d = 64 or 128,
 * 2 <= 2h / h_kv <= 16 and even.  A sequence length outside [1, L_max] is
 * recorded as DA_ERR_BOUNDS in the device status word and its output row is
 * written as zeros. */
typedef struct {
  int B, h, h_kv, d, L_max, d_model;
  float softmax_scale;   /* <= 0 selects 1/sqrt(d) */
  const void* q;
  da_t4 k_cache, v_cache;
  const int* seqlens;
  const float* gate;
  const void* x;
  const void* w_lambda;
  void* out;
  int num_splits;
  void* workspace;
  size_t workspace_bytes;
} da_v2_decode_params;

int diffattn_v2_decode_num_splits(int B, int h_kv, int L_max);
size_t diffattn_v2_decode_workspace_size(int B, int h, int h_kv, int d,
                                         int L_max, int num_splits,
                                         int gate_given);
da_status diffattn_v2_decode(const da_v2_decode_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* V2 decode that allocates nothing and takes no workspace.  The method pages
 * have no counterpart: this is a service for callers that cannot allocate
 * device memory at all — an inference runtime that carves its memory once at
 * start-up and forbids allocation inside the token loop, a program driving
 * the GPU through a context it does not own, a plugin whose host framework
 * hands it inputs and outputs but no scratch buffers.
 *
 * Same parameters and result as diffattn_v2_decode; `workspace` and
 * `workspace_bytes` are ignored.  The split partials (and the gate, when it
 * is computed from x) go to one fixed device array of
 * DIFFATTN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library keeps until the process exits.  With num_splits = 0 the
 * usual split count is lowered until the partials fit; a problem that needs
 * more than the array even with one split (or an explicit num_splits that
 * does not fit) returns DA_ERR_WORKSPACE without launching — use
 * diffattn_v2_decode with a workspace for those.
 *
 * The first call on a device looks up the array's device address once (a
 * CUDA runtime query with that device current); make that first call before
 * any stream capture begins.  The address stays cached for the life of the
 * process, so do not call the library again after a cudaDeviceReset (the
 * same holds for every entry point: the device status word's address is
 * cached the same way).  Shape errors are reported as by
 * diffattn_v2_decode, before the size check.  All calls share the array and each call
 * overwrites what the previous one left there (nothing needs to start at
 * zero), so calls that may overlap on the GPU — other streams, other host
 * threads — race and must be serialised by the caller. */
#define DIFFATTN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
da_status diffattn_v2_decode_noalloc(const da_v2_decode_params* p, void* cuda_stream);

/* ------------------------------------------------------------------------ */
/* Device status word.  Kernels record the first error they detect (a bounded
 * wait that expired, a failed index check) in a per-device word instead of
 * trapping.  diffattn_get_device_status synchronises `cuda_stream`, returns
 * the recorded status (DA_OK if none) and clears the word.
 * diffattn_get_device_status_detail additionally returns the raw word
 * (status in the low byte, a kernel-specific site code above it).
 * The word's device address is looked up once per device and cached for the
 * life of the process: after a cudaDeviceReset the library must not be used
 * again in that process. */
da_status diffattn_get_device_status(void* cuda_stream);
da_status diffattn_get_device_status_detail(void* cuda_stream, uint32_t* raw);

const char* diffattn_status_string(da_status s);

/* ------------------------------------------------------------------------ */
/* Test hook for the failure path of the bounded waits.  Every mbarrier wait
 * in the tcgen05 kernels gives up after about 2 s, records DA_ERR_TIMEOUT
 * (with a site code) in the device status word, raises a per-CTA abort flag
 * so that the CTA's other roles leave their loops, lets its own in-flight
 * copies land and frees its TMEM before returning; the context stays usable.
 * DA_FAULT_V2_FWD_SKIP_LOAD makes the NEXT diffattn_v2_fwd call (only that
 * one) leave the first K tile of its first CTA unloaded, so the wait for it
 * expires: that call's outputs are incomplete, diffattn_get_device_status
 * then returns DA_ERR_TIMEOUT, and later calls run normally.
 * DA_FAULT_NONE cancels a pending injection.  Returns DA_ERR_INVALID_ARG for
 * any other value.  Host-side state of the library (not per device). */
typedef enum { DA_FAULT_NONE = 0, DA_FAULT_V2_FWD_SKIP_LOAD = 1 } da_fault;
da_status diffattn_debug_inject_fault(int fault);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H */
