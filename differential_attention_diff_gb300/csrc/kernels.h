// kernels.h — internal launch interface between api.cu (argument checks,
// workspace carving, stream handling) and the kernel translation units.
// Every launcher returns a cudaError_t from the launch itself.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "diffattn.h"

namespace da {

// ---- V2 gate: gate[t, p] = sigmoid(x[t, :] . w[:, p]) ---------------------
struct GateArgs {
  int T, d_model, h;
  const void* x;
  int64_t x_stride;
  const void* w;
  float* gate;
  uint32_t* status;  // device status word for bounded waits (may be null)
};
cudaError_t launch_gate(const GateArgs& a, cudaStream_t s);
// dX = dz W^T of the gate projection on tensor cores (gate_grads.cu), for
// T >= 128, h <= 64 with h % 8 == 0, d_model % 64 == 0
bool gate_dx_tc_ok(int T, int d_model, int h);
// partial sums of dW = X^T dz per chunk of chunk_tokens tokens (a multiple of
// 64) on tensor cores, part = fp32 [chunks][d_model][h]; for T >= 64, h <= 64
// with h % 8 == 0, d_model % 128 == 0
bool gate_dw_tc_ok(int T, int d_model, int h);
cudaError_t launch_gate_dw_tc(int T, int d_model, int h, int chunk_tokens, int chunks, const float* dz, const void* X,
                              float* part, uint32_t* status, cudaStream_t s);
cudaError_t launch_gate_dx_tc(int T, int d_model, int h, const float* dz, const void* W, void* dx, uint32_t* status,
                              cudaStream_t s);

// ---- V2 decode: split-KV partials, then merge + even/odd gate ------------
struct DecodeArgs {
  int B, h, h_kv, d, L_max, num_splits;
  float scale_log2;  // softmax scale * log2(e)
  const void* q;
  da_t4 k, v;
  const int* seqlens;
  const float* gate;  // [B, h]
  void* out;          // bf16 [B, h, d]
  float* part_o;      // [splits, B, 2h, d]
  float* part_ml;     // [splits, B, 2h, 2]  (running max in log2 units, sum)
  uint32_t* status;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
// The split count is a grid dimension (at most 65535).
constexpr int kMaxDecodeSplits = 65535;
// Every argument check of diffattn_v2_decode except the split count chosen
// by the library and the workspace; DA_OK or the status the call returns.
da_status check_v2_decode_args(const da_v2_decode_params* p);

// ---- V1 decode: split-KV partials of both streams, then merge + RMSNorm ----
struct V1DecodeArgs {
  int B, H, d_qk, d_v, L_max, num_splits;  // (d_qk, d_v) = (128, 256) or (64, 128)
  float scale_log2, lambda_init, rms_eps;
  const void* q1;  // bf16 [B, H, d_qk]
  const void* q2;
  da_t4 k1, k2, v;  // [B, L_max, H, d_qk | d_qk | d_v]
  const int* seqlens;
  const float *lq1, *lk1, *lq2, *lk2;
  void* out;       // bf16 [B, H, d_v]
  float* part_o;   // [splits, B, H, 2, d_v]
  float* part_ml;  // [splits, B, H, 2, 2]  (running max in log2 units, sum)
  uint32_t* status;
  const float* rms_weight;  // [d_v] or nullptr (unit)
};
cudaError_t launch_v1_decode(const V1DecodeArgs& a, cudaStream_t s);

// ---- V1 forward, fp32 SIMT path ------------------------------------------
struct V1F32Args {
  int B, N, H, d_qk, d_v, causal;
  float scale, lambda_init, rms_eps;
  da_t4 q1, q2, k1, k2, v, out, o2;
  const float *lq1, *lk1, *lq2, *lk2;
  float *lse1, *lse2, *rstd, *lambda_out;
  const float* rms_weight;  // [d_v] or nullptr (unit)
};
cudaError_t launch_v1_fwd_f32(const V1F32Args& a, cudaStream_t s);

// ---- V2 forward, tcgen05 -------------------------------------------------
struct V2FwdArgs {
  int B, N, h, h_kv, d, causal;
  float scale_log2;
  da_t4 q, k, v, out;
  const float* gate;  // [B, N, h]
  float* lse;         // optional [B, 2h, N] (natural log)
  da_t4 o_heads;      // optional [B, N, 2h, d] per-head outputs
  uint32_t* status;
  int num_sms;
  int fault;          // test hook: CTA 0 skips its first K tile load
};
cudaError_t launch_v2_fwd(const V2FwdArgs& a, cudaStream_t s);

// ---- grouped differential attention: combine per-head outputs -------------
struct GroupedArgs {
  int B, N, h, ratio;   // h output (signal) heads, ratio signal heads per noise head
  int d;                // head dim (a multiple of 8)
  da_t4 o_heads;        // [B, N, h (ratio + 1) / ratio, d] bf16
  const float* gate;    // [B, N, h]
  da_t4 out;            // [B, N, h, d] bf16
};
cudaError_t launch_grouped_combine(const GroupedArgs& a, cudaStream_t s);

// ---- V2 backward, bf16, tcgen05 --------------------------------------------
struct V2BwdArgs {
  int B, N, h, h_kv, d, d_model, causal;
  float scale;
  da_t4 q, k, v, o_heads, dout, dq, dk, dv;
  const float* gate;   // [B, N, h], or NULL: computed from x, w into the workspace
  const float* lse;    // [B, 2h, N] natural log
  const void* x;       // bf16 [B, N, d_model] (optional)
  const void* w;       // bf16 [d_model, h] (optional)
  float* dz;           // optional [B, N, h] output (else kept in the workspace)
  void* dx;            // optional bf16 [B, N, d_model]
  float* dw;           // optional fp32 [d_model, h]
  void* workspace;
  size_t workspace_bytes;
  uint32_t* status;
  int num_sms;
  // Grouped differential attention (ratio >= 2): the 2h query heads come in
  // groups of `ratio` signal heads and one noise head; dout, gate, dz, w and
  // dw have h_out = 2h ratio / (ratio + 1) output heads.  ratio <= 1 is V2
  // (h_out = h, even/odd pairs).
  int ratio;
  int h_out;
};
size_t v2_bwd_workspace_bytes(int B, int N, int h, int d_model);
// grouped: h_attn = Hq / 2 (half the query heads), h_out = the output heads
size_t grouped_bwd_workspace_bytes(int B, int N, int h_attn, int h_out, int d_model);
cudaError_t launch_v2_bwd(const V2BwdArgs& a, cudaStream_t s);

// ---- V1 forward, bf16, tcgen05 ---------------------------------------------
struct V1FwdArgs {
  int B, N, H, d_qk, d_v, causal;
  float scale_log2, lambda_init, rms_eps;
  da_t4 q1, q2, k1, k2, v, out, o2;
  const float *lq1, *lk1, *lq2, *lk2;
  float *lse1, *lse2, *rstd, *lambda_out;
  void* workspace;  // exchange slots of the CTA pairs
  size_t workspace_bytes;
  uint32_t* status;
  int num_sms;
  const float* rms_weight;  // [d_v] or nullptr (unit)
};
size_t v1_fwd_workspace_bytes(int num_sms);
cudaError_t launch_v1_fwd(const V1FwdArgs& a, cudaStream_t s);

// ---- V1 backward, bf16 -----------------------------------------------------
struct V1BwdArgs {
  int B, N, H, d_qk, d_v, causal;
  float scale, lambda_init, rms_eps;
  da_t4 q1, q2, k1, k2, v, out, dout, o2;
  const float *lq1, *lk1, *lq2, *lk2;
  const float *lse1, *lse2, *rstd;
  da_t4 dq1, dq2, dk1, dk2, dv;
  float *dlq1, *dlk1, *dlq2, *dlk2;
  void* workspace;
  size_t workspace_bytes;
  uint32_t* status;
  int num_sms;
  int deterministic;  // dQ through per-key-tile slots summed in a fixed order
  const float* rms_weight;  // [d_v] or nullptr (unit); entries nonzero
};
// deterministic dQ slots: the causal tile pairs when causal, all pairs otherwise
size_t v1_bwd_workspace_bytes(int B, int N, int H, int d_qk, int d_v, int deterministic, int causal);
cudaError_t launch_v1_bwd(const V1BwdArgs& a, cudaStream_t s);

// TMA descriptor encoding (driver entry point fetched through the runtime).
bool tma_available();

}  // namespace da
