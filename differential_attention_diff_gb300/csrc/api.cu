// api.cu — the extern "C" entry points of libdiffattn.so: argument checks,
// workspace carving, the per-device status word, and the launches.  No entry
// point allocates, frees or synchronises (diffattn_get_device_status
// synchronises the stream it is given, by its contract).
#include <cuda_runtime.h>

#include <cmath>
#include <atomic>
#include <mutex>

#include "diffattn.h"
#include "kernels.h"

namespace {

// Per-device status word (first error wins; see record_status).
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

struct DevInfo {
  uint32_t* status = nullptr;
  int num_sms = 0;
  bool ok = false;
};

DevInfo device_info() {
  DevInfo info;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return info;
  std::call_once(g_dev_once[dev], [dev]() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess)
      g_status_ptr[dev] = static_cast<uint32_t*>(p);
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      g_num_sms[dev] = sms;
  });
  info.status = g_status_ptr[dev];
  info.num_sms = g_num_sms[dev];
  info.ok = info.status != nullptr && info.num_sms > 0;
  return info;
}

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// A [B, N, H, D] operand: non-null, non-negative strides; bf16 operands go
// through TMA or 16-byte vector copies, so base and strides must be 16-byte
// multiples.
da_status check_t4(const da_t4& t, da_dtype dt) {
  if (t.ptr == nullptr) return DA_ERR_INVALID_ARG;
  if (t.sb < 0 || t.sn < 0 || t.sh < 0) return DA_ERR_INVALID_ARG;
  if (dt == DA_BF16) {
    if (!aligned(t.ptr, 16)) return DA_ERR_INVALID_ARG;
    if ((t.sb % 8) || (t.sn % 8) || (t.sh % 8)) return DA_ERR_INVALID_ARG;
  } else {
    if (!aligned(t.ptr, 4)) return DA_ERR_INVALID_ARG;
  }
  return DA_OK;
}

da_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DA_OK : DA_ERR_CUDA; }

// One-shot test hook (diffattn_debug_inject_fault): consumed by the next call
// it applies to.
std::atomic<int> g_fault{0};

constexpr float kLog2e = 1.4426950408889634f;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" {

float diffattn_lambda_init(int layer) {
  if (layer < 1) return NAN;
  return static_cast<float>(0.8 - 0.6 * std::exp(-0.3 * (static_cast<double>(layer) - 1.0)));
}

const char* diffattn_status_string(da_status s) {
  switch (s) {
    case DA_OK: return "ok";
    case DA_ERR_INVALID_ARG: return "invalid argument";
    case DA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case DA_ERR_CUDA: return "CUDA error";
    case DA_ERR_TIMEOUT: return "device wait timed out";
    case DA_ERR_BOUNDS: return "device index check failed";
    case DA_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

da_status diffattn_get_device_status_detail(void* stream, uint32_t* raw) {
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0, zero = 0;
  if (cudaMemcpyAsync(&word, d.status, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DA_ERR_CUDA;
  if (cudaMemcpyAsync(d.status, &zero, sizeof(zero), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DA_ERR_CUDA;
  if (raw) *raw = word;
  return static_cast<da_status>(word & 0xffu);
}

da_status diffattn_debug_inject_fault(int fault) {
  if (fault != DA_FAULT_NONE && fault != DA_FAULT_V2_FWD_SKIP_LOAD) return DA_ERR_INVALID_ARG;
  g_fault.store(fault);
  return DA_OK;
}

da_status diffattn_get_device_status(void* stream) {
  return diffattn_get_device_status_detail(stream, nullptr);
}

// --------------------------------------------------------------- gate ------
da_status diffattn_v2_gate(const da_v2_gate_params* p, void* stream) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->T < 0 || p->d_model <= 0 || p->h <= 0) return DA_ERR_INVALID_ARG;
  if (p->T == 0) return DA_OK;
  if (!p->x || !p->w_lambda || !p->gate) return DA_ERR_INVALID_ARG;
  if (!aligned(p->x, 16) || !aligned(p->w_lambda, 16) || !aligned(p->gate, 4))
    return DA_ERR_INVALID_ARG;
  if (p->x_stride < p->d_model || (p->x_stride % 8)) return DA_ERR_INVALID_ARG;
  if ((p->d_model % 64) || p->h > 64) return DA_ERR_UNSUPPORTED;
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  da::GateArgs a{p->T, p->d_model, p->h, p->x, p->x_stride, p->w_lambda, p->gate, d.status};
  return cuda_status(da::launch_gate(a, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------- decode ------
int diffattn_v2_decode_num_splits(int B, int h_kv, int L_max) {
  if (B <= 0 || h_kv <= 0 || L_max <= 0) return 1;
  // Enough CTAs for about 12 waves of the one resident CTA per SM (longer
  // splits stream better; 12 measured best at B64 L32768 among 8-32), but
  // no split shorter than 1024 keys (8 tiles).
  int sms = 152;
  DevInfo d = device_info();
  if (d.ok) sms = d.num_sms;
  const long units = static_cast<long>(B) * h_kv;
  long s = (12L * sms + units - 1) / units;
  const long max_s = (L_max + 1023) / 1024;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

size_t diffattn_v2_decode_workspace_size(int B, int h, int h_kv, int d, int L_max,
                                         int num_splits, int gate_given) {
  if (B <= 0 || h <= 0 || d <= 0) return 0;
  if (num_splits <= 0) num_splits = diffattn_v2_decode_num_splits(B, h_kv, L_max);
  const size_t po = static_cast<size_t>(num_splits) * B * 2 * h * d * sizeof(float);
  const size_t pml = static_cast<size_t>(num_splits) * B * 2 * h * 2 * sizeof(float);
  const size_t g = gate_given ? 0 : static_cast<size_t>(B) * h * sizeof(float);
  return align256(po) + align256(pml) + align256(g);
}

}  // extern "C"

// Every check of a V2 decode call except those of the split count and the
// workspace (shared with the entry point that brings its own scratch).
da_status da::check_v2_decode_args(const da_v2_decode_params* p) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->B <= 0 || p->h <= 0 || p->h_kv <= 0 || p->d <= 0 || p->L_max <= 0)
    return DA_ERR_INVALID_ARG;
  if ((2 * p->h) % p->h_kv) return DA_ERR_INVALID_ARG;
  const int G = 2 * p->h / p->h_kv;
  if (G % 2) return DA_ERR_INVALID_ARG;  // a pair must sit in one K/V group
  if ((p->d != 64 && p->d != 128) || G > 16) return DA_ERR_UNSUPPORTED;
  if (!p->q || !p->out || !aligned(p->q, 16) || !aligned(p->out, 16)) return DA_ERR_INVALID_ARG;
  if (check_t4(p->k_cache, DA_BF16) != DA_OK || check_t4(p->v_cache, DA_BF16) != DA_OK)
    return DA_ERR_INVALID_ARG;
  if (p->gate == nullptr) {
    if (!p->x || !p->w_lambda || p->d_model <= 0) return DA_ERR_INVALID_ARG;
    if ((p->d_model % 64) || p->h > 64) return DA_ERR_UNSUPPORTED;
  } else if (!aligned(p->gate, 4)) {
    return DA_ERR_INVALID_ARG;
  }
  if (p->num_splits > da::kMaxDecodeSplits) return DA_ERR_INVALID_ARG;
  return DA_OK;
}

extern "C" {

da_status diffattn_v2_decode(const da_v2_decode_params* p, void* stream) {
  const da_status chk = da::check_v2_decode_args(p);
  if (chk != DA_OK) return chk;
  const int splits = p->num_splits > 0 ? p->num_splits
                                       : diffattn_v2_decode_num_splits(p->B, p->h_kv, p->L_max);
  if (splits > da::kMaxDecodeSplits) return DA_ERR_INVALID_ARG;
  const size_t need = diffattn_v2_decode_workspace_size(p->B, p->h, p->h_kv, p->d, p->L_max,
                                                        splits, p->gate != nullptr);
  if (p->workspace == nullptr || p->workspace_bytes < need || !aligned(p->workspace, 256))
    return DA_ERR_WORKSPACE;
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  uint8_t* ws = static_cast<uint8_t*>(p->workspace);
  const size_t po = static_cast<size_t>(splits) * p->B * 2 * p->h * p->d * sizeof(float);
  const size_t pml = static_cast<size_t>(splits) * p->B * 2 * p->h * 2 * sizeof(float);
  float* part_o = reinterpret_cast<float*>(ws);
  float* part_ml = reinterpret_cast<float*>(ws + align256(po));
  const float* gate = p->gate;
  if (gate == nullptr) {
    float* g = reinterpret_cast<float*>(ws + align256(po) + align256(pml));
    da::GateArgs ga{p->B, p->d_model, p->h, p->x, p->d_model, p->w_lambda, g, d.status};
    cudaError_t e = da::launch_gate(ga, s);
    if (e != cudaSuccess) return DA_ERR_CUDA;
    gate = g;
  }
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.f / std::sqrt(static_cast<float>(p->d));
  da::DecodeArgs a{p->B, p->h, p->h_kv, p->d, p->L_max, splits, scale * kLog2e,
                   p->q, p->k_cache, p->v_cache, p->seqlens, gate, p->out,
                   part_o, part_ml, d.status};
  return cuda_status(da::launch_decode(a, s));
}

// ----------------------------------------------------------- V1 fwd --------
size_t diffattn_v1_fwd_workspace_size(int B, int N, int H, int d_qk, int d_v, da_dtype dtype) {
  if (dtype != DA_BF16 || B <= 0 || N <= 0 || H <= 0 || d_qk <= 0 || d_v <= 0) return 0;
  DevInfo d = device_info();
  const size_t n = da::v1_fwd_workspace_bytes(d.ok ? d.num_sms : 0);
  return n ? align256(n) : 0;
}

da_status diffattn_v1_fwd(const da_v1_fwd_params* p, void* stream) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->B < 0 || p->N < 0 || p->H < 0 || p->d_qk <= 0 || p->d_v <= 0) return DA_ERR_INVALID_ARG;
  if (p->dtype != DA_F32 && p->dtype != DA_BF16) return DA_ERR_INVALID_ARG;
  if (!(p->rms_eps >= 0.f)) return DA_ERR_INVALID_ARG;
  if (!p->lq1 || !p->lk1 || !p->lq2 || !p->lk2) return DA_ERR_INVALID_ARG;
  if (p->rms_weight && !aligned(p->rms_weight, 4)) return DA_ERR_INVALID_ARG;
  if (p->B == 0 || p->N == 0 || p->H == 0) return DA_OK;
  for (const da_t4* t : {&p->q1, &p->q2, &p->k1, &p->k2, &p->v, &p->out})
    if (check_t4(*t, p->dtype) != DA_OK) return DA_ERR_INVALID_ARG;
  if (p->o2.ptr && check_t4(p->o2, p->dtype) != DA_OK) return DA_ERR_INVALID_ARG;
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale
                                             : 1.f / std::sqrt(static_cast<float>(p->d_qk));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  if (p->dtype == DA_F32) {
    if (p->d_qk > 128 || p->d_v > 256 || (p->d_v % 32)) return DA_ERR_UNSUPPORTED;
    da::V1F32Args a{p->B, p->N, p->H, p->d_qk, p->d_v, p->causal, scale, p->lambda_init,
                    p->rms_eps, p->q1, p->q2, p->k1, p->k2, p->v, p->out, p->o2,
                    p->lq1, p->lk1, p->lq2, p->lk2, p->lse1, p->lse2, p->rstd, p->lambda_out,
                    p->rms_weight};
    return cuda_status(da::launch_v1_fwd_f32(a, s));
  }
  if (!((p->d_qk == 128 && p->d_v == 256) || (p->d_qk == 64 && p->d_v == 128))) return DA_ERR_UNSUPPORTED;
  const size_t need = da::v1_fwd_workspace_bytes(d.num_sms);
  if (need && (p->workspace == nullptr || p->workspace_bytes < need || !aligned(p->workspace, 256)))
    return DA_ERR_WORKSPACE;
  if (!da::tma_available()) return DA_ERR_CUDA;
  da::V1FwdArgs a{p->B, p->N, p->H, p->d_qk, p->d_v, p->causal, scale * kLog2e,
                  p->lambda_init, p->rms_eps, p->q1, p->q2, p->k1, p->k2, p->v,
                  p->out, p->o2, p->lq1, p->lk1, p->lq2, p->lk2, p->lse1, p->lse2,
                  p->rstd, p->lambda_out, p->workspace, p->workspace_bytes, d.status,
                  d.num_sms, p->rms_weight};
  return cuda_status(da::launch_v1_fwd(a, s));
}

// ----------------------------------------------------------- V1 bwd --------
size_t diffattn_v1_bwd_workspace_size(int B, int N, int H, int d_qk, int d_v, int deterministic) {
  if (B <= 0 || N <= 0 || H <= 0) return 0;
  // without the mask flag, size for every (key tile, query tile) pair: enough
  // for a causal call too
  return da::v1_bwd_workspace_bytes(B, N, H, d_qk, d_v, deterministic != 0, 0);
}

da_status diffattn_v1_bwd(const da_v1_bwd_params* p, void* stream) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->B < 0 || p->N < 0 || p->H < 0 || p->d_qk <= 0 || p->d_v <= 0) return DA_ERR_INVALID_ARG;
  if (p->dtype != DA_BF16 && p->dtype != DA_F32) return DA_ERR_INVALID_ARG;
  if (!p->lq1 || !p->lk1 || !p->lq2 || !p->lk2) return DA_ERR_INVALID_ARG;
  if (!p->dlq1 || !p->dlk1 || !p->dlq2 || !p->dlk2) return DA_ERR_INVALID_ARG;
  if (p->rms_weight && !aligned(p->rms_weight, 4)) return DA_ERR_INVALID_ARG;
  if (p->B == 0 || p->N == 0 || p->H == 0) return DA_OK;
  if (p->dtype != DA_BF16 || !((p->d_qk == 128 && p->d_v == 256) || (p->d_qk == 64 && p->d_v == 128)))
    return DA_ERR_UNSUPPORTED;
  for (const da_t4* t : {&p->q1, &p->q2, &p->k1, &p->k2, &p->v, &p->out, &p->dout, &p->o2,
                         &p->dq1, &p->dq2, &p->dk1, &p->dk2, &p->dv})
    if (check_t4(*t, p->dtype) != DA_OK) return DA_ERR_INVALID_ARG;
  if (!p->lse1 || !p->lse2 || !p->rstd) return DA_ERR_INVALID_ARG;
  const size_t need =
      da::v1_bwd_workspace_bytes(p->B, p->N, p->H, p->d_qk, p->d_v, p->deterministic != 0, p->causal != 0);
  if (p->workspace == nullptr || p->workspace_bytes < need || !aligned(p->workspace, 256))
    return DA_ERR_WORKSPACE;
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale
                                             : 1.f / std::sqrt(static_cast<float>(p->d_qk));
  da::V1BwdArgs a{p->B, p->N, p->H, p->d_qk, p->d_v, p->causal, scale, p->lambda_init,
                  p->rms_eps, p->q1, p->q2, p->k1, p->k2, p->v, p->out, p->dout, p->o2,
                  p->lq1, p->lk1, p->lq2, p->lk2, p->lse1, p->lse2, p->rstd,
                  p->dq1, p->dq2, p->dk1, p->dk2, p->dv, p->dlq1, p->dlk1, p->dlq2, p->dlk2,
                  p->workspace, p->workspace_bytes, d.status, d.num_sms, p->deterministic != 0,
                  p->rms_weight};
  return cuda_status(da::launch_v1_bwd(a, static_cast<cudaStream_t>(stream)));
}

// ----------------------------------------------------------- V2 fwd --------
size_t diffattn_v2_fwd_workspace_size(int B, int N, int h, int gate_given) {
  if (gate_given || B <= 0 || N <= 0 || h <= 0) return 0;
  return align256(static_cast<size_t>(B) * N * h * sizeof(float));
}

da_status diffattn_v2_fwd(const da_v2_fwd_params* p, void* stream) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->B < 0 || p->N < 0 || p->h <= 0 || p->h_kv <= 0 || p->d <= 0) return DA_ERR_INVALID_ARG;
  if ((2 * p->h) % p->h_kv) return DA_ERR_INVALID_ARG;
  if ((2 * p->h / p->h_kv) % 2) return DA_ERR_INVALID_ARG;
  if (p->B == 0 || p->N == 0) return DA_OK;
  if (p->d != 64 && p->d != 128) return DA_ERR_UNSUPPORTED;
  for (const da_t4* t : {&p->q, &p->k, &p->v, &p->out})
    if (check_t4(*t, DA_BF16) != DA_OK) return DA_ERR_INVALID_ARG;
  if (p->o_heads.ptr && check_t4(p->o_heads, DA_BF16) != DA_OK) return DA_ERR_INVALID_ARG;
  if (p->lse && !aligned(p->lse, 4)) return DA_ERR_INVALID_ARG;
  if (p->gate == nullptr) {
    if (!p->x || !p->w_lambda || p->d_model <= 0) return DA_ERR_INVALID_ARG;
    if ((p->d_model % 64) || p->h > 64) return DA_ERR_UNSUPPORTED;
    const size_t need = diffattn_v2_fwd_workspace_size(p->B, p->N, p->h, 0);
    if (p->workspace == nullptr || p->workspace_bytes < need || !aligned(p->workspace, 256))
      return DA_ERR_WORKSPACE;
  } else if (!aligned(p->gate, 4)) {
    return DA_ERR_INVALID_ARG;
  }
  if (!da::tma_available()) return DA_ERR_CUDA;
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float* gate = p->gate;
  if (gate == nullptr) {
    float* g = static_cast<float*>(p->workspace);
    da::GateArgs ga{p->B * p->N, p->d_model, p->h, p->x, p->d_model, p->w_lambda, g, d.status};
    if (da::launch_gate(ga, s) != cudaSuccess) return DA_ERR_CUDA;
    gate = g;
  }
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale
                                             : 1.f / std::sqrt(static_cast<float>(p->d));
  const int fault = g_fault.exchange(0) == DA_FAULT_V2_FWD_SKIP_LOAD ? 1 : 0;
  da::V2FwdArgs a{p->B, p->N, p->h, p->h_kv, p->d, p->causal, scale * kLog2e,
                  p->q, p->k, p->v, p->out, gate, p->lse, p->o_heads, d.status, d.num_sms, fault};
  return cuda_status(da::launch_v2_fwd(a, s));
}

// ----------------------------------------------------------- V2 bwd --------
size_t diffattn_v2_bwd_workspace_size(int B, int N, int h, int d_model) {
  if (B <= 0 || N <= 0 || h <= 0 || d_model < 0) return 0;
  return da::v2_bwd_workspace_bytes(B, N, h, d_model);
}

da_status diffattn_v2_bwd(const da_v2_bwd_params* p, void* stream) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->B < 0 || p->N < 0 || p->h <= 0 || p->h_kv <= 0 || p->d <= 0) return DA_ERR_INVALID_ARG;
  if ((2 * p->h) % p->h_kv) return DA_ERR_INVALID_ARG;
  if ((2 * p->h / p->h_kv) % 2) return DA_ERR_INVALID_ARG;
  if (p->B == 0 || p->N == 0) return DA_OK;
  if (p->d != 64 && p->d != 128) return DA_ERR_UNSUPPORTED;
  for (const da_t4* t : {&p->q, &p->k, &p->v, &p->o_heads, &p->dout, &p->dq, &p->dk, &p->dv})
    if (check_t4(*t, DA_BF16) != DA_OK) return DA_ERR_INVALID_ARG;
  if (p->lse == nullptr || !aligned(p->lse, 4)) return DA_ERR_INVALID_ARG;
  const bool need_xw = p->gate == nullptr || p->dx != nullptr || p->dw_lambda != nullptr;
  if (need_xw) {
    if (!p->x || !p->w_lambda || p->d_model <= 0) return DA_ERR_INVALID_ARG;
    if (!aligned(p->x, 16) || !aligned(p->w_lambda, 16)) return DA_ERR_INVALID_ARG;
    if ((p->d_model % 64) || p->h > 64) return DA_ERR_UNSUPPORTED;
  }
  if (p->gate && !aligned(p->gate, 4)) return DA_ERR_INVALID_ARG;
  if (p->dgate_logit && !aligned(p->dgate_logit, 4)) return DA_ERR_INVALID_ARG;
  if (p->dx && !aligned(p->dx, 16)) return DA_ERR_INVALID_ARG;
  if (p->dw_lambda && !aligned(p->dw_lambda, 4)) return DA_ERR_INVALID_ARG;
  const size_t need = da::v2_bwd_workspace_bytes(p->B, p->N, p->h, p->dw_lambda ? p->d_model : 0);
  if (p->workspace == nullptr || p->workspace_bytes < need || !aligned(p->workspace, 256))
    return DA_ERR_WORKSPACE;
  if (!da::tma_available()) return DA_ERR_CUDA;
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale
                                             : 1.f / std::sqrt(static_cast<float>(p->d));
  da::V2BwdArgs a{p->B, p->N, p->h, p->h_kv, p->d, p->d_model, p->causal, scale,
                  p->q, p->k, p->v, p->o_heads, p->dout, p->dq, p->dk, p->dv,
                  p->gate, p->lse, p->x, p->w_lambda, p->dgate_logit, p->dx, p->dw_lambda,
                  p->workspace, p->workspace_bytes, d.status, d.num_sms, 1, p->h};
  return cuda_status(da::launch_v2_bwd(a, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------ V1 decode ----
int diffattn_v1_decode_num_splits(int B, int H, int L_max) {
  if (B <= 0 || H <= 0 || L_max <= 0) return 1;
  // one 192 KB CTA per SM: about 6 waves (at B64 L32768 H16, 1, 2, 3, 4, 6,
  // 8 splits gave 7.31, 7.22, 7.14, 7.18, 7.16, 7.10 TB/s), no split shorter
  // than 1024 keys
  int sms = 152;
  DevInfo d = device_info();
  if (d.ok) sms = d.num_sms;
  const long units = static_cast<long>(B) * H;
  long s = (6L * sms + units - 1) / units;
  const long max_s = (L_max + 1023) / 1024;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

size_t diffattn_v1_decode_workspace_size(int B, int H, int d_v, int L_max, int num_splits) {
  if (B <= 0 || H <= 0 || d_v <= 0) return 0;
  if (num_splits <= 0) num_splits = diffattn_v1_decode_num_splits(B, H, L_max);
  const size_t po = static_cast<size_t>(num_splits) * B * H * 2 * d_v * sizeof(float);
  const size_t pml = static_cast<size_t>(num_splits) * B * H * 2 * 2 * sizeof(float);
  return align256(po) + align256(pml);
}

da_status diffattn_v1_decode(const da_v1_decode_params* p, void* stream) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->B <= 0 || p->H <= 0 || p->d_qk <= 0 || p->d_v <= 0 || p->L_max <= 0) return DA_ERR_INVALID_ARG;
  if (!(p->rms_eps >= 0.f)) return DA_ERR_INVALID_ARG;
  if (!((p->d_qk == 128 && p->d_v == 256) || (p->d_qk == 64 && p->d_v == 128))) return DA_ERR_UNSUPPORTED;
  if (!p->q1 || !p->q2 || !p->out || !aligned(p->q1, 16) || !aligned(p->q2, 16) || !aligned(p->out, 16))
    return DA_ERR_INVALID_ARG;
  if (!p->lq1 || !p->lk1 || !p->lq2 || !p->lk2) return DA_ERR_INVALID_ARG;
  if (p->rms_weight && !aligned(p->rms_weight, 4)) return DA_ERR_INVALID_ARG;
  for (const da_t4* t : {&p->k1_cache, &p->k2_cache, &p->v_cache})
    if (check_t4(*t, DA_BF16) != DA_OK) return DA_ERR_INVALID_ARG;
  const int splits = p->num_splits > 0 ? p->num_splits : diffattn_v1_decode_num_splits(p->B, p->H, p->L_max);
  if (splits > 65535) return DA_ERR_INVALID_ARG;
  const size_t need = diffattn_v1_decode_workspace_size(p->B, p->H, p->d_v, p->L_max, splits);
  if (p->workspace == nullptr || p->workspace_bytes < need || !aligned(p->workspace, 256))
    return DA_ERR_WORKSPACE;
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(p->workspace);
  const size_t po = static_cast<size_t>(splits) * p->B * p->H * 2 * p->d_v * sizeof(float);
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale
                                             : 1.f / std::sqrt(static_cast<float>(p->d_qk));
  da::V1DecodeArgs a{p->B, p->H, p->d_qk, p->d_v, p->L_max, splits, scale * kLog2e, p->lambda_init, p->rms_eps,
                     p->q1, p->q2, p->k1_cache, p->k2_cache, p->v_cache, p->seqlens,
                     p->lq1, p->lk1, p->lq2, p->lk2, p->out,
                     reinterpret_cast<float*>(ws), reinterpret_cast<float*>(ws + align256(po)), d.status,
                     p->rms_weight};
  return cuda_status(da::launch_v1_decode(a, static_cast<cudaStream_t>(stream)));
}

// --------------------------------------------------------- grouped fwd -----
size_t diffattn_grouped_fwd_workspace_size(int B, int N, int h, int ratio, int d, int gate_given,
                                           int heads_given) {
  if (B <= 0 || N <= 0 || h <= 0 || ratio <= 0 || d <= 0 || h % ratio) return 0;
  const size_t Hq = static_cast<size_t>(h) / ratio * (ratio + 1);
  const size_t g = gate_given ? 0 : static_cast<size_t>(B) * N * h * sizeof(float);
  const size_t o = heads_given ? 0 : static_cast<size_t>(B) * N * Hq * d * 2;
  return align256(g) + align256(o);
}

da_status diffattn_grouped_fwd(const da_grouped_fwd_params* p, void* stream) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->B < 0 || p->N < 0 || p->h <= 0 || p->ratio <= 0 || p->h_kv <= 0 || p->d <= 0)
    return DA_ERR_INVALID_ARG;
  if (p->h % p->ratio) return DA_ERR_INVALID_ARG;
  const int Hq = p->h / p->ratio * (p->ratio + 1);
  if (Hq % p->h_kv) return DA_ERR_INVALID_ARG;
  const int G = Hq / p->h_kv;
  if (G % (p->ratio + 1)) return DA_ERR_INVALID_ARG;  // a group must sit in one K/V group
  if (p->B == 0 || p->N == 0) return DA_OK;
  if ((p->d != 64 && p->d != 128) || (G % 2)) return DA_ERR_UNSUPPORTED;
  for (const da_t4* t : {&p->q, &p->k, &p->v, &p->out})
    if (check_t4(*t, DA_BF16) != DA_OK) return DA_ERR_INVALID_ARG;
  if (p->o_heads.ptr && check_t4(p->o_heads, DA_BF16) != DA_OK) return DA_ERR_INVALID_ARG;
  if (p->lse && !aligned(p->lse, 4)) return DA_ERR_INVALID_ARG;
  if (p->gate == nullptr) {
    if (!p->x || !p->w_lambda || p->d_model <= 0) return DA_ERR_INVALID_ARG;
    if ((p->d_model % 64) || p->h > 64) return DA_ERR_UNSUPPORTED;
  } else if (!aligned(p->gate, 4)) {
    return DA_ERR_INVALID_ARG;
  }
  const size_t need = diffattn_grouped_fwd_workspace_size(p->B, p->N, p->h, p->ratio, p->d, p->gate != nullptr,
                                                          p->o_heads.ptr != nullptr);
  if (need && (p->workspace == nullptr || p->workspace_bytes < need || !aligned(p->workspace, 256)))
    return DA_ERR_WORKSPACE;
  if (!da::tma_available()) return DA_ERR_CUDA;
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(p->workspace);
  const float* gate = p->gate;
  size_t off = 0;
  if (gate == nullptr) {
    float* g = reinterpret_cast<float*>(ws);
    da::GateArgs ga{p->B * p->N, p->d_model, p->h, p->x, p->d_model, p->w_lambda, g, d.status};
    if (da::launch_gate(ga, s) != cudaSuccess) return DA_ERR_CUDA;
    gate = g;
    off = align256(static_cast<size_t>(p->B) * p->N * p->h * sizeof(float));
  }
  da_t4 heads = p->o_heads;
  if (heads.ptr == nullptr) {
    const int64_t sn = static_cast<int64_t>(Hq) * p->d;
    heads = da_t4{ws + off, static_cast<int64_t>(p->N) * sn, sn, p->d};
  }
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale
                                             : 1.f / std::sqrt(static_cast<float>(p->d));
  // the attention over all Hq heads (taken two at a time), per-head outputs only
  da::V2FwdArgs fa{p->B, p->N, Hq / 2, p->h_kv, p->d, p->causal, scale * kLog2e,
                   p->q, p->k, p->v, da_t4{nullptr, 0, 0, 0}, nullptr, p->lse, heads, d.status, d.num_sms, 0};
  if (da::launch_v2_fwd(fa, s) != cudaSuccess) return DA_ERR_CUDA;
  da::GroupedArgs ca{p->B, p->N, p->h, p->ratio, p->d, heads, gate, p->out};
  return cuda_status(da::launch_grouped_combine(ca, s));
}

// ------------------------------------------------------------ grouped bwd ----
size_t diffattn_grouped_bwd_workspace_size(int B, int N, int h, int ratio, int d_model) {
  if (B <= 0 || N <= 0 || h <= 0 || ratio <= 0 || h % ratio) return 0;
  const int Hq = h / ratio * (ratio + 1);
  if (Hq % 2) return 0;
  return da::grouped_bwd_workspace_bytes(B, N, Hq / 2, h, d_model > 0 ? d_model : 0);
}

da_status diffattn_grouped_bwd(const da_grouped_bwd_params* p, void* stream) {
  if (p == nullptr) return DA_ERR_INVALID_ARG;
  if (p->B < 0 || p->N < 0 || p->h <= 0 || p->ratio <= 0 || p->h_kv <= 0 || p->d <= 0)
    return DA_ERR_INVALID_ARG;
  if (p->h % p->ratio) return DA_ERR_INVALID_ARG;
  const int Hq = p->h / p->ratio * (p->ratio + 1);
  if (Hq % p->h_kv) return DA_ERR_INVALID_ARG;
  const int G = Hq / p->h_kv;
  if (G % (p->ratio + 1)) return DA_ERR_INVALID_ARG;  // a group must sit in one K/V group
  if (p->B == 0 || p->N == 0) return DA_OK;
  if ((p->d != 64 && p->d != 128) || (G % 2)) return DA_ERR_UNSUPPORTED;
  for (const da_t4* t : {&p->q, &p->k, &p->v, &p->o_heads, &p->dout, &p->dq, &p->dk, &p->dv})
    if (check_t4(*t, DA_BF16) != DA_OK) return DA_ERR_INVALID_ARG;
  if (p->lse == nullptr || !aligned(p->lse, 4)) return DA_ERR_INVALID_ARG;
  const bool need_xw = p->gate == nullptr || p->dx != nullptr || p->dw_lambda != nullptr;
  if (need_xw) {
    if (!p->x || !p->w_lambda || p->d_model <= 0) return DA_ERR_INVALID_ARG;
    if (!aligned(p->x, 16) || !aligned(p->w_lambda, 16)) return DA_ERR_INVALID_ARG;
    if ((p->d_model % 64) || p->h > 64) return DA_ERR_UNSUPPORTED;
  }
  if (p->gate && !aligned(p->gate, 4)) return DA_ERR_INVALID_ARG;
  if (p->dgate_logit && !aligned(p->dgate_logit, 4)) return DA_ERR_INVALID_ARG;
  if (p->dx && !aligned(p->dx, 16)) return DA_ERR_INVALID_ARG;
  if (p->dw_lambda && !aligned(p->dw_lambda, 4)) return DA_ERR_INVALID_ARG;
  const size_t need = da::grouped_bwd_workspace_bytes(p->B, p->N, Hq / 2, p->h, p->dw_lambda ? p->d_model : 0);
  if (p->workspace == nullptr || p->workspace_bytes < need || !aligned(p->workspace, 256))
    return DA_ERR_WORKSPACE;
  if (!da::tma_available()) return DA_ERR_CUDA;
  DevInfo d = device_info();
  if (!d.ok) return DA_ERR_CUDA;
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale
                                             : 1.f / std::sqrt(static_cast<float>(p->d));
  da::V2BwdArgs a{p->B, p->N, Hq / 2, p->h_kv, p->d, p->d_model, p->causal, scale,
                  p->q, p->k, p->v, p->o_heads, p->dout, p->dq, p->dk, p->dv,
                  p->gate, p->lse, p->x, p->w_lambda, p->dgate_logit, p->dx, p->dw_lambda,
                  p->workspace, p->workspace_bytes, d.status, d.num_sms, p->ratio, p->h};
  return cuda_status(da::launch_v2_bwd(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
