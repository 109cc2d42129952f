// v1_f32.cu — V1 differential attention forward in fp32 (SIMT FMA).
//
// "Differential Transformer | ICLR 2025 Oral" (dainus.ai), "Differential
// Attention: 빼기의 힘": O = (softmax(s Q1 K1^T) - lambda softmax(s Q2 K2^T)) V;
// "Differential Transformer V2" (pogovet.com), §1: per-head RMS
// normalisation after the subtraction and the per-layer scale.
//
// This is the exact-precision path (fp32 operands and accumulation; the tensor
// cores' tf32 mode would not hold a 1e-4 relative bar), meant for small
// correctness shapes.  One warp owns one query row: lanes take 32 keys at a
// time for the two score streams (online max / sum per stream, warp
// reductions), then every lane accumulates its d_v/32 output features of
// both streams; the epilogue forms O1/l1 - lambda O2/l2, the RMS over d_v
// and the (1 - lambda_init) scale.
#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxDqk = 128;
constexpr int kMaxDv = 256;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ float lambda_of(const V1F32Args& a, int lane) {
  float d1 = 0.f, d2 = 0.f;
  for (int x = lane; x < a.d_qk; x += 32) {
    d1 += a.lq1[x] * a.lk1[x];
    d2 += a.lq2[x] * a.lk2[x];
  }
  d1 = warp_sum(d1);
  d2 = warp_sum(d2);
  return expf(d1) - expf(d2) + a.lambda_init;
}

__global__ void __launch_bounds__(kWarps * 32)
v1_fwd_f32_kernel(V1F32Args a) {
  __shared__ float sq[kWarps][2][kMaxDqk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarps + warp;  // query row
  const int h = blockIdx.y, b = blockIdx.z;
  if (i >= a.N) return;
  const float lam = lambda_of(a, lane);
  if (a.lambda_out && i == 0 && h == 0 && b == 0 && lane == 0) *a.lambda_out = lam;

  const float* q1 = static_cast<const float*>(a.q1.ptr) + b * a.q1.sb + i * a.q1.sn + h * a.q1.sh;
  const float* q2 = static_cast<const float*>(a.q2.ptr) + b * a.q2.sb + i * a.q2.sn + h * a.q2.sh;
  for (int x = lane; x < a.d_qk; x += 32) {
    sq[warp][0][x] = q1[x];
    sq[warp][1][x] = q2[x];
  }
  __syncwarp();

  const float* k1 = static_cast<const float*>(a.k1.ptr) + b * a.k1.sb + h * a.k1.sh;
  const float* k2 = static_cast<const float*>(a.k2.ptr) + b * a.k2.sb + h * a.k2.sh;
  const float* v = static_cast<const float*>(a.v.ptr) + b * a.v.sb + h * a.v.sh;
  const int nv = a.d_v / 32;  // features per lane
  float o1[kMaxDv / 32], o2[kMaxDv / 32];
#pragma unroll
  for (int c = 0; c < kMaxDv / 32; ++c) o1[c] = o2[c] = 0.f;
  float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
  const int n_keys = a.causal ? i + 1 : a.N;

  for (int j0 = 0; j0 < n_keys; j0 += 32) {
    const int j = j0 + lane;
    float s1 = -INFINITY, s2 = -INFINITY;
    if (j < n_keys) {
      const float* kr1 = k1 + j * a.k1.sn;
      const float* kr2 = k2 + j * a.k2.sn;
      float d1 = 0.f, d2 = 0.f;
      for (int x = 0; x < a.d_qk; ++x) {
        d1 = fmaf(sq[warp][0][x], kr1[x], d1);
        d2 = fmaf(sq[warp][1][x], kr2[x], d2);
      }
      s1 = d1 * a.scale;
      s2 = d2 * a.scale;
    }
    const float n1 = fmaxf(m1, warp_max(s1));
    const float n2 = fmaxf(m2, warp_max(s2));
    const float c1 = expf(m1 - n1), c2 = expf(m2 - n2);
    const float p1 = j < n_keys ? expf(s1 - n1) : 0.f;
    const float p2 = j < n_keys ? expf(s2 - n2) : 0.f;
    l1 = l1 * c1 + warp_sum(p1);
    l2 = l2 * c2 + warp_sum(p2);
    m1 = n1;
    m2 = n2;
#pragma unroll
    for (int c = 0; c < kMaxDv / 32; ++c) {
      o1[c] *= c1;
      o2[c] *= c2;
    }
    const int cnt = min(32, n_keys - j0);
    for (int kk = 0; kk < cnt; ++kk) {
      const float w1 = __shfl_sync(0xffffffffu, p1, kk);
      const float w2 = __shfl_sync(0xffffffffu, p2, kk);
      const float* vr = v + (j0 + kk) * a.v.sn;
#pragma unroll
      for (int c = 0; c < kMaxDv / 32; ++c) {
        if (c < nv) {
          const float vv = vr[lane + 32 * c];
          o1[c] = fmaf(w1, vv, o1[c]);
          o2[c] = fmaf(w2, vv, o2[c]);
        }
      }
    }
  }

  const float inv1 = 1.f / l1, inv2 = 1.f / l2;
  float o[kMaxDv / 32];
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < kMaxDv / 32; ++c) {
    o[c] = 0.f;
    if (c < nv) {
      o2[c] *= inv2;
      o[c] = __fsub_rn(__fmul_rn(o1[c], inv1), __fmul_rn(lam, o2[c]));
      ss += o[c] * o[c];
    }
  }
  ss = warp_sum(ss);
  const float rstd = 1.f / sqrtf(ss / a.d_v + a.rms_eps);
  const float cs = (1.f - a.lambda_init) * rstd;
  float* out = static_cast<float*>(a.out.ptr) + b * a.out.sb + i * a.out.sn + h * a.out.sh;
  float* o2p = a.o2.ptr ? static_cast<float*>(a.o2.ptr) + b * a.o2.sb + i * a.o2.sn + h * a.o2.sh
                        : nullptr;
#pragma unroll
  for (int c = 0; c < kMaxDv / 32; ++c) {
    if (c < nv) {
      out[lane + 32 * c] = a.rms_weight ? (o[c] * cs) * a.rms_weight[lane + 32 * c] : o[c] * cs;
      if (o2p) o2p[lane + 32 * c] = o2[c];
    }
  }
  if (lane == 0) {
    const int64_t st = (static_cast<int64_t>(b) * a.H + h) * a.N + i;
    if (a.lse1) a.lse1[st] = m1 + logf(l1);
    if (a.lse2) a.lse2[st] = m2 + logf(l2);
    if (a.rstd) a.rstd[st] = rstd;
  }
}

}  // namespace

cudaError_t launch_v1_fwd_f32(const V1F32Args& a, cudaStream_t s) {
  dim3 grid((a.N + kWarps - 1) / kWarps, a.H, a.B);
  if (a.N == 0 || a.H == 0 || a.B == 0) return cudaSuccess;
  v1_fwd_f32_kernel<<<grid, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace da
