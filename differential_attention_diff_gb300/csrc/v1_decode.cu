// v1_decode.cu — V1 decode: one new token per sequence over bf16 K1, K2 and V
// caches.
//
// "Differential Transformer | ICLR 2025 Oral" (dainus.ai), "Differential
// Attention: 빼기의 힘": two softmax maps over two key sets and one shared value
// set, the second map scaled by lambda and subtracted; "V2로의 진화" names LLM
// decoding as the memory-bound case.  "Differential Transformer V2"
// (pogovet.com), §1: per-head RMS normalisation after the subtraction, then
// the (1 - lambda_init) scale.  Every cache byte is read once per step (1 KB
// per key and head: K1 and K2 rows of 256 B, a V row of 512 B), so the kernel
// is shaped by streaming the caches.
//
// Stage 1 (split-KV): grid (splits, H, B), 8 warps.  K1, K2 and V tiles of 64
// keys go through a 3-deep cp.async ring (16-byte chunks, XOR-swizzled rows).
// Warp w owns keys 16 (w mod 4) .. +15 of a tile and half (w / 4) of the
// 256-wide V.  The scores run on the warp MMA with the two streams' queries
// as M rows 0 and 1 (q1 against the K1 tile, q2 against the K2 tile: one
// pass each); the online softmax keeps one (max, sum) per row, and both rows
// of P multiply the shared V tile in one P.V pass.  Per split it writes the
// unnormalised partial O of each stream and its (max in log2 units, sum).
// Stage 2 (merge): grid (H, B), one thread per V feature: the log-sum-exp
// merge of each stream, O = O1 - lambda O2 (each product rounded on its own,
// so equal streams with lambda 1 cancel exactly), the RMS over the d_v
// features, and Y = (1 - lambda_init) O / sqrt(mean O^2 + eps) in bf16.
#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int kTileKeys = 64;
constexpr int kStages = 3;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
// Head dims (DQK, DV = 2 DQK) = (128, 256) or (64, 128): K rows of DQK * 2
// bytes, V rows of DV * 2 bytes, K1 + K2 + V tiles of 64 keys per stage
// (64 KB for (128, 256)).
template <int DQK, int DV>
struct Cfg {
  static constexpr int kKRow = DQK * 2;
  static constexpr int kVRow = DV * 2;
  static constexpr int kKTile = kTileKeys * kKRow;
  static constexpr int kVTile = kTileKeys * kVRow;
  static constexpr int kStageBytes = 2 * kKTile + kVTile;
  static constexpr int kSmemBytes = kStages * kStageBytes;
};

// 16-byte chunk c of row r: the low 3 chunk bits XORed with the row, so that
// 8 consecutive rows at one logical chunk land in 8 different bank groups.
__device__ __forceinline__ uint32_t row_off(int r, int c, int row_bytes) {
  return static_cast<uint32_t>(r * row_bytes + ((c ^ (r & 7)) << 4));
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
v1_decode_split_kernel(V1DecodeArgs a) {
  using C = Cfg<DQK, DV>;
  constexpr int kDqk = DQK, kDv = DV, kHalf = DV / 2;
  constexpr int kKRow = C::kKRow, kVRow = C::kVRow, kKTile = C::kKTile, kStageBytes = C::kStageBytes;
  constexpr int kKC = DQK / 8, kVC = DV / 8;  // 16-byte chunks per K / V row
  extern __shared__ __align__(1024) uint8_t smem[];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int L = a.seqlens ? a.seqlens[b] : a.L_max;
  if (L < 1 || L > a.L_max) {
    if (tid == 0) record_status(a.status, DA_ERR_BOUNDS, 0x0E01);
    L = 0;
  }
  int chunk = (L + a.num_splits - 1) / a.num_splits;
  chunk = (chunk + kTileKeys - 1) / kTileKeys * kTileKeys;
  const int k_begin = min(L, split * chunk);
  const int k_end = min(L, k_begin + chunk);
  const int n_tiles = (k_end - k_begin + kTileKeys - 1) / kTileKeys;

  const __nv_bfloat16* k1base = static_cast<const __nv_bfloat16*>(a.k1.ptr) + b * a.k1.sb + h * a.k1.sh;
  const __nv_bfloat16* k2base = static_cast<const __nv_bfloat16*>(a.k2.ptr) + b * a.k2.sb + h * a.k2.sh;
  const __nv_bfloat16* vbase = static_cast<const __nv_bfloat16*>(a.v.ptr) + b * a.v.sb + h * a.v.sh;
  const uint32_t sbase = smem_u32(smem);

  auto issue_tile = [&](int t) {
    if (t < n_tiles) {
      const int key0 = k_begin + t * kTileKeys;
      const uint32_t ks1 = sbase + (t % kStages) * kStageBytes;
      const uint32_t ks2 = ks1 + kKTile;
      const uint32_t vs = ks2 + kKTile;
#pragma unroll
      for (int i = 0; i < (kTileKeys * kKC) / kThreads; ++i) {
        const int idx = i * kThreads + tid;
        const int r = idx / kKC, c = idx % kKC;
        const int key = key0 + r;
        const bool ok = key < k_end;
        const int kk = ok ? key : k_begin;  // any in-range row when masked
        cp_async_16(ks1 + row_off(r, c, kKRow), k1base + static_cast<int64_t>(kk) * a.k1.sn + c * 8, ok ? 16 : 0);
        cp_async_16(ks2 + row_off(r, c, kKRow), k2base + static_cast<int64_t>(kk) * a.k2.sn + c * 8, ok ? 16 : 0);
      }
#pragma unroll
      for (int i = 0; i < (kTileKeys * kVC) / kThreads; ++i) {
        const int idx = i * kThreads + tid;
        const int r = idx / kVC, c = idx % kVC;
        const int key = key0 + r;
        const bool ok = key < k_end;
        const int kk = ok ? key : k_begin;
        cp_async_16(vs + row_off(r, c, kVRow), vbase + static_cast<int64_t>(kk) * a.v.sn + c * 8, ok ? 16 : 0);
      }
    }
    cp_async_commit();
  };

  // A fragments: row 0 = q1 (held by lanes with gr == 0), row 1 = q2 (gr ==
  // 1); the other 14 rows are zero.  Only the (row gr, k) halves of the
  // fragment can be non-zero, so two registers per k-step and stream.
  const int gr = lane >> 2, tq = lane & 3;
  uint32_t q1a[kDqk / 16][2], q2a[kDqk / 16][2];
  {
    const int64_t qoff = (static_cast<int64_t>(b) * a.H + h) * kDqk;
    const __nv_bfloat16* q1p = static_cast<const __nv_bfloat16*>(a.q1) + qoff;
    const __nv_bfloat16* q2p = static_cast<const __nv_bfloat16*>(a.q2) + qoff;
#pragma unroll
    for (int ks = 0; ks < kDqk / 16; ++ks) {
      const int c0 = ks * 16 + 2 * tq;
      q1a[ks][0] = gr == 0 ? *reinterpret_cast<const uint32_t*>(q1p + c0) : 0u;
      q1a[ks][1] = gr == 0 ? *reinterpret_cast<const uint32_t*>(q1p + c0 + 8) : 0u;
      q2a[ks][0] = gr == 1 ? *reinterpret_cast<const uint32_t*>(q2p + c0) : 0u;
      q2a[ks][1] = gr == 1 ? *reinterpret_cast<const uint32_t*>(q2p + c0 + 8) : 0u;
    }
  }

  float o[kHalf / 8][4];
#pragma unroll
  for (int i = 0; i < kHalf / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  const int wk0 = (warp & 3) * 16;  // this warp's keys within a tile
  const int fh = warp >> 2;         // this warp's half of the V features

#pragma unroll
  for (int t = 0; t < kStages - 1; ++t) issue_tile(t);

  for (int t = 0; t < n_tiles; ++t) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    issue_tile(t + kStages - 1);

    const uint32_t ks1 = sbase + (t % kStages) * kStageBytes;
    const uint32_t ks2 = ks1 + kKTile;
    const uint32_t vs = ks2 + kKTile;

    // scores: stream 1 in row 0 (K1 tile), stream 2 in row 1 (K2 tile)
    float s1[2][4], s2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s1[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int kp = 0; kp < kDqk / 32; ++kp) {
        const int r = wk0 + nt * 8 + (lane & 7);
        const int c = kp * 4 + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(ks1 + row_off(r, c, kKRow), b0, b1, b2, b3);
        {
          const uint32_t fa[4] = {q1a[2 * kp][0], 0u, q1a[2 * kp][1], 0u};
          const uint32_t fb[4] = {q1a[2 * kp + 1][0], 0u, q1a[2 * kp + 1][1], 0u};
          mma_bf16_16816(s1[nt], fa, b0, b1);
          mma_bf16_16816(s1[nt], fb, b2, b3);
        }
        ldmatrix_x4(ks2 + row_off(r, c, kKRow), b0, b1, b2, b3);
        {
          const uint32_t fa[4] = {q2a[2 * kp][0], 0u, q2a[2 * kp][1], 0u};
          const uint32_t fb[4] = {q2a[2 * kp + 1][0], 0u, q2a[2 * kp + 1][1], 0u};
          mma_bf16_16816(s2[nt], fa, b0, b1);
          mma_bf16_16816(s2[nt], fb, b2, b3);
        }
      }
    }
    // this lane's row gr takes its stream's scores; mask keys past the split
    // end and scale into log2 units
    const int key_base = k_begin + t * kTileKeys + wk0;
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key_base + nt * 8 + 2 * tq + (e & 1);
        const float v = gr == 1 ? s2[nt][e] : s1[nt][e];
        s[nt][e] = key < k_end ? v * a.scale_log2 : -INFINITY;
      }
    }
    // online softmax per row (rows gr and gr + 8; only rows 0 and 1 are used)
    float mx_lo = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mx_hi = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float base_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
    const float base_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    const float al_lo = fast_exp2(m_lo - base_lo), al_hi = fast_exp2(m_hi - base_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[nt][0] = fast_exp2(s[nt][0] - base_lo);
      p[nt][1] = fast_exp2(s[nt][1] - base_lo);
      p[nt][2] = fast_exp2(s[nt][2] - base_hi);
      p[nt][3] = fast_exp2(s[nt][3] - base_hi);
    }
    l_lo = l_lo * al_lo + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
    l_hi = l_hi * al_hi + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
#pragma unroll
    for (int i = 0; i < kHalf / 8; ++i) {
      o[i][0] *= al_lo;
      o[i][1] *= al_lo;
      o[i][2] *= al_hi;
      o[i][3] *= al_hi;
    }
    uint32_t pa[4];
    pa[0] = pack_bf16x2(p[0][0], p[0][1]);
    pa[1] = pack_bf16x2(p[0][2], p[0][3]);
    pa[2] = pack_bf16x2(p[1][0], p[1][1]);
    pa[3] = pack_bf16x2(p[1][2], p[1][3]);
    // O[16 x DV/2 (this half)] += P[16 x 16 keys] . V[16 keys x DV/2]
#pragma unroll
    for (int np = 0; np < kHalf / 16; ++np) {
      const int r = wk0 + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int c = fh * (kHalf / 8) + np * 2 + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(vs + row_off(r, c, kVRow), b0, b1, b2, b3);
      mma_bf16_16816(o[2 * np], pa, b0, b1);
      mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);

  // merge the 4 key-warps of each feature half (rows 0 and 1 only) through
  // shared memory, reusing the ring
  float* so = reinterpret_cast<float*>(smem);  // [warp][row 0..1][DV/2]
  float* sml = so + kWarps * 2 * kHalf;        // [warp][row 0..1][max, sum]
  if (gr < 2) {
#pragma unroll
    for (int nt = 0; nt < kHalf / 8; ++nt) {
      const int col = nt * 8 + 2 * tq;
      so[(warp * 2 + gr) * kHalf + col] = o[nt][0];
      so[(warp * 2 + gr) * kHalf + col + 1] = o[nt][1];
    }
    if (tq == 0) {
      sml[(warp * 2 + gr) * 2] = m_lo;
      sml[(warp * 2 + gr) * 2 + 1] = l_lo;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < 2 * kDv; idx += kThreads) {
    const int row = idx / kDv, f = idx % kDv;
    const int half = f / kHalf, col = f % kHalf;
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) mt = fmaxf(mt, sml[((half * 4 + j) * 2 + row) * 2]);
    const float base = mt == -INFINITY ? 0.f : mt;
    float lt = 0.f, ot = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int w = half * 4 + j;
      const float fct = fast_exp2(sml[(w * 2 + row) * 2] - base);
      lt += sml[(w * 2 + row) * 2 + 1] * fct;
      ot += so[(w * 2 + row) * kHalf + col] * fct;
    }
    const int64_t pidx = ((static_cast<int64_t>(split) * a.B + b) * a.H + h) * 2 + row;
    a.part_o[pidx * kDv + f] = ot;
    if (f == 0) {
      a.part_ml[pidx * 2] = mt;
      a.part_ml[pidx * 2 + 1] = lt;
    }
  }
}

// Merge the splits of both streams, the difference, the RMSNorm and the
// scale.  Block = d_v threads (<= 256), one V feature each; grid (H, B).
__global__ void __launch_bounds__(256)
v1_decode_merge_kernel(V1DecodeArgs a) {
  const int dqk = a.d_qk, dv = a.d_v;
  __shared__ float s_lam;
  __shared__ float s_red[8];
  const int h = blockIdx.x, b = blockIdx.y, f = threadIdx.x;
  const int warp = f >> 5, lane = f & 31;
  if (warp == 0) {
    float d1 = 0.f, d2 = 0.f;
    for (int x = lane; x < dqk; x += 32) {
      d1 = fmaf(a.lq1[x], a.lk1[x], d1);
      d2 = fmaf(a.lq2[x], a.lk2[x], d2);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      d1 += __shfl_xor_sync(0xffffffffu, d1, o);
      d2 += __shfl_xor_sync(0xffffffffu, d2, o);
    }
    if (lane == 0) s_lam = expf(d1) - expf(d2) + a.lambda_init;
  }
  float res[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float mt = -INFINITY;
    for (int s = 0; s < a.num_splits; ++s)
      mt = fmaxf(mt, a.part_ml[(((static_cast<int64_t>(s) * a.B + b) * a.H + h) * 2 + e) * 2]);
    const float base = mt == -INFINITY ? 0.f : mt;
    float lt = 0.f, ot = 0.f;
    for (int s = 0; s < a.num_splits; ++s) {
      const int64_t pidx = ((static_cast<int64_t>(s) * a.B + b) * a.H + h) * 2 + e;
      const float fct = exp2f(a.part_ml[pidx * 2] - base);
      lt += a.part_ml[pidx * 2 + 1] * fct;
      ot += a.part_o[pidx * dv + f] * fct;
    }
    res[e] = lt > 0.f ? ot / lt : 0.f;
  }
  __syncthreads();  // s_lam
  const float o = __fsub_rn(res[0], __fmul_rn(s_lam, res[1]));
  float ss = o * o;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if (lane == 0) s_red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w)
    if (w < dv / 32) tot += s_red[w];
  const float rstd = 1.f / sqrtf(tot * (1.f / dv) + a.rms_eps);
  const float w = a.rms_weight ? a.rms_weight[f] : 1.f;
  static_cast<__nv_bfloat16*>(a.out)[(static_cast<int64_t>(b) * a.H + h) * dv + f] =
      __float2bfloat16_rn((1.f - a.lambda_init) * o * rstd * w);
}

template <int DQK, int DV>
cudaError_t launch_split(const V1DecodeArgs& a, cudaStream_t s) {
  constexpr int kSmem = Cfg<DQK, DV>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(v1_decode_split_kernel<DQK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  v1_decode_split_kernel<DQK, DV><<<dim3(a.num_splits, a.H, a.B), kThreads, kSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_v1_decode(const V1DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = (a.d_qk == 128 && a.d_v == 256) ? launch_split<128, 256>(a, s)
                  : (a.d_qk == 64 && a.d_v == 128) ? launch_split<64, 128>(a, s)
                                                   : cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  v1_decode_merge_kernel<<<dim3(a.H, a.B), a.d_v, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace da
