// decode.cu — V2 decode: one new token per sequence over a bf16 KV cache.
//
// "Differential Transformer V2" (pogovet.com), §2: the query heads double
// but the K/V heads and the cache do not, so decode stays bound by reading
// the cache.  The kernel is built around that: every (batch, kv head) group
// streams its K and V rows exactly once and serves all 2h/h_kv query heads of
// the group from the same shared-memory tile (the even/odd pair of a
// difference always sits in one group).
//
// Stage 1 (split-KV): grid (splits, h_kv, B), 8 warps, one CTA per SM.  K/V
// tiles of 128 keys are staged through a 3-deep cp.async ring (16-byte
// chunks, XOR-swizzled rows; up to 128 KB in flight per SM, which the HBM
// latency needs); each warp owns 16 keys of a tile and runs the scores and P.V on the
// warp MMA with the group's query heads as the M rows (16 rows, the unused
// ones zero).  Per split it writes an unnormalised partial O plus the running
// max (log2 units) and sum.
// Stage 2 (merge): grid (h, B); merges the splits of heads 2p and 2p+1 with
// the log-sum-exp rule and writes out = O_2p - gate * O_2p+1 in bf16.
#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int kTileKeys = 128;   // keys per pipeline stage (16 per warp)
constexpr int kStages = 3;
constexpr int kWarps = 8;
// Per head dim D (64 or 128): key rows of D * 2 bytes (D / 8 16-byte chunks),
// K + V tiles of 64 keys per stage.
template <int D>
struct Cfg {
  static constexpr int kChunks = D / 8;
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kTileKeys * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K + V
};
constexpr int kSmemBytes = kStages * Cfg<128>::kStageBytes;  // 192 KB (the D = 128 ring)

// Byte offset of 16-byte chunk c of key row r inside a tile (rows of D / 8
// chunks; the low 3 chunk bits are XORed with the row so that 8 consecutive
// rows at one logical chunk hit 8 different bank groups).
template <int D>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return static_cast<uint32_t>(r * Cfg<D>::kRowBytes + ((c ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32, 1)
decode_split_kernel(DecodeArgs a) {
  constexpr int kD = D;
  constexpr int kChunks = Cfg<D>::kChunks;
  constexpr int kTileBytes = Cfg<D>::kTileBytes;
  constexpr int kStageBytes = Cfg<D>::kStageBytes;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = (2 * a.h) / a.h_kv;  // query heads of this group
  const int qh0 = g * G;

  int L = a.seqlens ? a.seqlens[b] : a.L_max;
  const bool bad = (L < 1 || L > a.L_max);
  if (bad) {
    if (tid == 0) record_status(a.status, DA_ERR_BOUNDS, 0x0D01);
    L = 0;
  }
  // key range of this split: equal chunks of the sequence, rounded to tiles
  int chunk = (L + a.num_splits - 1) / a.num_splits;
  chunk = (chunk + kTileKeys - 1) / kTileKeys * kTileKeys;
  const int k_begin = min(L, split * chunk);
  const int k_end = min(L, k_begin + chunk);
  const int n_tiles = (k_end - k_begin + kTileKeys - 1) / kTileKeys;

  const __nv_bfloat16* kbase = static_cast<const __nv_bfloat16*>(a.k.ptr) +
                               b * a.k.sb + g * a.k.sh;
  const __nv_bfloat16* vbase = static_cast<const __nv_bfloat16*>(a.v.ptr) +
                               b * a.v.sb + g * a.v.sh;
  const uint32_t sbase = smem_u32(smem);

  auto issue_tile = [&](int t) {
    if (t < n_tiles) {
      const int stage = t % kStages;
      const int key0 = k_begin + t * kTileKeys;
      const uint32_t ks = sbase + stage * kStageBytes;
      const uint32_t vs = ks + kTileBytes;
#pragma unroll
      for (int i = 0; i < (kTileKeys * kChunks) / (kWarps * 32); ++i) {
        const int idx = i * kWarps * 32 + tid;
        const int r = idx / kChunks, c = idx % kChunks;
        const int key = key0 + r;
        const bool ok = key < k_end;
        const int kk = ok ? key : k_begin;  // any in-range row when masked
        cp_async_16(ks + tile_off<D>(r, c), kbase + kk * a.k.sn + c * 8, ok ? 16 : 0);
        cp_async_16(vs + tile_off<D>(r, c), vbase + kk * a.v.sn + c * 8, ok ? 16 : 0);
      }
    }
    cp_async_commit();
  };

  // query rows as MMA A fragments: row = head (G <= 16), k = feature
  const int gr = lane >> 2, tq = lane & 3;
  uint32_t qa[kD / 16][4];
  {
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q) +
                              (static_cast<int64_t>(b) * 2 * a.h + qh0) * kD;
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
      const int c0 = ks * 16 + 2 * tq;
      auto ld = [&](int row, int col) -> uint32_t {
        if (row >= G) return 0u;
        return *reinterpret_cast<const uint32_t*>(qb + row * kD + col);
      };
      qa[ks][0] = ld(gr, c0);
      qa[ks][1] = ld(gr + 8, c0);
      qa[ks][2] = ld(gr, c0 + 8);
      qa[ks][3] = ld(gr + 8, c0 + 8);
    }
  }

  float o[kD / 8][4];
#pragma unroll
  for (int i = 0; i < kD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

#pragma unroll
  for (int t = 0; t < kStages - 1; ++t) issue_tile(t);

  for (int t = 0; t < n_tiles; ++t) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    issue_tile(t + kStages - 1);

    const int stage = t % kStages;
    const uint32_t ks = sbase + stage * kStageBytes;
    const uint32_t vs = ks + kTileBytes;
    const int wkey0 = warp * 16;  // this warp's 16 keys within the tile

    // S[16 heads x 16 keys] = Q . K^T
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int kp = 0; kp < kD / 32; ++kp) {  // pairs of k-steps (32 features)
        // matrix m (0..3) = keys nt*8..+7, features kp*32 + m*8 .. +7
        const int r = wkey0 + nt * 8 + (lane & 7);
        const int c = kp * 4 + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(ks + tile_off<D>(r, c), b0, b1, b2, b3);
        mma_bf16_16816(s[nt], qa[2 * kp], b0, b1);
        mma_bf16_16816(s[nt], qa[2 * kp + 1], b2, b3);
      }
    }
    // mask keys past the split end, scale into log2 units
    const int key_base = k_begin + t * kTileKeys + wkey0;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key_base + nt * 8 + 2 * tq + (e & 1);
        s[nt][e] = key < k_end ? s[nt][e] * a.scale_log2 : -INFINITY;
      }
    }
    // online softmax per row (rows gr and gr + 8)
    float mx_lo = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mx_hi = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    // a row whose keys are all masked so far keeps max -inf: use 0 as base
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
    for (int i = 0; i < kD / 8; ++i) {
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
    // O[16 x D] += P[16 x 16 keys] . V[16 keys x D]
#pragma unroll
    for (int np = 0; np < kD / 16; ++np) {  // pairs of 8-wide feature tiles
      // matrices: (keys 0-7, f 0-7), (keys 8-15, f 0-7), (keys 0-7, f 8-15), (keys 8-15, f 8-15)
      const int r = wkey0 + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int c = np * 2 + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(vs + tile_off<D>(r, c), b0, b1, b2, b3);
      mma_bf16_16816(o[2 * np], pa, b0, b1);
      mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // full row sums inside each quad
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);

  // merge the 4 warps through shared memory (reuses the ring)
  float* so = reinterpret_cast<float*>(smem);            // [warps][16][D]
  float* sml = so + kWarps * 16 * kD;                    // [warps][16][2]
#pragma unroll
  for (int nt = 0; nt < kD / 8; ++nt) {
    const int col = nt * 8 + 2 * tq;
    so[(warp * 16 + gr) * kD + col] = o[nt][0];
    so[(warp * 16 + gr) * kD + col + 1] = o[nt][1];
    so[(warp * 16 + gr + 8) * kD + col] = o[nt][2];
    so[(warp * 16 + gr + 8) * kD + col + 1] = o[nt][3];
  }
  if (tq == 0) {
    sml[(warp * 16 + gr) * 2] = m_lo;
    sml[(warp * 16 + gr) * 2 + 1] = l_lo;
    sml[(warp * 16 + gr + 8) * 2] = m_hi;
    sml[(warp * 16 + gr + 8) * 2 + 1] = l_hi;
  }
  __syncthreads();
  const int H2 = 2 * a.h;
  for (int idx = tid; idx < G * kD; idx += kWarps * 32) {
    const int row = idx / kD, col = idx % kD;
    float mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mt = fmaxf(mt, sml[(w * 16 + row) * 2]);
    const float base = mt == -INFINITY ? 0.f : mt;
    float lt = 0.f, ot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = fast_exp2(sml[(w * 16 + row) * 2] - base);
      lt += sml[(w * 16 + row) * 2 + 1] * f;
      ot += so[(w * 16 + row) * kD + col] * f;
    }
    const int64_t pidx = (static_cast<int64_t>(split) * a.B + b) * H2 + qh0 + row;
    a.part_o[pidx * kD + col] = ot;
    if (col == 0) {
      a.part_ml[pidx * 2] = mt;
      a.part_ml[pidx * 2 + 1] = lt;
    }
  }
}

// Merge the splits of one pair and apply the gate.  Block = d threads, one
// feature each; grid (h, B).
__global__ void __launch_bounds__(128)
decode_merge_kernel(DecodeArgs a) {
  const int p = blockIdx.x, b = blockIdx.y, col = threadIdx.x;
  const int H2 = 2 * a.h;
  float res[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = 2 * p + e;
    float mt = -INFINITY;
    for (int s = 0; s < a.num_splits; ++s)
      mt = fmaxf(mt, a.part_ml[((static_cast<int64_t>(s) * a.B + b) * H2 + j) * 2]);
    const float base = mt == -INFINITY ? 0.f : mt;
    float lt = 0.f, ot = 0.f;
    for (int s = 0; s < a.num_splits; ++s) {
      const int64_t pidx = (static_cast<int64_t>(s) * a.B + b) * H2 + j;
      const float f = exp2f(a.part_ml[pidx * 2] - base);
      lt += a.part_ml[pidx * 2 + 1] * f;
      ot += a.part_o[pidx * a.d + col] * f;
    }
    res[e] = lt > 0.f ? ot / lt : 0.f;
  }
  const float gte = a.gate[static_cast<int64_t>(b) * a.h + p];
  const float y = __fsub_rn(res[0], __fmul_rn(gte, res[1]));
  static_cast<__nv_bfloat16*>(a.out)[(static_cast<int64_t>(b) * a.h + p) * a.d + col] =
      __float2bfloat16_rn(y);
}

template <int D>
cudaError_t launch_split(const DecodeArgs& a, cudaStream_t s) {
  // set on every launch: the attribute is per device, and the call is cheap
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 g1(a.num_splits, a.h_kv, a.B);
  decode_split_kernel<D><<<g1, kWarps * 32, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = a.d == 128 ? launch_split<128>(a, s) : a.d == 64 ? launch_split<64>(a, s)
                                                                    : cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  dim3 g2(a.h, a.B);
  decode_merge_kernel<<<g2, a.d, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace da
