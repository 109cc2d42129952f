// gate.cu — V2 gate: gate[t, p] = sigmoid(sum_k x[t, k] * w_lambda[k, p]).
//
// "Differential Transformer V2" (pogovet.com), §1 and §4: the coefficient of
// the second (odd) head is projected per token and per head from the input X
// and passed through a sigmoid.  The projection is a skinny GEMM
// [T, d_model] x [d_model, h] with h <= 64, so the kernel is bound by reading
// X once from HBM: 64 tokens per CTA, X and W chunks of 64 features staged by
// a 4-deep cp.async ring (three chunks in flight while one is consumed), the
// warp MMA for the products (each warp owns 16 tokens and all h outputs), and
// the sigmoid fused into the store.
// Few tokens (decode: one per sequence) leave most SMs idle and one CTA
// streaming all of d_model, so the feature range is split over a cluster of
// S CTAs (S = 1 .. 8, chosen from the token count): each sums its slice, and
// rank r adds the S partial sums of its share of the tokens in rank order
// through distributed shared memory (a fixed order: the gate does not depend
// on timing) before the sigmoid.
#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int kTok = 64;    // tokens per CTA
constexpr int kChunk = 64;  // features per stage
constexpr int kMaxH = 64;
constexpr int kStages = 4;
constexpr int kRow = 128;   // bytes per staged row (64 bf16)
constexpr int kXBytes = kTok * kRow;
constexpr int kWBytes = kChunk * kRow;
constexpr int kStageBytes = kXBytes + kWBytes;

__device__ __forceinline__ uint32_t off8(int r, int c) {
  return static_cast<uint32_t>(r * kRow + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t cluster_rank_y() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// grid (token blocks, S); clusters of (1, S): cluster rank = feature slice
__global__ void __launch_bounds__(128)
gate_kernel(GateArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTok;
  const int S = static_cast<int>(gridDim.y);
  const int slice = S > 1 ? static_cast<int>(cluster_rank_y()) : 0;
  const int nchunks = a.d_model / kChunk / S;  // chunks of this CTA's feature slice
  const int fbase = slice * nchunks * kChunk;
  const int hc = (a.h + 7) / 8;  // 16-byte chunks per W row (padded)
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
  const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(a.w);
  const uint32_t sb = smem_u32(smem);

  auto issue = [&](int ch) {
    if (ch < nchunks) {
      const uint32_t xs = sb + (ch % kStages) * kStageBytes;
      const uint32_t ws = xs + kXBytes;
      const int f0 = fbase + ch * kChunk;
#pragma unroll
      for (int i = 0; i < (kTok * 8) / 128; ++i) {
        const int idx = i * 128 + tid;
        const int r = idx >> 3, c = idx & 7;
        const int t = t0 + r;
        const bool ok = t < a.T;
        cp_async_16(xs + off8(r, c), x + static_cast<int64_t>(ok ? t : 0) * a.x_stride + f0 + c * 8,
                    ok ? 16 : 0);
      }
      if ((a.h & 7) == 0) {
        for (int idx = tid; idx < kChunk * hc; idx += 128) {
          const int r = idx / hc, c = idx % hc;
          cp_async_16(ws + off8(r, c), w + static_cast<int64_t>(f0 + r) * a.h + c * 8, 16);
        }
      } else {
        // h not a multiple of 8: element loads, zero padding up to the chunk edge
        uint8_t* wsg = smem + (ch % kStages) * kStageBytes + kXBytes;
        for (int idx = tid; idx < kChunk * hc * 8; idx += 128) {
          const int r = idx / (hc * 8), col = idx % (hc * 8);
          const __nv_bfloat16 v = col < a.h ? w[static_cast<int64_t>(f0 + r) * a.h + col]
                                            : __float2bfloat16_rn(0.f);
          *reinterpret_cast<__nv_bfloat16*>(wsg + off8(r, col >> 3) + (col & 7) * 2) = v;
        }
      }
    }
    cp_async_commit();
  };

  float acc[kMaxH / 8][4];
#pragma unroll
  for (int i = 0; i < kMaxH / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

#pragma unroll
  for (int ch = 0; ch < kStages - 1; ++ch) issue(ch);
  for (int ch = 0; ch < nchunks; ++ch) {
    issue(ch + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const uint32_t xs = sb + (ch % kStages) * kStageBytes;
    const uint32_t ws = xs + kXBytes;
#pragma unroll
    for (int ks = 0; ks < kChunk / 16; ++ks) {
      uint32_t af[4];
      {
        // A: tokens warp*16 .. +15, features ks*16 .. +15
        const int r = warp * 16 + (lane & 15);
        const int c = ks * 2 + (lane >> 4);
        ldmatrix_x4(xs + off8(r, c), af[0], af[1], af[2], af[3]);
      }
#pragma unroll
      for (int np = 0; np < kMaxH / 16; ++np) {
        if (np * 2 < hc) {
          // B = W[k][n]: matrices (k 0-7, n 0-7), (k 8-15, n 0-7), (k 0-7, n 8-15), (k 8-15, n 8-15)
          const int r = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int c = np * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(ws + off8(r, c), b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * np], af, b0, b1);
          mma_bf16_16816(acc[2 * np + 1], af, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  const int gr = lane >> 2, tq = lane & 3;
  if (S == 1) {
#pragma unroll
    for (int nt = 0; nt < kMaxH / 8; ++nt) {
      if (nt < hc) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int t = t0 + warp * 16 + gr + half * 8;
          if (t < a.T) {
            const int col = nt * 8 + 2 * tq;
            float* gp = a.gate + static_cast<int64_t>(t) * a.h + col;
            if (col < a.h) gp[0] = 1.f / (1.f + expf(-acc[nt][half * 2]));
            if (col + 1 < a.h) gp[1] = 1.f / (1.f + expf(-acc[nt][half * 2 + 1]));
          }
        }
      }
    }
    return;
  }
  // partial sums of this slice: [64 tokens][64 columns] fp32 in the (now
  // idle) ring; every rank reads its share of the tokens from all S ranks
  float* part = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int nt = 0; nt < kMaxH / 8; ++nt) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = warp * 16 + gr + half * 8;
      const int col = nt * 8 + 2 * tq;
      part[r * kMaxH + col] = acc[nt][half * 2];
      part[r * kMaxH + col + 1] = acc[nt][half * 2 + 1];
    }
  }
  cluster_barrier();  // every rank's partials are written
  const int rows = kTok / S;  // tokens this rank finishes
  const uint32_t pbase = smem_u32(smem);
  for (int idx = tid; idx < rows * a.h; idx += 128) {
    const int r = slice * rows + idx / a.h, col = idx % a.h;
    const int t = t0 + r;
    float z = 0.f;
    for (int q = 0; q < S; ++q) z += ld_cluster_f32(pbase + static_cast<uint32_t>(r * kMaxH + col) * 4u, q);
    if (t < a.T) a.gate[static_cast<int64_t>(t) * a.h + col] = 1.f / (1.f + expf(-z));
  }
  cluster_barrier();  // no rank leaves while another may still read its partials
}

}  // namespace

cudaError_t launch_gate(const GateArgs& a, cudaStream_t s) {
  const int blocks = (a.T + kTok - 1) / kTok;
  if (blocks == 0) return cudaSuccess;
  // feature slices per token block: enough CTAs for about four per SM
  // (608 on 152 SMs), a power of two up to 8 that divides the chunk count
  const int nchunks = a.d_model / kChunk;
  int S = 1;
  while (S < 8 && blocks * S * 2 <= 608 && nchunks % (S * 2) == 0) S *= 2;
  // set on every launch: the attribute is per device, and the call is cheap
  cudaError_t e = cudaFuncSetAttribute(gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStages * kStageBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = S;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(blocks, S, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = kStages * kStageBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gate_kernel, a);
}

}  // namespace da
