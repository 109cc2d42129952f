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
//
// Many tokens (prefill) take gate_tc_kernel instead: the warp MMA above runs
// at a small fraction of the tensor cores' rate on this GPU, and at B N =
// 16384 tokens its MMAs, not HBM, set the time.  gate_tc_kernel issues
// tcgen05 MMAs (M = 128 tokens, N = 64 heads with the columns past h zero,
// K = 128 features per stage) into a TMEM accumulator, with X and W chunks
// staged by TMA (128-byte swizzle) through a 4-deep ring; one thread loads,
// one issues the MMAs, four warps read the accumulator.  With fewer token
// blocks than half the SMs the features are split over a cluster of S CTAs
// whose partials are summed through distributed shared memory in rank order,
// as above.
#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace da {
namespace {

constexpr int kTok = 64;    // tokens per CTA
constexpr int kChunk = 64;  // features per stage
constexpr int kMaxH = 64;
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
// tcgen05.ld of 8 consecutive 32-bit TMEM columns of this warp's 32 lanes
// (thread i reads lane i of the warp's quadrant)
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// grid (token blocks, S); clusters of (1, S): cluster rank = feature slice;
// kStages-deep ring
template <int kStages>
__global__ void __launch_bounds__(128)
gate_kernel(GateArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTok;
  const int S = static_cast<int>(gridDim.y);
  const int slice = S > 1 ? static_cast<int>(cluster_rank_y()) : 0;
  const int nchunks = a.d_model / kChunk / S;  // chunks of this CTA's feature slice
  // slice s takes the 64-feature chunks s, s + S, s + 2S, ...: at any moment
  // the S CTAs of a cluster read neighbouring 128-byte pieces of the same X
  // rows (S of them contiguous), not S pieces d_model / S apart
  const int hc = (a.h + 7) / 8;  // 16-byte chunks per W row (padded)
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
  const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(a.w);
  const uint32_t sb = smem_u32(smem);

  auto issue = [&](int ch) {
    if (ch < nchunks) {
      const uint32_t xs = sb + (ch % kStages) * kStageBytes;
      const uint32_t ws = xs + kXBytes;
      const int f0 = (ch * S + slice) * kChunk;
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

// ------------------------------------------------------ tcgen05 variant ----
constexpr int kTcTok = 128;                       // tokens per CTA (MMA M)
constexpr int kTcX = kTcTok * kRow;               // 16 KB: 128 tokens x 64 features (one box)
constexpr int kTcW = kChunk * kRow;               // 8 KB: 64 features x 64 heads (one box)
constexpr int kTcThreads = 192;                   // producer, MMA, 4 epilogue warps
// a stage holds kNB 64-feature boxes of X and of W
__host__ __device__ constexpr int tc_stage(int nb) { return nb * (kTcX + kTcW); }
__host__ __device__ constexpr int tc_smem(int stages, int nb) { return stages * tc_stage(nb) + 1024 + 256; }
constexpr uint32_t kTcIdesc = idesc_bf16(128, 64, 1);  // X K-major, W MN-major

// grid (token blocks, S); clusters of (1, S): rank = feature slice (a
// contiguous 1/S of d_model); a kTcStages-deep ring of kNB-box stages
template <int kTcStages, int kNB>
__global__ void __launch_bounds__(kTcThreads, 1)
gate_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, GateArgs a,
               int box_rows) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gen = smem_raw + (sb - raw);
  constexpr int kTcStage = tc_stage(kNB);
  constexpr int kStageF = kNB * kChunk;  // features per stage
  const uint32_t bars = sb + kTcStages * kTcStage;
  auto full = [&](int st) { return bars + 8 * st; };
  auto empty = [&](int st) { return bars + 8 * (kTcStages + st); };
  const uint32_t accbar = bars + 8 * 2 * kTcStages;
  uint8_t* ctrl = gen + kTcStages * kTcStage + 8 * (2 * kTcStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = static_cast<int>(gridDim.y);
  const int slice = S > 1 ? static_cast<int>(cluster_rank_y()) : 0;
  const int nchunks = a.d_model / kStageF / S;
  const int f_base = slice * nchunks * kStageF;
  const int t0 = blockIdx.x * box_rows;  // box_rows <= 128 tokens (MMA M = 128)
  // Stage ch carries the feature chunk (ch + blockIdx.x) mod nchunks: the CTAs
  // start at different chunks, so at any moment they read different rows of
  // W (and different column ranges of X) instead of all hitting the same W
  // lines together (measured 31.7 -> 30.9 us mean at 16384 tokens x 4096).
  // The accumulation order is fixed by the launch shape.
  auto load_stage = [&](int ch) {
    const int st = ch % kTcStages;
    const uint32_t xs = sb + st * kTcStage;
    const int f0 = f_base + ((ch + static_cast<int>(blockIdx.x)) % nchunks) * kStageF;
    mbar_arrive_expect_tx(full(st), kNB * (box_rows * kRow + kTcW));
    for (int bx = 0; bx < kNB; ++bx) {
      tma_load_4d(xs + bx * kTcX, &tm_x, full(st), f0 + bx * kChunk, 0, t0, 0);
      tma_load_4d(xs + kNB * kTcX + bx * kTcW, &tm_w, full(st), 0, 0, f0 + bx * kChunk, 0);
    }
  };

  if (threadIdx.x == 0) {
    for (int st = 0; st < kTcStages; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), 1);
    }
    mbar_init(accbar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // the first stages go out before the TMEM allocation and the block-wide
    // sync: the ring's first bytes are in flight while the CTA sets up
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
    for (int ch = 0; ch < kTcStages && ch < nchunks; ++ch) load_stage(ch);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------- TMA producer --
      int issued = min(kTcStages, nchunks);  // issued during set-up
      for (int ch = issued; ch < nchunks; ++ch) {
        const int st = ch % kTcStages, use = ch / kTcStages;
        if (!mbar_wait(empty(st), (use - 1) & 1, a.status, 0x7001)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        load_stage(ch);
        issued = ch + 1;
      }
      // every load issued lands before the CTA can leave (already true
      // unless a wait gave up)
      for (int ch = issued - 1; ch >= 0 && ch >= issued - kTcStages; --ch)
        mbar_wait(full(ch % kTcStages), (ch / kTcStages) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------- MMA issuer --
      bool ok = true;
      for (int ch = 0; ch < nchunks && ok; ++ch) {
        const int st = ch % kTcStages, use = ch / kTcStages;
        if (!mbar_wait(full(st), use & 1, a.status, 0x7002) || *abort_flag) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t xs = sb + st * kTcStage;
        const uint32_t ws = xs + kNB * kTcX;
#pragma unroll
        for (int kk = 0; kk < kStageF / 16; ++kk)
          tc_mma_ss(tmem, sdesc_sw128(xs + (kk >> 2) * kTcX + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(ws + (kk >> 2) * kTcW + (kk & 3) * 2048, kTcW, 1024), kTcIdesc,
                    (ch > 0 || kk > 0) ? 1u : 0u);
        tc_commit(empty(st));
      }
      (void)ok;
      tc_commit(accbar);  // also on the way out: every MMA issued completes first
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;          // token within the block
    const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool ok = mbar_wait(accbar, 0, a.status, 0x7003) && !*abort_flag;
    if (!ok) *abort_flag = 1;
    tc_fence_after();
    const int t = t0 + row;
    if (S == 1) {
      // eight heads at a time in a loop that is not unrolled: this tail runs
      // once per CTA from a cold instruction cache, and 64 inlined sigmoids
      // cost more in instruction fetch than in arithmetic (measured 30.7 ->
      // 28.9 us median at 16384 tokens x 4096 x 32 heads); h is a multiple of 8
      const bool mine = ok && row < box_rows && t < a.T;
      float* gp = a.gate + static_cast<int64_t>(t) * a.h;
#pragma unroll 1
      for (int c0 = 0; c0 < a.h; c0 += 8) {
        uint32_t r8[8];
        tmem_ld8(taddr + c0, r8);  // warp-collective: every lane, every group
        tmem_ld_wait();
        if (mine) {
#pragma unroll
          for (int e = 0; e < 8; ++e) gp[c0 + e] = 1.f / (1.f + expf(-__uint_as_float(r8[e])));
        }
      }
    } else {
      uint32_t v[64];
      tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      // partials into the (idle) ring: [128 tokens][64 heads] fp32
      float* part = reinterpret_cast<float*>(gen);
#pragma unroll
      for (int c = 0; c < 64; ++c) part[row * 64 + ((c + row) & 63)] = __uint_as_float(v[c]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (S > 1) {
    cluster_barrier();  // every rank's partials are written
    const int rows = kTcTok / S;  // tokens this rank finishes
    const uint32_t pbase = sb;
    if (warp >= 2 && !*abort_flag) {
      for (int idx = threadIdx.x - 64; idx < rows * a.h; idx += 128) {
        const int r = slice * rows + idx / a.h, col = idx % a.h;
        const int t = t0 + r;
        float z = 0.f;
        for (int qq = 0; qq < S; ++qq)
          z += ld_cluster_f32(pbase + static_cast<uint32_t>(r * 64 + ((col + r) & 63)) * 4u, qq);
        if (r < box_rows && t < a.T) a.gate[static_cast<int64_t>(t) * a.h + col] = 1.f / (1.f + expf(-z));
      }
    }
    cluster_barrier();  // no rank leaves while another may still read its partials
  }
  if (warp == 1) tmem_dealloc(tmem, 64);
}

}  // namespace

// S feature slices per token block (a power of two, at most 8, dividing the
// chunk count), a kStages-deep ring
template <int kStages>
cudaError_t launch_gate_slices(const GateArgs& a, int S, cudaStream_t s) {
  const int blocks = (a.T + kTok - 1) / kTok;
  if (blocks == 0) return cudaSuccess;
  // set on every launch: the attribute is per device, and the call is cheap
  cudaError_t e = cudaFuncSetAttribute(gate_kernel<kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kStages * kStageBytes);
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
  return cudaLaunchKernelEx(&cfg, gate_kernel<kStages>, a);
}

// tcgen05 path with S feature slices per 128-token block
// box_rows (a multiple of 8, at most 128) tokens per CTA
template <int kTcStages, int kNB>
cudaError_t launch_gate_tc(const GateArgs& a, int S, int box_rows, cudaStream_t s) {
  {
    if (box_rows <= 0 || box_rows > kTcTok || (box_rows % 8) || (a.h % 8) || a.h > 64) return cudaErrorInvalidValue;
    const int tblocks = (a.T + box_rows - 1) / box_rows;
    CUtensorMap tx, tw;
    const da_t4 xt{const_cast<void*>(a.x), 0, a.x_stride, 0};
    const da_t4 wt{const_cast<void*>(a.w), 0, a.h, 0};
    if (!encode_tmap_bf16_4d(&tx, xt, 1, a.T, 1, a.d_model, box_rows) ||
        !encode_tmap_bf16_4d(&tw, wt, 1, a.d_model, 1, a.h, kChunk))
      return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gate_tc_kernel<kTcStages, kNB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tc_smem(kTcStages, kNB));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = S;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(tblocks, S, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = tc_smem(kTcStages, kNB);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gate_tc_kernel<kTcStages, kNB>, tx, tw, a, box_rows);
  }
}

cudaError_t launch_gate(const GateArgs& a, cudaStream_t s) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 152;
  if (a.T >= 8 * kTcTok && (a.h % 8) == 0 && (a.x_stride % 8) == 0 && (a.d_model % 128) == 0) {
    // tcgen05 path, 128 tokens per CTA, stages of 128 features (256 bytes of
    // every X row: at B8192 x 4096, 64-feature stages measured 34.4 us, these
    // 30.4 us); fewer token blocks than half the SMs split d_model over a
    // cluster (S a power of two up to 4 dividing the stage count); more
    // slices at 128 blocks measured slower (2 slices: 35.5 us)
    const int tblocks = (a.T + kTcTok - 1) / kTcTok;
    const int nst = a.d_model / 128;
    int S = 1;
    while (S < 4 && 2 * tblocks * S < sms && nst % (S * 2) == 0) S *= 2;
    return launch_gate_tc<4, 2>(a, S, kTcTok, s);
  }
  const int blocks = (a.T + kTok - 1) / kTok;
  // feature slices per token block: enough CTAs for about four per SM
  // (608 on 152 SMs), a power of two up to 8 that divides the chunk count
  const int nchunks = a.d_model / kChunk;
  int S = 1;
  while (S < 8 && blocks * S * 2 <= 608 && nchunks % (S * 2) == 0) S *= 2;
  return launch_gate_slices<4>(a, S, s);
}

}  // namespace da
