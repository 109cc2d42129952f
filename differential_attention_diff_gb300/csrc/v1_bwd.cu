// v1_bwd.cu — V1 differential attention backward (bf16) on tcgen05 + TMEM +
// TMA with 2-CTA clusters, sm_103a.
//
// The method pages ("Differential Transformer | ICLR 2025 Oral", dainus.ai,
// "Differential Attention: 빼기의 힘"; "Differential Transformer V2",
// pogovet.com, §1) define the forward; this is its chain rule.  With
// c = 1 - lambda_init, w the RMSNorm weight (fixed; unit by default),
// Yhat = Y / (c w) = O * rstd, G = dY, s = softmax scale:
//   dO  = c * rstd * (w G - Yhat * mean(w G * Yhat))    (RMSNorm backward)
//   D1  = <dO, A1 V> = <dO, O + lambda O2>,   D2 = <dO, A2 V>
//   dP  = dO V^T  (shared by both streams)
//   dS1 = A1 (dP - D1),   dS2 = -lambda A2 (dP - D2)
//   dQt = s dSt Kt,  dKt = s dSt^T Qt,  dV = (A1 - lambda A2)^T dO
//   dlambda = -sum D2;  lambda = e^a - e^b + lambda_init with a = lq1.lk1,
//   b = lq2.lk2:  dlq1 = dlambda e^a lk1, dlk1 = dlambda e^a lq1,
//   dlq2 = -dlambda e^b lk2, dlk2 = -dlambda e^b lq2.
//
// Three launches:
//  1. preprocess (one warp per row): dO (bf16, workspace), D1, D2, the LSEs in
//     log2 units (padded to whole 64-row tiles), zeroed dQ accumulators, and
//     per-block partial sums of -D2 for dlambda;
//  2. main (tcgen05): a work item is (batch, head, 128-key tile); a cluster
//     of two CTAs runs it, rank 0 for stream 1 and rank 1 for stream 2.  Each
//     CTA keeps its K tile and the V tile in shared memory and walks the
//     64-row query tiles at and after the diagonal (all of them when not
//     causal):
//        S^T  = K Q^T          (TMEM, 64 columns)
//        dP^T = V dO^T         (TMEM, 64 columns)
//        softmax warps (thread = key row), in two steps so that each overlaps
//        an MMA: (1) once S^T is in, P = exp2(S^T s log2e - lse2) and P^T
//          as bf16 over the S^T columns just read, while dP^T is still
//          being computed;
//          (2) once dP^T is in, dS^T = sigma s P (dP^T - D) as bf16 into
//          shared memory, while dV runs
//        dV  += P^T dO         (TMEM, 256 columns; A operand from TMEM),
//                               issued after step (1); the stream's sign
//                               and lambda (sigma = 1 or -lambda) multiply
//                               the fp32 accumulator at the end
//        dQ^T = K^T dS^T       (TMEM, reusing the dP^T columns) -> read by the
//                               dQ warps, staged in shared memory in two
//                               halves and added to the fp32 accumulator
//                               with TMA reduce-adds
//        dK  += dS^T Q         (TMEM, 128 columns; A operand dS^T from shared
//                               memory, so that S^T of the next tile can be
//                               issued right after dV when its Q tile has
//                               landed, ahead of dQ^T and dK)
//     At the end each CTA writes its dK; the dV halves of the two streams,
//     each times its sigma, are summed through distributed shared memory and
//     written as bf16;
//  3. finalize: dQ accumulators -> bf16, and the lambda-vector gradients.
// Deterministic mode: the main kernel stores each dQ tile (TMA store) into a
// slot of its own, (key tile, query tile) compacted to the causal tiles (all
// pairs when not causal), and the finalize sums a row's slots in ascending
// key-tile order instead of
// reading an accumulator, so no result depends on the order in which CTAs
// finish.
//
// Warp roles (320 threads): 0-3 softmax / dS and the epilogue, 4-7 dQ readback
// and reduce, 8 TMA producer, 9 MMA issuer.  TMEM: [0,256) dV, [256,384) dK,
// [384,448) S^T (then P^T), [448,512) dP^T / dQ^T.  TMEM is full,
// so S^T and dP^T are single-buffered; taking the dQ readback off the softmax
// warps keeps it out of the per-tile chain.
// SMEM: K 32 KB, V 64 KB, 2 stages of (Q 16 KB, dO 32 KB), dQ staging of one
//       64-feature half (16 KB), dS^T 16 KB, lse2 and D of both stages (1 KB);
//       every bf16 operand in 128-byte-swizzled 64-column boxes.
#include <type_traits>

#include "kernels.h"
#include "softmax.cuh"
#include "tma.cuh"

namespace da {
namespace {

constexpr int kKT = 128;   // keys per item
constexpr int kQT = 64;    // queries per iteration
constexpr int kThreads = 320;
// Head dims (DQK, DV = 2 DQK) = (128, 256) or (64, 128).  The shared-memory
// layout below is the (128, 256) one; (64, 128) fills the first half of each
// K, V, Q and dO region.

constexpr int kBoxK = 128 * 128;   // 64 columns x 128 rows of bf16
constexpr int kBoxQ = 64 * 128;    // 64 columns x 64 rows
constexpr int kOffK = 0;                           // 2 boxes  (32 KB)
constexpr int kOffV = kOffK + 2 * kBoxK;           // 4 boxes  (64 KB)
constexpr int kOffStage = kOffV + 4 * kBoxK;       // 96 KB
constexpr int kStageQ = 0;                         // 2 boxes (16 KB)
constexpr int kStageDO = 2 * kBoxQ;                // 4 boxes (32 KB)
constexpr int kStageBytes = 6 * kBoxQ;             // 48 KB
constexpr int kOffStg = kOffStage + 2 * kStageBytes;  // dQ staging: fp32 [64 queries][64 features]
constexpr int kOffDS = kOffStg + kBoxK;            // 16 KB each
constexpr int kOffLse = kOffDS + kBoxK;            // [stage] {lse2[64], D[64]}: 512 B each
constexpr int kOffBar = kOffLse + 1024;
constexpr int kSmemBytes = kOffBar + 512 + 1024;   // 231936 <= 232448

enum {
  B_KV = 0, B_QFULL, B_QFULL1, B_QEMPTY, B_QEMPTY1, B_SFULL, B_DPFULL, B_PREADY, B_PFULL, B_DQFULL,
  B_DQFREE, B_ACC, B_RTR, B_DATA, B_STG0, B_STG1, B_FREE0, B_FREE1, B_COUNT
};

__host__ __device__ constexpr uint32_t idesc2(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kIdS = idesc2(128, 64, 0, 0);    // K (K-major) x Q (K-major)
constexpr uint32_t kIdDP = idesc2(128, 64, 0, 0);   // V (K-major) x dO (K-major)
constexpr uint32_t kIdDQ = idesc2(128, 64, 1, 1);   // K^T (MN-major) x dS^T (MN-major)
// per head dims: P^T (TMEM) x dO (MN-major) is idesc2(128, DV, 0, 1),
// dS^T (TMEM) x Q (MN-major) is idesc2(128, DQK, 0, 1)

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

struct Shared {
  uint32_t base;
  uint8_t* gen;
  __device__ uint32_t bar(int i) const { return base + kOffBar + 8 * i; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(gen + kOffBar + 256); }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(gen + kOffBar + 264);
  }
  __device__ float* lam() const { return reinterpret_cast<float*>(gen + kOffBar + 268); }
};

__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(const Shared& sh, uint32_t bar, uint32_t parity,
                                         uint32_t* status, uint32_t site) {
  auto poll = [&]() { return kCluster ? try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (poll()) return true;
    if (*sh.abort_flag()) return false;
    if (globaltimer() - t0 > 2000000000ull) {
      record_status(status, DA_ERR_TIMEOUT, site);
      *sh.abort_flag() = 1;
      return false;
    }
  }
}

// Non-blocking test of a phase (try_wait may suspend the thread for a
// while before it reports an incomplete phase; test_wait returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// an arrive on a cluster peer's barrier with a CTA-scope release: enough where
// the hand-off orders only tensor-core and asynchronous-proxy accesses (a
// cluster-scope release costs the arriving thread about a microsecond)
__device__ __forceinline__ void remote_arrive_cta(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// 16 bytes into a cluster peer's shared memory, completion counted in bytes
// on the peer's mbarrier
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar_cluster) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar_cluster)
               : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// --------------------------------------------------------------------------
// Workspace carve-up (all offsets 256-byte aligned).
struct BwdWs {
  __nv_bfloat16* dO;   // [B, N, H, d_v]
  float* lse2[2];      // [B, H, Npad]  (LSE * log2 e; +inf in padding rows)
  float* D[2];         // [B, H, Npad]
  float* dq[2];        // [B, N, H, d_qk] fp32 accumulators, or (deterministic)
                       // [B*H, n_slots, 64, d_qk] per-tile slots
  float* dlam_part;    // [preprocess blocks]
  int npad, pre_blocks;
  int det, causal, n_kt, n_qt, n_slots;
};

// Slot of the dQ tile of (key tile kt, query tile qt).  Causal: qt >= 2 kt,
// and the causal tiles of key tiles 0 .. kt-1 come first.  Not causal: every
// pair, key-tile major.
__host__ __device__ __forceinline__ int dq_slot(int kt, int qt, int n_qt, int causal) {
  return causal ? kt * n_qt - kt * (kt - 1) + (qt - 2 * kt) : kt * n_qt + qt;
}

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int kPreWarps = 8;

BwdWs carve(void* base, int B, int N, int H, int dqk, int dv, bool det, bool causal, size_t* total) {
  BwdWs w;
  w.npad = (N + kQT - 1) / kQT * kQT;
  w.det = det ? 1 : 0;
  w.causal = causal ? 1 : 0;
  w.n_kt = (N + kKT - 1) / kKT;
  w.n_qt = w.npad / kQT;
  w.n_slots = causal ? w.n_kt * w.n_qt - w.n_kt * (w.n_kt - 1) : w.n_kt * w.n_qt;
  w.pre_blocks = static_cast<int>((static_cast<long long>(B) * H * w.npad + kPreWarps - 1) / kPreWarps);
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* r = p ? p + off : nullptr;
    off += a256(bytes);
    return r;
  };
  const size_t rows = static_cast<size_t>(B) * N * H;
  const size_t srow = static_cast<size_t>(B) * H * w.npad;
  w.dO = reinterpret_cast<__nv_bfloat16*>(take(rows * dv * 2));
  for (int t = 0; t < 2; ++t) w.lse2[t] = reinterpret_cast<float*>(take(srow * 4));
  for (int t = 0; t < 2; ++t) w.D[t] = reinterpret_cast<float*>(take(srow * 4));
  const size_t dq_elems = det ? static_cast<size_t>(B) * H * w.n_slots * kQT * dqk : rows * dqk;
  for (int t = 0; t < 2; ++t) w.dq[t] = reinterpret_cast<float*>(take(dq_elems * 4));
  w.dlam_part = reinterpret_cast<float*>(take(static_cast<size_t>(w.pre_blocks) * 4));
  if (total) *total = off;
  return w;
}

__device__ __forceinline__ float lambda_dev(const V1BwdArgs& a, int lane, float* ea, float* eb) {
  float d1 = 0.f, d2 = 0.f;
  for (int x = lane; x < a.d_qk; x += 32) {
    d1 = fmaf(a.lq1[x], a.lk1[x], d1);
    d2 = fmaf(a.lq2[x], a.lk2[x], d2);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    d1 += __shfl_xor_sync(0xffffffffu, d1, o);
    d2 += __shfl_xor_sync(0xffffffffu, d2, o);
  }
  const float e1 = expf(d1), e2 = expf(d2);
  if (ea) *ea = e1;
  if (eb) *eb = e2;
  return e1 - e2 + a.lambda_init;
}

// ------------------------------------------------------------ preprocess --
// kF consecutive bf16 values (kF = 8 or 4) / zeroed fp32 values (4 or 2)
template <int kF>
__device__ __forceinline__ void ld_bf16(const __nv_bfloat16* p, __nv_bfloat16 (&v)[kF]) {
  if constexpr (kF == 8) {
    *reinterpret_cast<uint4*>(v) = *reinterpret_cast<const uint4*>(p);
  } else {
    *reinterpret_cast<uint2*>(v) = *reinterpret_cast<const uint2*>(p);
  }
}
template <int kF>
__device__ __forceinline__ void st_zero_f32(float* p) {
  if constexpr (kF == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    *reinterpret_cast<float2*>(p) = make_float2(0.f, 0.f);
  }
}

// one warp per row; lane = DV / 32 consecutive V features
template <int DQK, int DV>
__global__ void __launch_bounds__(kPreWarps * 32)
v1_bwd_pre_kernel(V1BwdArgs a, BwdWs w) {
  constexpr int kF = DV / 32, kFq = DQK / 32;
  __shared__ float s_lam;
  __shared__ float s_part[kPreWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    const float lam = lambda_dev(a, lane, nullptr, nullptr);
    if (lane == 0) s_lam = lam;
  }
  __syncthreads();
  const float lam = s_lam;
  const float c = 1.f - a.lambda_init;
  const long long row = static_cast<long long>(blockIdx.x) * kPreWarps + warp;  // over (b, h, n < npad)
  const long long total = static_cast<long long>(a.B) * a.H * w.npad;
  float part = 0.f;
  if (row < total) {
    const int n = static_cast<int>(row % w.npad);
    const int bh = static_cast<int>(row / w.npad);
    const int b = bh / a.H, h = bh % a.H;
    if (n < a.N) {
      const __nv_bfloat16* yp = static_cast<const __nv_bfloat16*>(a.out.ptr) + b * a.out.sb +
                                static_cast<int64_t>(n) * a.out.sn + h * a.out.sh + lane * kF;
      const __nv_bfloat16* gp = static_cast<const __nv_bfloat16*>(a.dout.ptr) + b * a.dout.sb +
                                static_cast<int64_t>(n) * a.dout.sn + h * a.dout.sh + lane * kF;
      const __nv_bfloat16* op = static_cast<const __nv_bfloat16*>(a.o2.ptr) + b * a.o2.sb +
                                static_cast<int64_t>(n) * a.o2.sn + h * a.o2.sh + lane * kF;
      __nv_bfloat16 ye[kF], ge[kF], oe[kF];
      ld_bf16<kF>(yp, ye);
      ld_bf16<kF>(gp, ge);
      ld_bf16<kF>(op, oe);
      const int64_t sidx = (static_cast<int64_t>(b) * a.H + h) * a.N + n;
      const float rstd = a.rstd[sidx];
      const float inv_c = c != 0.f ? 1.f / c : 0.f;
      // yh = Y / (c w) is the normalised O, g = w G; then dOhat = c g
      float yh[kF], g[kF], o2[kF], gy = 0.f;
#pragma unroll
      for (int e = 0; e < kF; ++e) {
        yh[e] = __bfloat162float(ye[e]) * inv_c;
        g[e] = __bfloat162float(ge[e]);
        if (a.rms_weight) {
          const float wv = a.rms_weight[lane * kF + e];
          yh[e] = yh[e] / wv;
          g[e] = g[e] * wv;
        }
        o2[e] = __bfloat162float(oe[e]);
        gy = fmaf(g[e], yh[e], gy);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gy += __shfl_xor_sync(0xffffffffu, gy, o);
      const float mean_gy = gy * (1.f / DV);
      const float k = c * rstd;
      const float inv_rstd = 1.f / rstd;
      float d1 = 0.f, d2 = 0.f;
      uint32_t pk[kF / 2];
#pragma unroll
      for (int e = 0; e < kF; e += 2) {
        const float do0 = k * (g[e] - yh[e] * mean_gy);
        const float do1 = k * (g[e + 1] - yh[e + 1] * mean_gy);
        // round dO to bf16 once; D1 / D2 use the rounded values the MMAs see
        pk[e / 2] = pack_bf16x2(do0, do1);
        const __nv_bfloat162 r = *reinterpret_cast<const __nv_bfloat162*>(&pk[e / 2]);
        const float r0 = __low2float(r), r1 = __high2float(r);
        const float o_0 = yh[e] * inv_rstd, o_1 = yh[e + 1] * inv_rstd;
        d1 = fmaf(r0, fmaf(lam, o2[e], o_0), d1);
        d1 = fmaf(r1, fmaf(lam, o2[e + 1], o_1), d1);
        d2 = fmaf(r0, o2[e], d2);
        d2 = fmaf(r1, o2[e + 1], d2);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        d1 += __shfl_xor_sync(0xffffffffu, d1, o);
        d2 += __shfl_xor_sync(0xffffffffu, d2, o);
      }
      const int64_t rrow = (static_cast<int64_t>(b) * a.N + n) * a.H + h;
      if constexpr (kF == 8) {
        *reinterpret_cast<uint4*>(w.dO + rrow * DV + lane * kF) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      } else {
        *reinterpret_cast<uint2*>(w.dO + rrow * DV + lane * kF) = make_uint2(pk[0], pk[1]);
      }
      if (!w.det) {
        st_zero_f32<kFq>(w.dq[0] + rrow * DQK + lane * kFq);
        st_zero_f32<kFq>(w.dq[1] + rrow * DQK + lane * kFq);
      }
      if (lane == 0) {
        const int64_t pidx = static_cast<int64_t>(bh) * w.npad + n;
        w.D[0][pidx] = d1;
        w.D[1][pidx] = d2;
        w.lse2[0][pidx] = a.lse1[sidx] * 1.4426950408889634f;
        w.lse2[1][pidx] = a.lse2[sidx] * 1.4426950408889634f;
        part = -d2;
      }
    } else if (lane == 0) {
      const int64_t pidx = static_cast<int64_t>(bh) * w.npad + n;
      w.D[0][pidx] = 0.f;
      w.D[1][pidx] = 0.f;
      w.lse2[0][pidx] = INFINITY;
      w.lse2[1][pidx] = INFINITY;
    }
  }
  if (lane == 0) s_part[warp] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int i = 0; i < kPreWarps; ++i) s += s_part[i];
    w.dlam_part[blockIdx.x] = s;
  }
}

// -------------------------------------------------------------- main -------
struct Item {
  int b, h, kt, i0, n_it;
};

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
v1_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q1, const __grid_constant__ CUtensorMap tm_q2,
                   const __grid_constant__ CUtensorMap tm_k1, const __grid_constant__ CUtensorMap tm_k2,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq1, const __grid_constant__ CUtensorMap tm_dq2,
                   V1BwdArgs a, BwdWs w) {
  extern __shared__ uint8_t smem_raw[];
  Shared sh;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t al = (raw + 1023u) & ~1023u;
    sh.base = al;
    sh.gen = smem_raw + (al - raw);
  }
  constexpr int kDqk = DQK, kDv = DV;
  constexpr int kNQ = DQK / 64, kNV = DV / 64;  // 64-column boxes per tile row
  constexpr uint32_t kIdDV = idesc2(128, DV, 0, 1);   // P^T (TMEM) x dO (MN-major)
  constexpr uint32_t kIdDK = idesc2(128, DQK, 0, 1);  // dS^T (TMEM) x Q (MN-major)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // stream index
  const uint32_t partner = rank ^ 1u;
  // items: heaviest (first key tiles: most query tiles) first
  const int n_qt = w.npad / kQT;
  Item it;
  {
    const int ci = blockIdx.x >> 1;
    const int units = a.B * a.H;
    it.kt = ci / units;
    const int u = ci % units;
    it.b = u / a.H;
    it.h = u % a.H;
    it.i0 = a.causal ? it.kt * (kKT / kQT) : 0;  // causal: query tiles from the diagonal on
    it.n_it = n_qt - it.i0;
  }
  const CUtensorMap* tq = rank == 0 ? &tm_q1 : &tm_q2;
  const CUtensorMap* tk = rank == 0 ? &tm_k1 : &tm_k2;
  const float* lse2 = w.lse2[rank];
  const CUtensorMap* tdq = rank == 0 ? &tm_dq1 : &tm_dq2;
  const float* Dv = w.D[rank];

  // the item's K and V tiles, and query tile k's Q, dO, lse2 and D into
  // stage k & 1 (issued by one thread)
  const size_t srow = (static_cast<size_t>(it.b) * a.H + it.h) * w.npad;
  auto load_kv = [&]() {
    mbar_arrive_expect_tx(sh.bar(B_KV), (kNQ + kNV) * kBoxK);
    for (int box = 0; box < kNQ; ++box)
      tma_load_4d(sh.base + kOffK + box * kBoxK, tk, sh.bar(B_KV), box * 64, it.h, it.kt * kKT, it.b);
    for (int box = 0; box < kNV; ++box)
      tma_load_4d(sh.base + kOffV + box * kBoxK, &tm_v, sh.bar(B_KV), box * 64, it.h, it.kt * kKT, it.b);
  };
  auto load_q = [&](int k) {
    const int st = k & 1;
    const int q0 = (it.i0 + k) * kQT;
    const uint32_t sb = sh.base + kOffStage + st * kStageBytes;
    mbar_arrive_expect_tx(sh.bar(B_QFULL + st), (kNQ + kNV) * kBoxQ + 512);
    for (int box = 0; box < kNQ; ++box)
      tma_load_4d(sb + kStageQ + box * kBoxQ, tq, sh.bar(B_QFULL + st), box * 64, it.h, q0, it.b);
    for (int box = 0; box < kNV; ++box)
      tma_load_4d(sb + kStageDO + box * kBoxQ, &tm_do, sh.bar(B_QFULL + st), box * 64, it.h, q0, it.b);
    const uint32_t lb = sh.base + kOffLse + st * 512;
    bulk_load(lb, lse2 + srow + q0, 256, sh.bar(B_QFULL + st));
    bulk_load(lb + 256, Dv + srow + q0, 256, sh.bar(B_QFULL + st));
  };
  if (threadIdx.x == 0) {
    mbar_init(sh.bar(B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(sh.bar(B_QFULL + s), 1);
      mbar_init(sh.bar(B_QEMPTY + s), 1);
    }
    mbar_init(sh.bar(B_SFULL), 1);
    mbar_init(sh.bar(B_DPFULL), 1);
    mbar_init(sh.bar(B_PREADY), 128);
    mbar_init(sh.bar(B_PFULL), 128);
    mbar_init(sh.bar(B_DQFULL), 1);
    mbar_init(sh.bar(B_DQFREE), 128);
    mbar_init(sh.bar(B_ACC), 1);
    mbar_init(sh.bar(B_RTR), 1);   // the partner's MMAs are done: its V region may take my half of dV
    mbar_init(sh.bar(B_DATA), 1);  // + the bytes of the partner's half
    for (int h = 0; h < 2; ++h) {
      mbar_init(sh.bar(B_STG0 + h), 64);
      mbar_init(sh.bar(B_FREE0 + h), 1);
    }
    *sh.abort_flag() = 0;
    fence_mbar_init();
    // the loads that need no stage released go out now, under the rest of
    // the set-up (TMEM allocation, lambda, the cluster barrier): they touch
    // only this CTA's shared memory and barriers
    load_kv();
    for (int k = 0; k < 2 && k < it.n_it; ++k) load_q(k);
  }
  if (warp == 0) {
    const float lam = lambda_dev(a, lane, nullptr, nullptr);
    if (lane == 0) *sh.lam() = lam;
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(sh.tmem_slot()), 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(tq);
    prefetch_tmap(tk);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
    prefetch_tmap(tdq);
  }
  if (DQK < 128 && warp < 4) {
    // dQ^T = K^T dS^T runs with M = 128 feature rows: with d_qk = 64 the
    // second 64-column box of the K tile is never loaded, so zero it once
    // (feature rows 64-127 of dQ^T come out zero and are not staged)
    uint4* zk = reinterpret_cast<uint4*>(sh.gen + kOffK + kBoxK);
    for (int i = threadIdx.x; i < kBoxK / 16; i += 128) zk[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot();
  const uint32_t T_DV = tmem, T_DK = tmem + 256, T_S = tmem + 384, T_DP = tmem + 448;

  if (warp == 8) {
    // ---------------------------------------------------- TMA producer ----
    if (lane == 0) {
      // K, V and the first two query tiles were issued at set-up
      int last = min(2, it.n_it) - 1;
      bool ok = true;
      for (int k = 2; k < it.n_it; ++k) {
        const int st = k & 1, use = k >> 1;
        if (!wait_bar(sh, sh.bar(B_QEMPTY + st), (use - 1) & 1, a.status, 0x4001)) {
          ok = false;
          break;
        }
        load_q(k);
        last = k;
      }
      if (!ok) {
        // give the loads already issued (bounded) time to land before exit
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000000ull && !mbar_try_wait(sh.bar(B_KV), 0)) {
        }
        for (int k = last; k >= 0 && k > last - 2; --k)
          while (globaltimer() - t0 < 400000000ull && !mbar_try_wait(sh.bar(B_QFULL + (k & 1)), (k >> 1) & 1)) {
          }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0) {
      bool ok = wait_bar(sh, sh.bar(B_KV), 0, a.status, 0x4101);
      tc_fence_after();
      const uint32_t kA = sh.base + kOffK, vA = sh.base + kOffV;
      auto stage = [&](int k) { return sh.base + kOffStage + (k & 1) * kStageBytes; };
      auto issue_s = [&](int k) {  // S^T = K Q^T
        const uint32_t qb = stage(k) + kStageQ;
#pragma unroll
        for (int kk = 0; kk < kDqk / 16; ++kk) {
          const uint32_t offa = (kk >> 2) * kBoxK + (kk & 3) * 32;
          const uint32_t offb = (kk >> 2) * kBoxQ + (kk & 3) * 32;
          tc_mma_ss(T_S, sdesc_sw128(kA + offa, 16, 1024), sdesc_sw128(qb + offb, 16, 1024), kIdS, kk > 0);
        }
        tc_commit(sh.bar(B_SFULL));
      };
      auto issue_dp = [&](int k) {  // dP^T = V dO^T
        const uint32_t db = stage(k) + kStageDO;
#pragma unroll
        for (int kk = 0; kk < kDv / 16; ++kk) {
          const uint32_t offa = (kk >> 2) * kBoxK + (kk & 3) * 32;
          const uint32_t offb = (kk >> 2) * kBoxQ + (kk & 3) * 32;
          tc_mma_ss(T_DP, sdesc_sw128(vA + offa, 16, 1024), sdesc_sw128(db + offb, 16, 1024), kIdDP, kk > 0);
        }
        tc_commit(sh.bar(B_DPFULL));
      };
      const uint32_t dsA = sh.base + kOffDS;
      if (ok && it.n_it > 0) {
        if (wait_bar(sh, sh.bar(B_QFULL), 0, a.status, 0x4102)) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        } else {
          ok = false;
        }
      }
      for (int k = 0; k < it.n_it && ok; ++k) {
        const int ph = k & 1;
        const uint32_t db = stage(k) + kStageDO, qb = stage(k) + kStageQ;
        // dV += P^T dO as soon as P^T is in TMEM (S^T columns 0-31):
        // it runs while the softmax warps form dS^T
        if (!wait_bar(sh, sh.bar(B_PREADY), ph, a.status, 0x4106)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kQT / 16; ++kk)
          tc_mma_ts(T_DV, T_S + kk * 8, sdesc_sw128(db + kk * 2048, kBoxQ, 1024), kIdDV, (k > 0 || kk > 0) ? 1u : 0u);
        // S^T(k+1) may overwrite P^T(k) as soon as dV(k) is issued (in
        // order on the tensor pipe; dK takes dS^T from shared memory): issue
        // it now when its Q tile has landed, so the softmax warps can start
        // on it while dQ^T(k) and dK(k) run; else after them
        const int k1 = k + 1;
        bool s_next = false;
        if (k1 < it.n_it && mbar_test_wait(sh.bar(B_QFULL + (k1 & 1)), (k1 >> 1) & 1)) {
          tc_fence_after();
          issue_s(k1);
          s_next = true;
        }
        if (!wait_bar(sh, sh.bar(B_PFULL), ph, a.status, 0x4103)) { ok = false; break; }
        tc_fence_after();
        // dQ^T = K^T dS^T  (into the dP^T columns, already read)
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk)
          tc_mma_ss(T_DP, sdesc_sw128(kA + kk * 2048, kBoxK, 1024), sdesc_sw128(dsA + kk * 2048, kBoxQ, 1024),
                    kIdDQ, kk > 0);
        tc_commit(sh.bar(B_DQFULL));
        // dK += dS^T Q  (dS^T K-major in shared memory)
#pragma unroll
        for (int kk = 0; kk < kQT / 16; ++kk)
          tc_mma_ss(T_DK, sdesc_sw128(dsA + kk * 32, 16, 1024), sdesc_sw128(qb + kk * 2048, kBoxQ, 1024), kIdDK,
                    (k > 0 || kk > 0) ? 1u : 0u);
        tc_commit(sh.bar(B_QEMPTY + (k & 1)));
        if (k1 < it.n_it) {
          if (!s_next) {
            if (!wait_bar(sh, sh.bar(B_QFULL + (k1 & 1)), (k1 >> 1) & 1, a.status, 0x4104)) { ok = false; break; }
            tc_fence_after();
            issue_s(k1);
          }
          // dP^T(k+1) overwrites dQ^T(k) once the dQ warps have read it
          if (!wait_bar(sh, sh.bar(B_DQFREE), ph, a.status, 0x4105)) { ok = false; break; }
          tc_fence_after();
          issue_dp(k + 1);
        }
      }
      if (ok) tc_commit(sh.bar(B_ACC));
    }
  } else if (warp >= 4) {
    // ------------------------------------------------- dQ readback + reduce --
    // thread = feature of dQ^T (TMEM lane); warps 4-5 stage features 0-63,
    // warps 6-7 features 64-127, one half at a time through one 16 KB buffer
    const int r = (warp - 4) * 32 + lane;
    const uint32_t loff = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const int half = (warp - 4) >> 1;
    const int col = r - half * 64;
    float* stg = reinterpret_cast<float*>(sh.gen + kOffStg);
    bool ok = true;
    for (int k = 0; k < it.n_it && ok; ++k) {
      if (!wait_bar(sh, sh.bar(B_DQFULL), k & 1, a.status, 0x4301)) { ok = false; break; }
      tc_fence_after();
      uint32_t qv[64];
      tmem_ld32(T_DP + loff, *reinterpret_cast<uint32_t(*)[32]>(&qv[0]));
      tmem_ld32(T_DP + loff + 32, *reinterpret_cast<uint32_t(*)[32]>(&qv[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(sh.bar(B_DQFREE));
      if (DQK < 128 && half == 1) continue;  // feature rows 64-127: zero padding
      // the staging buffer alternates between the halves: half 0 of tile k
      // waits until half 1 of tile k-1 has been read (FREE0), half 1 until
      // half 0 of tile k has (FREE1).  One barrier per direction completes
      // once per tile, so no waiter can be two phases away from it even when
      // the warps that do not issue the copy run a tile ahead of the one that
      // does (a single barrier shared by both halves would let such a warp
      // match an older phase of the same parity and overwrite the buffer
      // while it is still being read).
      // With d_qk = 64 there is one half: it waits for its own copy of the
      // tile before (FREE1, arrived by its issuer), again once per tile.
      if (DQK < 128 ? (k > 0 && !wait_bar(sh, sh.bar(B_FREE1), (k - 1) & 1, a.status, 0x4302))
          : half == 0 ? (k > 0 && !wait_bar(sh, sh.bar(B_FREE0), (k - 1) & 1, a.status, 0x4302))
                      : !wait_bar(sh, sh.bar(B_FREE1), k & 1, a.status, 0x4302)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c = 0; c < kQT; ++c) stg[c * 64 + col] = __uint_as_float(qv[c]);
      fence_proxy_async_smem();
      mbar_arrive(sh.bar(B_STG0 + half));
      bool stg_ok = true;
      if (col == 0) {
        stg_ok = wait_bar(sh, sh.bar(B_STG0 + half), k & 1, a.status, 0x4303);
        if (stg_ok) {
          // add the [64 queries][64 features] tile into the fp32 accumulator
          // (rows past N are dropped by the unit), or store it into its slot
          if (w.det)
            tma_store_4d(tdq, sh.base + kOffStg, half * 64, 0, dq_slot(it.kt, it.i0 + k, w.n_qt, w.causal),
                         it.b * a.H + it.h);
          else
            tma_reduce_add_4d(tdq, sh.base + kOffStg, half * 64, it.h, (it.i0 + k) * kQT, it.b);
          bulk_commit();
          bulk_wait_read();
          mbar_arrive(sh.bar(half == 0 ? B_FREE1 : B_FREE0));
        }
      }
      // keep the issuing warp uniform for the warp-collective TMEM loads
      if ((warp & 1) == 0) stg_ok = __shfl_sync(0xffffffffu, stg_ok, 0);
      if (!stg_ok) ok = false;
    }
    if (col == 0) bulk_wait_all();
  } else {
    // --------------------------------------------- softmax / dS, epilogue --
    const int r = warp * 32 + lane;  // key row within the tile = TMEM lane
    const uint32_t loff = static_cast<uint32_t>(warp * 32) << 16;
    const float lam = *sh.lam();
    const float sigma = rank == 0 ? 1.f : -lam;
    const float sds = sigma * a.scale;
    const float sl2 = a.scale * 1.4426950408889634f;
    const uint64_t sl2x2 = f2(sl2, sl2), sds2 = f2(sds, sds);
    const int key = it.kt * kKT + r;
    bool ok = true;
    uint8_t* dsbuf = sh.gen + kOffDS;
    for (int k = 0; k < it.n_it && ok; ++k) {
      const int ph = k & 1;
      const int q0 = (it.i0 + k) * kQT;
      if (!wait_bar(sh, sh.bar(B_SFULL), ph, a.status, 0x4201)) { ok = false; break; }
      tc_fence_after();
      const float4* l2v = reinterpret_cast<const float4*>(sh.gen + kOffLse + (k & 1) * 512);
      const float4* ddv = l2v + 16;
      // causal: a query of this tile may precede a key.  (Not causal: keys
      // past N are zero rows of K and V, which give dQ no contribution, and
      // their dK / dV rows are never stored.)
      const bool diag = a.causal && q0 < it.kt * kKT + kKT;
      // (1) P = exp2(S s log2e - lse2), P^T (bf16) over the S^T columns
      //     just read, the dV MMA's operand; P stays in registers for dS.
      //     sigma is applied to the fp32 dV accumulator at the end, not to
      //     this operand: bf16(-lambda P) would make even an exact P = 1
      //     inexact, and dV = P1^T dO - lambda P2^T dO can cancel strongly
      float p[64];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sv[32];
        tmem_ld32(T_S + loff + hf * 32, sv);
        tmem_ld_wait();
        uint32_t pw[16];
        auto ptile = [&](auto masked) {
          constexpr bool kMask = decltype(masked)::value;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {  // 4 queries at a time
            const float4 lq = l2v[hf * 8 + q4];
            const int c = q4 * 4;
            const int qa = q0 + hf * 32 + c;
            const uint64_t x01 = fma_f32x2(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2,
                                           f2(-lq.x, -lq.y));
            const uint64_t x23 = fma_f32x2(f2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sl2x2,
                                           f2(-lq.z, -lq.w));
            float p0 = fast_exp2(f2_lo(x01)), p1 = fast_exp2(f2_hi(x01));
            float p2 = fast_exp2(f2_lo(x23)), p3 = fast_exp2(f2_hi(x23));
            if (kMask) {
              if (key > qa) p0 = 0.f;
              if (key > qa + 1) p1 = 0.f;
              if (key > qa + 2) p2 = 0.f;
              if (key > qa + 3) p3 = 0.f;
            }
            p[hf * 32 + c] = p0;
            p[hf * 32 + c + 1] = p1;
            p[hf * 32 + c + 2] = p2;
            p[hf * 32 + c + 3] = p3;
            pw[q4 * 2] = pack_bf16x2(p0, p1);
            pw[q4 * 2 + 1] = pack_bf16x2(p2, p3);
          }
        };
        if (diag) ptile(std::true_type{});
        else ptile(std::false_type{});
        tmem_st16(T_S + loff + hf * 16, pw);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(sh.bar(B_PREADY));  // the dV MMA may read P^T
      // (2) dS^T = sigma s P (dP^T - D) (bf16) into shared memory, the
      //     operand of the dQ^T and dK MMAs (its previous readers, those MMAs
      //     of the tile before, completed before dP^T of this tile was
      //     signalled: dP^T is issued after them)
      if (!wait_bar(sh, sh.bar(B_DPFULL), ph, a.status, 0x4202)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t dp[32];
        tmem_ld32(T_DP + loff + hf * 32, dp);
        tmem_ld_wait();
        uint32_t dw[16];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 dq4 = ddv[hf * 8 + q4];
          const int c = q4 * 4;
          const uint64_t t01 = add_f32x2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), f2(-dq4.x, -dq4.y));
          const uint64_t t23 =
              add_f32x2(f2(__uint_as_float(dp[c + 2]), __uint_as_float(dp[c + 3])), f2(-dq4.z, -dq4.w));
          const uint64_t d01 = mul_f32x2(mul_f32x2(t01, f2(p[hf * 32 + c], p[hf * 32 + c + 1])), sds2);
          const uint64_t d23 = mul_f32x2(mul_f32x2(t23, f2(p[hf * 32 + c + 2], p[hf * 32 + c + 3])), sds2);
          dw[q4 * 2] = pack_bf16x2(f2_lo(d01), f2_hi(d01));
          dw[q4 * 2 + 1] = pack_bf16x2(f2_lo(d23), f2_hi(d23));
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int ch = hf * 4 + cc;
          const int off = r * 128 + ((ch ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dsbuf + off) = make_uint4(dw[cc * 4], dw[cc * 4 + 1], dw[cc * 4 + 2], dw[cc * 4 + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(sh.bar(B_PFULL));
    }
    // ----------------------------------------------------------- epilogue --
    if (ok && wait_bar(sh, sh.bar(B_ACC), 0, a.status, 0x4205)) {
      tc_fence_after();
      const bool live = key < a.N;
      // (1) dV: swap halves with the partner (the other stream) through
      //     DSMEM.  Receive buffer = this CTA's V tile region, idle now that
      //     its MMAs are done (which one arrive on the partner's RTR says):
      //     128 rows of d_v / 2 fp32, float4 j of row r at [j * 128 + r] so
      //     that a warp's 16-byte accesses are consecutive.  The partner's
      //     rows arrive as asynchronous stores counted in bytes on DATA, while
      //     this CTA writes its dK.
      constexpr int kHalf = kDv / 2;
      const int give = (1 - static_cast<int>(rank)) * kHalf, keep = static_cast<int>(rank) * kHalf;
      if (r == 0) {
        mbar_arrive_expect_tx(sh.bar(B_DATA), 128 * kHalf * 4);
        remote_arrive_cta(map_to_rank(sh.bar(B_RTR), partner));
      }
      const bool rtr = wait_bar<true>(sh, sh.bar(B_RTR), 0, a.status, 0x4206);
      if (rtr) {
        const uint32_t rx = map_to_rank(sh.base + kOffV + r * 16, partner);
        const uint32_t rx_bar = map_to_rank(sh.bar(B_DATA), partner);
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(T_DV + loff + give + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            st_async_v4(rx + ((c * 32 + e) / 4) * 128 * 16,
                        make_float4(__uint_as_float(v[e]) * sigma, __uint_as_float(v[e + 1]) * sigma,
                                    __uint_as_float(v[e + 2]) * sigma, __uint_as_float(v[e + 3]) * sigma),
                        rx_bar);
        }
      }
      // (2) dK of this stream
      __nv_bfloat16* dkp = static_cast<__nv_bfloat16*>(rank == 0 ? a.dk1.ptr : a.dk2.ptr);
      const da_t4& dkt = rank == 0 ? a.dk1 : a.dk2;
#pragma unroll 1
      for (int c = 0; c < kDqk / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(T_DK + loff + c * 32, v);
        tmem_ld_wait();
        if (live) {
          __nv_bfloat16* dst = dkp + it.b * dkt.sb + static_cast<int64_t>(key) * dkt.sn + it.h * dkt.sh + c * 32;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            *reinterpret_cast<uint4*>(dst + e) = make_uint4(
                pack_bf16x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                pack_bf16x2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])),
                pack_bf16x2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5])),
                pack_bf16x2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7])));
          }
        }
      }
      // (3) dV of my columns: my stream's half plus the partner's
      if (rtr) {
        if (!wait_bar<true>(sh, sh.bar(B_DATA), 0, a.status, 0x4207)) {
          // abort path: the partner's asynchronous stores into this CTA's
          // shared memory may still be in flight; give them a short, bounded
          // time to land before this CTA can leave (barrier.cluster does not
          // wait for them)
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 100000000ull && !try_wait_cluster(sh.bar(B_DATA), 0)) {
          }
        } else {
          const float4* mine = reinterpret_cast<const float4*>(sh.gen + kOffV) + r;
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dv.ptr) + it.b * a.dv.sb +
                               static_cast<int64_t>(key) * a.dv.sn + it.h * a.dv.sh + keep;
#pragma unroll 1
          for (int c = 0; c < kHalf / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(T_DV + loff + keep + c * 32, v);
            tmem_ld_wait();
            if (live) {
#pragma unroll
              for (int e = 0; e < 32; e += 8) {
                float s8[8];
                float o8[8];
                *reinterpret_cast<float4*>(&o8[0]) = mine[((c * 32 + e) / 4) * 128];
                *reinterpret_cast<float4*>(&o8[4]) = mine[((c * 32 + e) / 4 + 1) * 128];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  // stream 1 + sigma stream 2 in a fixed order on both CTAs
                  const float own = __uint_as_float(v[e + u]) * sigma;
                  s8[u] = rank == 0 ? own + o8[u] : o8[u] + own;
                }
                *reinterpret_cast<uint4*>(dst + c * 32 + e) =
                    make_uint4(pack_bf16x2(s8[0], s8[1]), pack_bf16x2(s8[2], s8[3]),
                               pack_bf16x2(s8[4], s8[5]), pack_bf16x2(s8[6], s8[7]));
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

// -------------------------------------------------------------- finalize --
template <int DQK>
__global__ void __launch_bounds__(256)
v1_bwd_finalize_kernel(V1BwdArgs a, BwdWs w) {
  constexpr int kDqk = DQK;
  const long long rows = static_cast<long long>(a.B) * a.N * a.H;
  const long long total = rows * (kDqk / 8);
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = idx / (kDqk / 8);
    const int c8 = static_cast<int>(idx % (kDqk / 8)) * 8;
    const int h = static_cast<int>(row % a.H);
    const long long bn = row / a.H;
    const int n = static_cast<int>(bn % a.N), b = static_cast<int>(bn / a.N);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      float4 x0, x1;
      if (w.det) {
        // the key tiles that reach this query row (0 .. qt / 2 when causal,
        // all of them otherwise), in that order
        const int qt = n / kQT;
        const int kt_end = w.causal ? qt / 2 : w.n_kt - 1;
        const float* base = w.dq[t] + (static_cast<int64_t>(b) * a.H + h) * w.n_slots * (kQT * kDqk) +
                            (n % kQT) * kDqk + c8;
        x0 = make_float4(0.f, 0.f, 0.f, 0.f);
        x1 = x0;
        for (int kt = 0; kt <= kt_end; ++kt) {
          const float* src = base + static_cast<int64_t>(dq_slot(kt, qt, w.n_qt, w.causal)) * (kQT * kDqk);
          const float4 y0 = *reinterpret_cast<const float4*>(src);
          const float4 y1 = *reinterpret_cast<const float4*>(src + 4);
          x0.x += y0.x; x0.y += y0.y; x0.z += y0.z; x0.w += y0.w;
          x1.x += y1.x; x1.y += y1.y; x1.z += y1.z; x1.w += y1.w;
        }
      } else {
        const float* src = w.dq[t] + row * kDqk + c8;
        x0 = *reinterpret_cast<const float4*>(src);
        x1 = *reinterpret_cast<const float4*>(src + 4);
      }
      const da_t4& o = t == 0 ? a.dq1 : a.dq2;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(o.ptr) + b * o.sb + static_cast<int64_t>(n) * o.sn +
                           h * o.sh + c8;
      *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w),
                                                  pack_bf16x2(x1.x, x1.y), pack_bf16x2(x1.z, x1.w));
    }
  }
  if (blockIdx.x == 0) {
    __shared__ float red[256];
    float s = 0.f;
    for (int i = threadIdx.x; i < w.pre_blocks; i += 256) s += w.dlam_part[i];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
      if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
      __syncthreads();
    }
    const float dlam = red[0];
    __shared__ float ea, eb;
    if (threadIdx.x < 32) {
      float e1, e2;
      lambda_dev(a, threadIdx.x, &e1, &e2);
      if (threadIdx.x == 0) {
        ea = e1;
        eb = e2;
      }
    }
    __syncthreads();
    for (int x = threadIdx.x; x < a.d_qk; x += 256) {
      a.dlq1[x] = dlam * ea * a.lk1[x];
      a.dlk1[x] = dlam * ea * a.lq1[x];
      a.dlq2[x] = -dlam * eb * a.lk2[x];
      a.dlk2[x] = -dlam * eb * a.lq2[x];
    }
  }
}

template <int DQK, int DV>
cudaError_t launch_dims(const V1BwdArgs& a, cudaStream_t s) {
  constexpr int kDqk = DQK, kDv = DV;
  size_t total = 0;
  BwdWs w = carve(a.workspace, a.B, a.N, a.H, DQK, DV, a.deterministic != 0, a.causal != 0, &total);
  if (total > a.workspace_bytes) return cudaErrorInvalidValue;

  v1_bwd_pre_kernel<DQK, DV><<<w.pre_blocks, kPreWarps * 32, 0, s>>>(a, w);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap tq1, tq2, tk1, tk2, tv, tdo;
  da_t4 dot{w.dO, static_cast<int64_t>(a.N) * a.H * kDv, static_cast<int64_t>(a.H) * kDv, kDv};
  if (!encode_tmap_bf16_4d(&tq1, a.q1, a.B, a.N, a.H, kDqk, kQT) ||
      !encode_tmap_bf16_4d(&tq2, a.q2, a.B, a.N, a.H, kDqk, kQT) ||
      !encode_tmap_bf16_4d(&tk1, a.k1, a.B, a.N, a.H, kDqk, kKT) ||
      !encode_tmap_bf16_4d(&tk2, a.k2, a.B, a.N, a.H, kDqk, kKT) ||
      !encode_tmap_bf16_4d(&tv, a.v, a.B, a.N, a.H, kDv, kKT) ||
      !encode_tmap_bf16_4d(&tdo, dot, a.B, a.N, a.H, kDv, kQT))
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(v1_bwd_main_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_kt = (a.N + kKT - 1) / kKT;
  const int items = n_kt * a.B * a.H;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * items, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  CUtensorMap tdq1, tdq2;
  // dQ tiles leave in two 64-feature halves
  if (w.det) {
    if (!encode_tmap_f32_slots(&tdq1, w.dq[0], a.B * a.H, w.n_slots, kQT, kDqk, 64) ||
        !encode_tmap_f32_slots(&tdq2, w.dq[1], a.B * a.H, w.n_slots, kQT, kDqk, 64))
      return cudaErrorInvalidValue;
  } else if (!encode_tmap_f32_4d(&tdq1, w.dq[0], a.B, a.N, a.H, kDqk, kQT, 64) ||
             !encode_tmap_f32_4d(&tdq2, w.dq[1], a.B, a.N, a.H, kDqk, kQT, 64)) {
    return cudaErrorInvalidValue;
  }
  e = cudaLaunchKernelEx(&cfg, v1_bwd_main_kernel<DQK, DV>, tq1, tq2, tk1, tk2, tv, tdo, tdq1, tdq2, a, w);
  if (e != cudaSuccess) return e;

  const long long work = static_cast<long long>(a.B) * a.N * a.H * (kDqk / 8);
  int grid = static_cast<int>((work + 255) / 256);
  if (grid > 4 * 152) grid = 4 * 152;
  if (grid < 1) grid = 1;
  v1_bwd_finalize_kernel<DQK><<<grid, 256, 0, s>>>(a, w);
  return cudaGetLastError();
}

}  // namespace

size_t v1_bwd_workspace_bytes(int B, int N, int H, int d_qk, int d_v, int deterministic, int causal) {
  size_t total = 0;
  carve(nullptr, B, N, H, d_qk, d_v, deterministic != 0, causal != 0, &total);
  return total;
}

cudaError_t launch_v1_bwd(const V1BwdArgs& a, cudaStream_t s) {
  if (a.d_qk == 128 && a.d_v == 256) return launch_dims<128, 256>(a, s);
  if (a.d_qk == 64 && a.d_v == 128) return launch_dims<64, 128>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace da
