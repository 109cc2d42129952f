// v2_bwd.cu — V2 differential attention backward (bf16) on tcgen05 + TMEM +
// TMA, sm_103a, plus the gradients of the gate projection.
//
// "Differential Transformer V2" (pogovet.com), §1 and §4 define the forward:
// one causal GQA attention over 2h query heads, then per token t and pair p
//   out[t, p] = O[t, 2p] - g[t, p] O[t, 2p + 1],   g = sigmoid(x[t] . W[:, p]).
// This file is its chain rule.  With G = dOut[t, p] and s the softmax scale:
//   dO_2p = G,  dO_2p+1 = -g G,  dz = -<G, O_2p+1> g (1 - g)
//   dW = X^T dz,  dX = dz W^T
//   per query head j of K/V group c:  P = exp(s Q_j K_c^T - lse_j) (causal),
//   dP = dO_j V_c^T,  dS = s P (dP - D_j),  D_j = <dO_j, O_j>
//   dQ_j = dS K_c,  dK_c += dS^T Q_j,  dV_c += P^T dO_j.
//
// Launches:
//  1. (gate from x and W when the caller passes none: the gate kernel)
//  2. preprocess (one warp per (token, pair)): dO of the odd head as bf16,
//     D of both heads, the LSEs in log2 units padded to whole 64-row tiles,
//     dz, and zeroed fp32 dQ accumulators;
//  3. main (tcgen05): a work item is (batch, K/V group, 128-key tile); one
//     CTA keeps the K and V tiles in shared memory and walks every query head
//     of the group and its 64-row query tiles at and after the diagonal (all
//     of them when not causal),
//     accumulating dK and dV of the group in TMEM across the heads:
//        S^T  = K Q^T,  dP^T = V dO^T  (TMEM, double-buffered, issued while
//                                       the softmax warps work on the tile
//                                       before)
//        softmax warps (thread = key row): P^T and dS^T as bf16 into the
//                                       S^T columns just read (TMEM), dS^T
//                                       also into shared memory
//        dQ^T = K^T dS^T   (TMEM, in the dP^T buffer just consumed) -> the
//                          dQ warps stage it in shared memory and one thread
//                          adds it to the fp32 accumulator by TMA reduce-add
//        dV  += P^T dO,  dK += dS^T Q   (A operands from TMEM; 128 columns
//                                        of TMEM each)
//     then the softmax warps write dK and the dQ warps dV, as bf16;
//  4. finalize: dQ accumulators -> bf16;
//  5. (when asked) dX = dz W^T, and dW = X^T dz as per-chunk partial sums
//     reduced in a fixed order.
//
// Warp roles (320 threads): 0-3 softmax / dK epilogue, 4-7 dQ readback and
// reduce / dV epilogue, 8 TMA producer, 9 MMA issuer.
// TMEM: [0,128) dV, [128,256) dK, [256,384) S^T x 2, [384,512) dP^T / dQ^T x 2.
// Head dim d = 128 or 64 (d = 64: half of each K, V, Q, dO tile, dV and dK
// in the first 64 columns of their regions, dQ^T with 64 zero feature rows).
// SMEM: K 32 KB, V 32 KB, 3 stages of (Q 16 KB, dO 16 KB), dS^T x 2
//       (16 KB each), dQ staging 32 KB, per-stage lse2 / D (1.5 KB); every
//       bf16 operand in 128-byte-swizzled 64-column boxes.  The MMAs are
//       bound by shared-memory reads, which is why P^T and dS^T reach dV and
//       dK through TMEM.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records
// DA_ERR_TIMEOUT, raises an abort flag that the other roles see, and leaves.
//
// Grouped differential attention (the 3:1 / 4:1 signal:noise follow-up named
// in "Differential Transformer | ICLR 2025 Oral", "같은 문제, 다른 접근", read
// in the V2 form): the query heads come in groups of r signal heads and one
// noise head, out[t, p] = O[t, signal(p)] - g[t, p] O[t, noise(p)].  Its
// chain rule differs from V2's only in the preprocess: dO of signal head p is
// dOut_p itself, dO of a group's noise head is -sum_p g_p dOut_p (rounded to
// bf16 once), dz_p = -<dOut_p, O_noise> g_p (1 - g_p); the main kernel, the
// finalize and the gate-projection gradients are shared (r = 1 is V2).
#include <type_traits>

#include "kernels.h"
#include "softmax.cuh"
#include "tma.cuh"

namespace da {
namespace {

constexpr int kKT = 128;  // keys per item
constexpr int kQT = 64;   // queries per iteration
constexpr int kD = 128;   // the largest head dim: shared-memory layout and workspace sizing
constexpr int kThreads = 320;
constexpr int kStages = 3;

constexpr int kBoxK = 128 * 128;  // 64 columns x 128 rows of bf16
constexpr int kBoxQ = 64 * 128;   // 64 columns x 64 rows
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + 2 * kBoxK;
constexpr int kOffStage = kOffV + 2 * kBoxK;  // 65536
constexpr int kStageQ = 0;
constexpr int kStageDO = 2 * kBoxQ;
constexpr int kStageBytes = 4 * kBoxQ;                  // 32 KB
constexpr int kOffDS = kOffStage + kStages * kStageBytes;  // 163840: [2][128 keys][64 queries]
constexpr int kOffDQ = kOffDS + 2 * kBoxK;                // fp32 [64][128]
constexpr int kOffLse = kOffDQ + kQT * kD * 4;          // [stage] {lse2[64], D[64]}
constexpr int kOffBar = kOffLse + kStages * 512;
constexpr int kSmemBytes = kOffBar + 512 + 1024;        // 232448: the per-block limit

enum {
  B_KV = 0, B_QFULL, B_QEMPTY = B_QFULL + kStages, B_SFULL = B_QEMPTY + kStages, B_PFULL = B_SFULL + 2,
  B_DQFULL = B_PFULL + 2, B_DQFREE = B_DQFULL + 2, B_DSFREE = B_DQFREE + 2, B_STG = B_DSFREE + 2, B_STGFREE, B_ACC,
  B_COUNT
};
static_assert(B_COUNT * 8 <= 256, "barrier area");

__host__ __device__ constexpr uint32_t idesc2(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kIdS = idesc2(128, 64, 0, 0);    // K (K-major) x Q (K-major); V x dO
constexpr uint32_t kIdDQ = idesc2(128, 64, 1, 1);   // K^T (MN-major) x dS^T (MN-major)
// (P^T / dS^T (TMEM) x dO / Q (MN-major) is idesc2(128, D, 0, 1) per head dim)

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
};

__device__ __forceinline__ bool wait_bar(const Shared& sh, uint32_t bar, uint32_t parity,
                                         uint32_t* status, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*sh.abort_flag()) return false;
    if (globaltimer() - t0 > 2000000000ull) {
      record_status(status, DA_ERR_TIMEOUT, site);
      *sh.abort_flag() = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// --------------------------------------------------------------------------
// Workspace carve-up (all offsets 256-byte aligned).  Every region is always
// reserved so that the size depends only on (B, N, h, d_model).
constexpr int kDwChunk = 1024;  // tokens per dW partial sum

struct BwdWs {
  __nv_bfloat16* dodd;  // [B, N, h, d]  dO of the odd heads = -g G (room for d = 128);
                        // grouped: dO of the noise heads [B, N, 2h / (r + 1), d]
  float* lse2;          // [B, 2h, Npad]   LSE * log2 e; +inf in padding rows
  float* D;             // [B, 2h, Npad]
  float* dq;            // [B, N, 2h, d] fp32 accumulators (room for d = 128)
  float* gate;          // [B, N, h_out]  when computed here
  float* dz;            // [B, N, h_out]  when the caller keeps none
  float* dw_part;       // [chunks, d_model, h_out]
  int npad, chunks;
};

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

// h: half the query heads (V2: the pairs); h_out: the output heads (V2: h)
BwdWs carve(void* base, int B, int N, int h, int h_out, int d_model, size_t* total) {
  BwdWs w;
  w.npad = (N + kQT - 1) / kQT * kQT;
  const long long T = static_cast<long long>(B) * N;
  w.chunks = static_cast<int>((T + kDwChunk - 1) / kDwChunk);
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* r = p ? p + off : nullptr;
    off += a256(bytes);
    return r;
  };
  const size_t tok = static_cast<size_t>(T);
  const size_t srow = static_cast<size_t>(B) * 2 * h * w.npad;
  w.dodd = reinterpret_cast<__nv_bfloat16*>(take(tok * h * kD * 2));
  w.lse2 = reinterpret_cast<float*>(take(srow * 4));
  w.D = reinterpret_cast<float*>(take(srow * 4));
  w.dq = reinterpret_cast<float*>(take(tok * 2 * h * kD * 4));
  w.gate = reinterpret_cast<float*>(take(tok * h_out * 4));
  w.dz = reinterpret_cast<float*>(take(tok * h_out * 4));
  w.dw_part = reinterpret_cast<float*>(
      take(d_model > 0 ? static_cast<size_t>(w.chunks) * d_model * h_out * 4 : 0));
  if (total) *total = off;
  return w;
}

// ------------------------------------------------------------ preprocess --
constexpr int kPreWarps = 8;

// kF consecutive bf16 / fp32 values of one lane (kF = 4 or 2)
template <int kF>
__device__ __forceinline__ void ld_bf16(const __nv_bfloat16* p, __nv_bfloat16 (&v)[kF]) {
  if constexpr (kF == 4) {
    *reinterpret_cast<uint2*>(v) = *reinterpret_cast<const uint2*>(p);
  } else {
    *reinterpret_cast<uint32_t*>(v) = *reinterpret_cast<const uint32_t*>(p);
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
// The grouped preprocess zeroes the dQ accumulators of a (token, group) -
// (r + 1) contiguous rows - with bulk copies (the TMA unit writes them, not
// the load/store path the kernel's reads use): each block keeps a zeroed
// buffer of kZeroBytes in shared memory, and each warp copies it over its
// rows.  (For the two rows of a V2 pair the per-lane stores measured faster:
// 205 against 228 us at B2 N8192 with 64 query heads.)
constexpr int kZeroBytes = 4096;
__device__ __forceinline__ void zero_init(float* zbuf) {
  for (int i = threadIdx.x; i < kZeroBytes / 16; i += blockDim.x)
    reinterpret_cast<float4*>(zbuf)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  fence_proxy_async_smem();
  __syncthreads();
}
// `bytes` (a multiple of 16) of zeros at dst (16-byte aligned), one lane
__device__ __forceinline__ void bulk_zero(float* dst, const float* zbuf, uint32_t bytes) {
  for (uint32_t off = 0; off < bytes; off += kZeroBytes) {
    const uint32_t n = min(bytes - off, static_cast<uint32_t>(kZeroBytes));
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint8_t*>(dst) + off),
                 "r"(smem_u32(zbuf)), "r"(n)
                 : "memory");
  }
  bulk_commit();
}

// one warp per (token, pair); lane = D / 32 consecutive features
template <int D>
__global__ void __launch_bounds__(kPreWarps * 32)
v2_bwd_pre_kernel(V2BwdArgs a, BwdWs w, const float* __restrict__ gate, float* __restrict__ dz) {
  constexpr int kF = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kPreWarps + warp;  // (b, p, n < npad)
  const long long total = static_cast<long long>(a.B) * a.h * w.npad;
  if (row >= total) return;
  const int n = static_cast<int>(row % w.npad);
  const int bp = static_cast<int>(row / w.npad);
  const int b = bp / a.h, p = bp % a.h;
  const int he = 2 * p;
  const int64_t se = (static_cast<int64_t>(b) * 2 * a.h + he) * w.npad + n;  // padded rows
  const int64_t so = se + w.npad;
  if (n >= a.N) {
    if (lane == 0) {
      w.lse2[se] = INFINITY;
      w.lse2[so] = INFINITY;
      w.D[se] = 0.f;
      w.D[so] = 0.f;
    }
    return;
  }
  const __nv_bfloat16* gp = static_cast<const __nv_bfloat16*>(a.dout.ptr) + b * a.dout.sb +
                            static_cast<int64_t>(n) * a.dout.sn + p * a.dout.sh + lane * kF;
  const __nv_bfloat16* op = static_cast<const __nv_bfloat16*>(a.o_heads.ptr) + b * a.o_heads.sb +
                            static_cast<int64_t>(n) * a.o_heads.sn + he * a.o_heads.sh + lane * kF;
  __nv_bfloat16 ge[kF], ee[kF], oe[kF];
  ld_bf16<kF>(gp, ge);
  ld_bf16<kF>(op, ee);
  ld_bf16<kF>(op + a.o_heads.sh, oe);
  const int64_t tp = (static_cast<int64_t>(b) * a.N + n) * a.h + p;
  const float g = gate[tp];
  float de = 0.f, dd = 0.f, go = 0.f;
  uint32_t pk[kF / 2];
#pragma unroll
  for (int e = 0; e < kF; e += 2) {
    const float g0 = __bfloat162float(ge[e]), g1 = __bfloat162float(ge[e + 1]);
    // the odd head's dO is an MMA operand: round it once, and take D from
    // the rounded values the MMAs see
    pk[e / 2] = pack_bf16x2(-g * g0, -g * g1);
    const __nv_bfloat162 r = *reinterpret_cast<const __nv_bfloat162*>(&pk[e / 2]);
    const float o0 = __bfloat162float(oe[e]), o1 = __bfloat162float(oe[e + 1]);
    de = fmaf(g0, __bfloat162float(ee[e]), de);
    de = fmaf(g1, __bfloat162float(ee[e + 1]), de);
    dd = fmaf(__low2float(r), o0, dd);
    dd = fmaf(__high2float(r), o1, dd);
    go = fmaf(g0, o0, go);
    go = fmaf(g1, o1, go);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    de += __shfl_xor_sync(0xffffffffu, de, o);
    dd += __shfl_xor_sync(0xffffffffu, dd, o);
    go += __shfl_xor_sync(0xffffffffu, go, o);
  }
  if constexpr (kF == 4) {
    *reinterpret_cast<uint2*>(w.dodd + tp * D + lane * kF) = make_uint2(pk[0], pk[1]);
  } else {
    *reinterpret_cast<uint32_t*>(w.dodd + tp * D + lane * kF) = pk[0];
  }
  const int64_t qrow = (static_cast<int64_t>(b) * a.N + n) * 2 * a.h + he;
  st_zero_f32<kF>(w.dq + qrow * D + lane * kF);
  st_zero_f32<kF>(w.dq + (qrow + 1) * D + lane * kF);
  if (lane == 0) {
    const int64_t le = (static_cast<int64_t>(b) * 2 * a.h + he) * a.N + n;
    w.lse2[se] = a.lse[le] * 1.4426950408889634f;
    w.lse2[so] = a.lse[le + a.N] * 1.4426950408889634f;
    w.D[se] = de;
    w.D[so] = dd;
    dz[tp] = -go * g * (1.f - g);
  }
}

// Grouped: one warp per (token, group of r signal heads + 1 noise head);
// lane = D / 32 consecutive features.  Signal head i of group gi is query head
// gi (r+1) + i and output head p = gi r + i; its dO is dOut_p (read by the main
// kernel directly), D = <dOut_p, O_i>, dz_p = -<dOut_p, O_noise> g_p (1 - g_p).
// The noise head's dO = -sum_i g_p dOut_p is accumulated in fp32, rounded to
// bf16 once (an MMA operand), and its D taken from the rounded values.
template <int D>
__global__ void __launch_bounds__(kPreWarps * 32)
grouped_bwd_pre_kernel(V2BwdArgs a, BwdWs w, const float* __restrict__ gate, float* __restrict__ dz) {
  constexpr int kF = D / 32;
  __shared__ __align__(128) float zbuf[kZeroBytes / 4];
  zero_init(zbuf);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = a.ratio;
  const int n_groups = 2 * a.h / (r + 1);
  const long long row = static_cast<long long>(blockIdx.x) * kPreWarps + warp;  // (b, group, n < npad)
  const long long total = static_cast<long long>(a.B) * n_groups * w.npad;
  if (row >= total) return;
  const int n = static_cast<int>(row % w.npad);
  const int bg = static_cast<int>(row / w.npad);
  const int b = bg / n_groups, gi = bg % n_groups;
  const int hq0 = gi * (r + 1), noise = hq0 + r;
  auto srow = [&](int j) { return (static_cast<int64_t>(b) * 2 * a.h + j) * w.npad + n; };
  if (n >= a.N) {
    if (lane == 0)
      for (int j = hq0; j <= noise; ++j) {
        w.lse2[srow(j)] = INFINITY;
        w.D[srow(j)] = 0.f;
      }
    return;
  }
  const __nv_bfloat16* ob = static_cast<const __nv_bfloat16*>(a.o_heads.ptr) + b * a.o_heads.sb +
                            static_cast<int64_t>(n) * a.o_heads.sn + lane * kF;
  __nv_bfloat16 ne[kF];
  ld_bf16<kF>(ob + noise * a.o_heads.sh, ne);
  float on[kF], dn[kF];
#pragma unroll
  for (int e = 0; e < kF; ++e) {
    on[e] = __bfloat162float(ne[e]);
    dn[e] = 0.f;
  }
  const int64_t tok = static_cast<int64_t>(b) * a.N + n;
  const int64_t qrow0 = tok * 2 * a.h;
  if (lane == 0) bulk_zero(w.dq + (qrow0 + hq0) * D, zbuf, (r + 1) * D * 4);  // the group's dQ rows
  for (int i = 0; i < r; ++i) {
    const int p = gi * r + i;
    const __nv_bfloat16* gp = static_cast<const __nv_bfloat16*>(a.dout.ptr) + b * a.dout.sb +
                              static_cast<int64_t>(n) * a.dout.sn + p * a.dout.sh + lane * kF;
    __nv_bfloat16 ge[kF], se[kF];
    ld_bf16<kF>(gp, ge);
    ld_bf16<kF>(ob + (hq0 + i) * a.o_heads.sh, se);
    const float g = gate[tok * a.h_out + p];
    float ds = 0.f, gn = 0.f;
#pragma unroll
    for (int e = 0; e < kF; ++e) {
      const float gv = __bfloat162float(ge[e]);
      ds = fmaf(gv, __bfloat162float(se[e]), ds);
      gn = fmaf(gv, on[e], gn);
      dn[e] = fmaf(-g, gv, dn[e]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ds += __shfl_xor_sync(0xffffffffu, ds, o);
      gn += __shfl_xor_sync(0xffffffffu, gn, o);
    }
    if (lane == 0) {
      const int64_t le = (static_cast<int64_t>(b) * 2 * a.h + hq0 + i) * a.N + n;
      w.lse2[srow(hq0 + i)] = a.lse[le] * 1.4426950408889634f;
      w.D[srow(hq0 + i)] = ds;
      dz[tok * a.h_out + p] = -gn * g * (1.f - g);
    }
  }
  uint32_t pk[kF / 2];
  float dd = 0.f;
#pragma unroll
  for (int e = 0; e < kF; e += 2) {
    pk[e / 2] = pack_bf16x2(dn[e], dn[e + 1]);
    const __nv_bfloat162 rr = *reinterpret_cast<const __nv_bfloat162*>(&pk[e / 2]);
    dd = fmaf(__low2float(rr), on[e], dd);
    dd = fmaf(__high2float(rr), on[e + 1], dd);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
  __nv_bfloat16* dst = w.dodd + (tok * n_groups + gi) * D + lane * kF;
  if constexpr (kF == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pk[0];
  }
  if (lane == 0) {
    bulk_wait_read();
    const int64_t le = (static_cast<int64_t>(b) * 2 * a.h + noise) * a.N + n;
    w.lse2[srow(noise)] = a.lse[le] * 1.4426950408889634f;
    w.D[srow(noise)] = dd;
  }
}

// -------------------------------------------------------------- main -------
struct Item {
  int b, g, kt, i0, n_ith, n_it;
};

// Items: (batch, K/V group, key tile), one per CTA, in launch order the
// heaviest key tiles (most query tiles) of every (batch, K/V group) unit
// first.  (Taking the units a block at a time, so that fewer dQ accumulators
// are live in L2, left the last block's heavy items to start late: at B2
// N8192 with 16 units in blocks of 5, 5, 5 and 1 the SMs were 82 % busy and
// the kernel 18 % slower.)
__device__ __forceinline__ Item item_of(int i, int n_qt, int units, int h_kv, int G, bool causal) {
  Item it;
  it.kt = i / units;
  const int u = i % units;
  it.b = u / h_kv;
  it.g = u % h_kv;
  it.i0 = causal ? it.kt * (kKT / kQT) : 0;  // causal: query tiles from the diagonal on
  it.n_ith = n_qt - it.i0;
  it.n_it = it.n_ith * G;
  return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
v2_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                   const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dq,
                   V2BwdArgs a, BwdWs w) {
  extern __shared__ uint8_t smem_raw[];
  Shared sh;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t al = (raw + 1023u) & ~1023u;
    sh.base = al;
    sh.gen = smem_raw + (al - raw);
  }
  constexpr int kNB = D / 64;  // 64-column boxes per tile row
  constexpr uint32_t kIdAcc = idesc2(128, D, 0, 1);  // P^T / dS^T (TMEM) x dO / Q (MN-major)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (2 * a.h) / a.h_kv;
  const int n_qt = w.npad / kQT;
  const bool causal = a.causal != 0;
  const int ratio = a.ratio > 1 ? a.ratio : 1;
  const Item it = item_of(blockIdx.x, n_qt, a.B * a.h_kv, a.h_kv, G, causal);

  if (threadIdx.x == 0) {
    mbar_init(sh.bar(B_KV), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(sh.bar(B_QFULL + s), 1);
      mbar_init(sh.bar(B_QEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sh.bar(B_SFULL + b), 1);
      mbar_init(sh.bar(B_DQFULL + b), 1);
      mbar_init(sh.bar(B_DQFREE + b), 128);
      mbar_init(sh.bar(B_DSFREE + b), 1);
      mbar_init(sh.bar(B_PFULL + b), 128);
    }
    mbar_init(sh.bar(B_STG), 128);
    mbar_init(sh.bar(B_STGFREE), 1);
    mbar_init(sh.bar(B_ACC), 1);
    *sh.abort_flag() = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(sh.tmem_slot()), 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_g);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_dq);
  }
  if (D < 128 && warp < 4) {
    // dQ^T = K^T dS^T runs with M = 128 feature rows: with head dim 64 the
    // second 64-column box of the K tile is never loaded, so zero it once
    // (feature rows 64-127 of dQ^T come out zero and are not stored)
    uint4* zk = reinterpret_cast<uint4*>(sh.gen + kOffK + kBoxK);
    for (int i = threadIdx.x; i < kBoxK / 16; i += 128) zk[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot();
  const uint32_t T_DV = tmem, T_DK = tmem + 128;
  auto t_s = [&](int b) { return tmem + 256 + b * 64; };
  auto t_d = [&](int b) { return tmem + 384 + b * 64; };
  // iteration k -> (query head within the group, first query row)
  auto head_of = [&](int k) { return k / it.n_ith; };
  auto q0_of = [&](int k) { return (it.i0 + k % it.n_ith) * kQT; };

  if (warp == 8) {
    // ---------------------------------------------------- TMA producer ----
    if (lane == 0) {
      mbar_arrive_expect_tx(sh.bar(B_KV), 2 * kNB * kBoxK);
      for (int box = 0; box < kNB; ++box)
        tma_load_4d(sh.base + kOffK + box * kBoxK, &tm_k, sh.bar(B_KV), box * 64, it.g, it.kt * kKT, it.b);
      for (int box = 0; box < kNB; ++box)
        tma_load_4d(sh.base + kOffV + box * kBoxK, &tm_v, sh.bar(B_KV), box * 64, it.g, it.kt * kKT, it.b);
      int last = -1;
      bool ok = true;
      for (int k = 0; k < it.n_it; ++k) {
        const int st = k % kStages, use = k / kStages;
        if (use > 0 && !wait_bar(sh, sh.bar(B_QEMPTY + st), (use - 1) & 1, a.status, 0x6001)) {
          ok = false;
          break;
        }
        const int qh = it.g * G + head_of(k);
        const int q0 = q0_of(k);
        const uint32_t sb = sh.base + kOffStage + st * kStageBytes;
        const uint32_t bar = sh.bar(B_QFULL + st);
        mbar_arrive_expect_tx(bar, 2 * kNB * kBoxQ + 512);
        for (int box = 0; box < kNB; ++box)
          tma_load_4d(sb + kStageQ + box * kBoxQ, &tm_q, bar, box * 64, qh, q0, it.b);
        // dO of a signal head (V2: an even head) is dOut itself, at output
        // head grp r + i; of a noise head (V2: odd), the workspace's
        // -sum g dOut, at index grp
        const int grp = qh / (ratio + 1), gsub = qh - grp * (ratio + 1);
        const bool signal = gsub < ratio;
        const CUtensorMap* tdo = signal ? &tm_g : &tm_do;
        const int dsel = signal ? grp * ratio + gsub : grp;
        for (int box = 0; box < kNB; ++box)
          tma_load_4d(sb + kStageDO + box * kBoxQ, tdo, bar, box * 64, dsel, q0, it.b);
        const size_t srow = (static_cast<size_t>(it.b) * 2 * a.h + qh) * w.npad + q0;
        const uint32_t lb = sh.base + kOffLse + st * 512;
        bulk_load(lb, w.lse2 + srow, 256, bar);
        bulk_load(lb + 256, w.D + srow, 256, bar);
        last = k;
      }
      if (!ok) {
        // give the loads already issued (bounded) time to land before exit
        const uint64_t t0 = globaltimer();
        if (!mbar_try_wait(sh.bar(B_KV), 0))
          while (globaltimer() - t0 < 200000000ull && !mbar_try_wait(sh.bar(B_KV), 0)) {
          }
        for (int k = last; k >= 0 && k > last - kStages; --k) {
          const uint32_t bar = sh.bar(B_QFULL + k % kStages);
          const uint32_t par = (k / kStages) & 1;
          while (globaltimer() - t0 < 400000000ull && !mbar_try_wait(bar, par)) {
          }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0) {
      bool ok = wait_bar(sh, sh.bar(B_KV), 0, a.status, 0x6101);
      tc_fence_after();
      const uint32_t kA = sh.base + kOffK, vA = sh.base + kOffV;
      auto dsA = [&](int b) { return sh.base + kOffDS + b * kBoxK; };
      auto stage = [&](int k) { return sh.base + kOffStage + (k % kStages) * kStageBytes; };
      auto issue_sdp = [&](int k) {  // S^T = K Q^T and dP^T = V dO^T into buffers k & 1
        const uint32_t qb = stage(k) + kStageQ, db = stage(k) + kStageDO;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = (kk >> 2) * kBoxK + (kk & 3) * 32;
          const uint32_t offb = (kk >> 2) * kBoxQ + (kk & 3) * 32;
          tc_mma_ss(t_s(k & 1), sdesc_sw128(kA + offa, 16, 1024), sdesc_sw128(qb + offb, 16, 1024), kIdS,
                    kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = (kk >> 2) * kBoxK + (kk & 3) * 32;
          const uint32_t offb = (kk >> 2) * kBoxQ + (kk & 3) * 32;
          tc_mma_ss(t_d(k & 1), sdesc_sw128(vA + offa, 16, 1024), sdesc_sw128(db + offb, 16, 1024), kIdS,
                    kk > 0);
        }
        tc_commit(sh.bar(B_SFULL + (k & 1)));
      };
      if (ok && it.n_it > 0) {
        if (wait_bar(sh, sh.bar(B_QFULL), 0, a.status, 0x6102)) {
          tc_fence_after();
          issue_sdp(0);
        } else {
          ok = false;
        }
      }
      for (int k = 0; k < it.n_it && ok; ++k) {
        const int b = k & 1;
        if (k + 1 < it.n_it) {
          // S / dP of the next tile run while the softmax warps work on this one
          const int k1 = k + 1;
          if (!wait_bar(sh, sh.bar(B_QFULL + k1 % kStages), (k1 / kStages) & 1, a.status, 0x6103)) {
            ok = false;
            break;
          }
          // its dP^T buffer held dQ^T(k - 1): wait until the dQ warps read it
          if (k >= 1 && !wait_bar(sh, sh.bar(B_DQFREE + (k1 & 1)), ((k - 1) >> 1) & 1, a.status, 0x6104)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_sdp(k1);
        }
        if (!wait_bar(sh, sh.bar(B_PFULL + b), (k >> 1) & 1, a.status, 0x6105)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dQ^T = K^T dS^T  (into the dP^T buffer of this tile, already read)
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk)
          tc_mma_ss(t_d(b), sdesc_sw128(kA + kk * 2048, kBoxK, 1024), sdesc_sw128(dsA(b) + kk * 2048, kBoxQ, 1024),
                    kIdDQ, kk > 0);
        tc_commit(sh.bar(B_DQFULL + b));
        tc_commit(sh.bar(B_DSFREE + b));
        // dV += P^T dO ; dK += dS^T Q  (P^T in columns 0-31 of the S^T
        // buffer, dS^T in columns 32-63)
        const uint32_t db = stage(k) + kStageDO, qb = stage(k) + kStageQ;
#pragma unroll
        for (int kk = 0; kk < kQT / 16; ++kk)
          tc_mma_ts(T_DV, t_s(b) + kk * 8, sdesc_sw128(db + kk * 2048, kBoxQ, 1024), kIdAcc,
                    (k > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kQT / 16; ++kk)
          tc_mma_ts(T_DK, t_s(b) + 32 + kk * 8, sdesc_sw128(qb + kk * 2048, kBoxQ, 1024), kIdAcc,
                    (k > 0 || kk > 0) ? 1u : 0u);
        tc_commit(sh.bar(B_QEMPTY + k % kStages));
      }
      if (ok) tc_commit(sh.bar(B_ACC));
    }
  } else if (warp < 4) {
    // ------------------------------------------ softmax / dS, dK epilogue --
    const int r = warp * 32 + lane;  // key row within the tile = TMEM lane
    const uint32_t loff = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;
    const uint64_t sl2x2 = f2(sl2, sl2), sc2 = f2(a.scale, a.scale);
    const int key = it.kt * kKT + r;
    bool ok = true;
    for (int k = 0; k < it.n_it && ok; ++k) {
      const int b = k & 1;
      const int q0 = q0_of(k);
      if (!wait_bar(sh, sh.bar(B_SFULL + b), (k >> 1) & 1, a.status, 0x6201)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4* l2v = reinterpret_cast<const float4*>(sh.gen + kOffLse + (k % kStages) * 512);
      const float4* ddv = l2v + 16;
      // causal: a query of this tile may precede a key.  (Not causal: keys
      // past N are zero rows of K and V, which give dQ no contribution, and
      // their dK / dV rows are never stored.)
      const bool diag = causal && q0 < it.kt * kKT + kKT;
      uint8_t* dsbuf = sh.gen + kOffDS + b * kBoxK;
      uint32_t dkeep[16];  // dS^T of the first half, stored to TMEM once the second half's S^T is read
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sv[32], dp[32];
        tmem_ld32(t_s(b) + loff + hf * 32, sv);
        tmem_ld32(t_d(b) + loff + hf * 32, dp);
        tmem_ld_wait();
        uint32_t pw[16], dw[16];
        auto half = [&](auto masked) {
          constexpr bool kMask = decltype(masked)::value;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {  // 4 queries at a time
            const float4 lq = l2v[hf * 8 + q4];
            const float4 dq4 = ddv[hf * 8 + q4];
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
            const uint64_t t01 = add_f32x2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), f2(-dq4.x, -dq4.y));
            const uint64_t t23 =
                add_f32x2(f2(__uint_as_float(dp[c + 2]), __uint_as_float(dp[c + 3])), f2(-dq4.z, -dq4.w));
            const uint64_t d01 = mul_f32x2(mul_f32x2(t01, f2(p0, p1)), sc2);
            const uint64_t d23 = mul_f32x2(mul_f32x2(t23, f2(p2, p3)), sc2);
            pw[q4 * 2] = pack_bf16x2(p0, p1);
            pw[q4 * 2 + 1] = pack_bf16x2(p2, p3);
            dw[q4 * 2] = pack_bf16x2(f2_lo(d01), f2_hi(d01));
            dw[q4 * 2 + 1] = pack_bf16x2(f2_lo(d23), f2_hi(d23));
          }
        };
        if (diag) half(std::true_type{});
        else half(std::false_type{});
        // P^T over S^T columns this thread has already read
        tmem_st16(t_s(b) + loff + hf * 16, pw);
        // the dS^T buffer is free once dQ of the tile two back has read it
        if (hf == 0 && k > 1 && !wait_bar(sh, sh.bar(B_DSFREE + b), ((k >> 1) - 1) & 1, a.status, 0x6202)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int ch = hf * 4 + cc;
          const int off = r * 128 + ((ch ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dsbuf + off) = make_uint4(dw[cc * 4], dw[cc * 4 + 1], dw[cc * 4 + 2], dw[cc * 4 + 3]);
        }
        if (hf == 0) {
#pragma unroll
          for (int e = 0; e < 16; ++e) dkeep[e] = dw[e];
        } else {
          tmem_st16(t_s(b) + loff + 32, dkeep);
          tmem_st16(t_s(b) + loff + 48, dw);
        }
      }
      if (!ok) break;
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      // one barrier per S^T buffer: this warpgroup can run two tiles ahead
      // of the MMA issuer's wait, never two uses of one buffer
      mbar_arrive(sh.bar(B_PFULL + b));
    }
    // ------------------------------------------------------- dK epilogue --
    if (ok && wait_bar(sh, sh.bar(B_ACC), 0, a.status, 0x6203)) {
      tc_fence_after();
      // the TMEM loads are warp-collective: every lane loads, live rows store
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dk.ptr) + it.b * a.dk.sb +
                           static_cast<int64_t>(key) * a.dk.sn + it.g * a.dk.sh;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(T_DK + loff + c * 32, v);
        tmem_ld_wait();
        if (key < a.N) {
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            *reinterpret_cast<uint4*>(dst + c * 32 + e) = make_uint4(
                pack_bf16x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                pack_bf16x2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])),
                pack_bf16x2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5])),
                pack_bf16x2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7])));
        }
      }
    }
  } else {
    // ------------------------------------- dQ readback + reduce, dV epilogue
    const int q4w = warp & 3;
    const int r = q4w * 32 + lane;  // feature of dQ^T = TMEM lane; key row in the epilogue
    const uint32_t loff = static_cast<uint32_t>(q4w * 32) << 16;
    float* stage_dq = reinterpret_cast<float*>(sh.gen + kOffDQ);
    bool ok = true;
    for (int k = 0; k < it.n_it && ok; ++k) {
      const int b = k & 1;
      if (!wait_bar(sh, sh.bar(B_DQFULL + b), (k >> 1) & 1, a.status, 0x6301)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t qv[64];
      tmem_ld32(t_d(b) + loff, *reinterpret_cast<uint32_t(*)[32]>(&qv[0]));
      tmem_ld32(t_d(b) + loff + 32, *reinterpret_cast<uint32_t(*)[32]>(&qv[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(sh.bar(B_DQFREE + b));
      // the staging buffer is free once the previous reduce has read it
      if (k > 0 && !wait_bar(sh, sh.bar(B_STGFREE), (k - 1) & 1, a.status, 0x6302)) {
        ok = false;
        break;
      }
      // [64 queries][D] fp32; feature rows past D (zero) are not staged
      if (r < D) {
#pragma unroll
        for (int c = 0; c < kQT; ++c) stage_dq[c * D + r] = __uint_as_float(qv[c]);
      }
      fence_proxy_async_smem();
      mbar_arrive(sh.bar(B_STG));
      bool stg_ok = true;
      if (r == 0) {
        stg_ok = wait_bar(sh, sh.bar(B_STG), k & 1, a.status, 0x6303);
        if (stg_ok) {
          // add the [64 queries][D] tile to the fp32 accumulator (rows
          // past N are dropped by the unit)
          tma_reduce_add_4d(&tm_dq, sh.base + kOffDQ, 0, it.g * G + head_of(k), q0_of(k), it.b);
          bulk_commit();
          bulk_wait_read();
          mbar_arrive(sh.bar(B_STGFREE));
        }
      }
      // keep warp 4 uniform for the warp-collective TMEM loads
      if (q4w == 0) stg_ok = __shfl_sync(0xffffffffu, stg_ok, 0);
      if (!stg_ok) ok = false;
    }
    if (r == 0) bulk_wait_all();
    // ------------------------------------------------------- dV epilogue --
    if (ok && wait_bar(sh, sh.bar(B_ACC), 0, a.status, 0x6304)) {
      tc_fence_after();
      const int key = it.kt * kKT + r;
      // the TMEM loads are warp-collective: every lane loads, live rows store
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dv.ptr) + it.b * a.dv.sb +
                           static_cast<int64_t>(key) * a.dv.sn + it.g * a.dv.sh;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(T_DV + loff + c * 32, v);
        tmem_ld_wait();
        if (key < a.N) {
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            *reinterpret_cast<uint4*>(dst + c * 32 + e) = make_uint4(
                pack_bf16x2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                pack_bf16x2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])),
                pack_bf16x2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5])),
                pack_bf16x2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7])));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

// -------------------------------------------------------------- finalize --
template <int D>
__global__ void __launch_bounds__(256)
v2_bwd_finalize_kernel(V2BwdArgs a, BwdWs w) {
  const int H2 = 2 * a.h;
  const long long rows = static_cast<long long>(a.B) * a.N * H2;
  const long long total = rows * (D / 8);
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = idx / (D / 8);
    const int c8 = static_cast<int>(idx % (D / 8)) * 8;
    const int hq = static_cast<int>(row % H2);
    const long long bn = row / H2;
    const int n = static_cast<int>(bn % a.N), b = static_cast<int>(bn / a.N);
    const float* src = w.dq + row * D + c8;
    const float4 x0 = *reinterpret_cast<const float4*>(src);
    const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq.ptr) + b * a.dq.sb +
                         static_cast<int64_t>(n) * a.dq.sn + hq * a.dq.sh + c8;
    *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w),
                                                pack_bf16x2(x1.x, x1.y), pack_bf16x2(x1.z, x1.w));
  }
}

// ------------------------------------------------- gate-projection grads --
// Both are 2 T d_model h FLOP on the FMA pipes with register tiles fed from
// shared memory (fp32 throughout, as exact as the gate itself):
//   dX[t, c] = sum_p dz[t, p] W[c, p]
//   dW[c, p] = sum_t X[t, c] dz[t, p]   (per-chunk partial sums, then a
//                                        fixed-order reduction)
constexpr int kGT = 64;    // tokens per staged tile
constexpr int kGC = 128;   // d_model columns per block
constexpr int kGP = 32;    // gate heads per block (dW) / per pass (dX)

// dX: block = 64 tokens x 128 columns, 256 threads; thread = 8 tokens x 4
// consecutive columns (32 accumulators).  W^T slice [p][128 columns] and the
// dz tile [64 tokens][p] in shared memory; p in passes of 32.
__global__ void __launch_bounds__(256)
v2_bwd_dx_kernel(int T, int d_model, int h, const float* __restrict__ dz,
                 const __nv_bfloat16* __restrict__ W, __nv_bfloat16* __restrict__ dx) {
  __shared__ float s_w[kGP][kGC];
  __shared__ float s_z[kGT][kGP + 1];
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int t0 = blockIdx.x * kGT, c0 = blockIdx.y * kGC;
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  for (int p0 = 0; p0 < h; p0 += kGP) {
    __syncthreads();
    for (int i = tid; i < kGP * kGC; i += 256) {
      // consecutive threads take consecutive columns: conflict-free stores of
      // the transposed slice (the 8 KB of W rows they read stay in L1)
      const int p = i / kGC, c = i % kGC;
      s_w[p][c] = (c0 + c < d_model && p0 + p < h) ? __bfloat162float(W[static_cast<int64_t>(c0 + c) * h + p0 + p])
                                                   : 0.f;
    }
    for (int i = tid; i < kGT * kGP; i += 256) {
      const int t = i / kGP, p = i % kGP;
      s_z[t][p] = (t0 + t < T && p0 + p < h) ? dz[static_cast<int64_t>(t0 + t) * h + p0 + p] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int p = 0; p < kGP; ++p) {
      const float4 w4 = *reinterpret_cast<const float4*>(&s_w[p][tx * 4]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float z = s_z[ty * 8 + i][p];
        acc[i][0] = fmaf(z, w4.x, acc[i][0]);
        acc[i][1] = fmaf(z, w4.y, acc[i][1]);
        acc[i][2] = fmaf(z, w4.z, acc[i][2]);
        acc[i][3] = fmaf(z, w4.w, acc[i][3]);
      }
    }
  }
  const int c = c0 + tx * 4;
  if (c >= d_model) return;  // d_model is a multiple of 64: all four columns or none
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t < T)
      *reinterpret_cast<uint2*>(dx + static_cast<int64_t>(t) * d_model + c) =
          make_uint2(pack_bf16x2(acc[i][0], acc[i][1]), pack_bf16x2(acc[i][2], acc[i][3]));
  }
}

// dW partials: block = 128 columns x 32 gate heads over one chunk of
// kDwChunk tokens, 256 threads; thread = 4 consecutive columns x 4 heads.
// X and dz staged 64 tokens at a time.
__global__ void __launch_bounds__(256)
v2_bwd_dw_partial_kernel(int T, int d_model, int h, const float* __restrict__ dz,
                         const __nv_bfloat16* __restrict__ X, float* __restrict__ part) {
  __shared__ __align__(16) __nv_bfloat16 s_x[kGT][kGC];
  __shared__ __align__(16) float s_z[kGT][kGP];
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int c0 = blockIdx.x * kGC, chunk = blockIdx.y, p0 = blockIdx.z * kGP;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const int tbeg = chunk * kDwChunk, tend = min(T, tbeg + kDwChunk);
  for (int ts = tbeg; ts < tend; ts += kGT) {
    __syncthreads();
    // X tile: 64 tokens x 128 columns, 16-byte loads (d_model % 64 == 0)
    for (int i = tid; i < kGT * (kGC / 8); i += 256) {
      const int t = i / (kGC / 8), c8 = (i % (kGC / 8)) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (ts + t < tend && c0 + c8 < d_model)
        v = *reinterpret_cast<const uint4*>(X + static_cast<int64_t>(ts + t) * d_model + c0 + c8);
      *reinterpret_cast<uint4*>(&s_x[t][c8]) = v;
    }
    for (int i = tid; i < kGT * kGP; i += 256) {
      const int t = i / kGP, p = i % kGP;
      s_z[t][p] = (ts + t < tend && p0 + p < h) ? dz[static_cast<int64_t>(ts + t) * h + p0 + p] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int t = 0; t < kGT; ++t) {
      const uint2 xr = *reinterpret_cast<const uint2*>(&s_x[t][tx * 4]);
      const float4 z4 = *reinterpret_cast<const float4*>(&s_z[t][ty * 4]);
      const __nv_bfloat162 x01 = *reinterpret_cast<const __nv_bfloat162*>(&xr.x);
      const __nv_bfloat162 x23 = *reinterpret_cast<const __nv_bfloat162*>(&xr.y);
      const float xv[4] = {__low2float(x01), __high2float(x01), __low2float(x23), __high2float(x23)};
      const float zv[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], zv[j], acc[i][j]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = c0 + tx * 4 + i;
    if (c >= d_model) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int p = p0 + ty * 4 + j;
      if (p < h) part[(static_cast<int64_t>(chunk) * d_model + c) * h + p] = acc[i][j];
    }
  }
}

__global__ void __launch_bounds__(256)
v2_bwd_dw_reduce_kernel(int d_model, int h, int chunks, const float* __restrict__ part,
                        float* __restrict__ dw) {
  const int64_t n = static_cast<int64_t>(d_model) * h;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int c = 0; c < chunks; ++c) s += part[c * n + i];
    dw[i] = s;
  }
}

cudaError_t launch_dx(int T, int d_model, int h, const float* dz, const void* W, void* dx, uint32_t* status,
                      cudaStream_t s) {
  // tensor cores (gate_grads.cu) where the shape allows; CUDA cores otherwise
  if (gate_dx_tc_ok(T, d_model, h)) return launch_gate_dx_tc(T, d_model, h, dz, W, dx, status, s);
  const dim3 grid((T + kGT - 1) / kGT, (d_model + kGC - 1) / kGC);
  v2_bwd_dx_kernel<<<grid, 256, 0, s>>>(T, d_model, h, dz, static_cast<const __nv_bfloat16*>(W),
                                        static_cast<__nv_bfloat16*>(dx));
  return cudaGetLastError();
}

// the attention part: preprocess, main, finalize for head dim D
template <int D>
cudaError_t launch_attn(const V2BwdArgs& a, const BwdWs& w, float* dz, cudaStream_t s) {
  const long long T = static_cast<long long>(a.B) * a.N;
  cudaError_t e;
  const int ratio = a.ratio > 1 ? a.ratio : 1;
  const int n_noise = 2 * a.h / (ratio + 1);  // V2: h odd heads
  if (ratio == 1) {
    const long long pre_rows = static_cast<long long>(a.B) * a.h * w.npad;
    v2_bwd_pre_kernel<D><<<static_cast<unsigned>((pre_rows + kPreWarps - 1) / kPreWarps), kPreWarps * 32, 0, s>>>(
        a, w, a.gate, dz);
  } else {
    const long long pre_rows = static_cast<long long>(a.B) * n_noise * w.npad;
    grouped_bwd_pre_kernel<D><<<static_cast<unsigned>((pre_rows + kPreWarps - 1) / kPreWarps), kPreWarps * 32, 0,
                                s>>>(a, w, a.gate, dz);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap tq, tk, tv, tg, tdo, tdq;
  const da_t4 dot{w.dodd, static_cast<int64_t>(a.N) * n_noise * D, static_cast<int64_t>(n_noise) * D, D};
  if (!encode_tmap_bf16_4d(&tq, a.q, a.B, a.N, 2 * a.h, D, kQT) ||
      !encode_tmap_bf16_4d(&tk, a.k, a.B, a.N, a.h_kv, D, kKT) ||
      !encode_tmap_bf16_4d(&tv, a.v, a.B, a.N, a.h_kv, D, kKT) ||
      !encode_tmap_bf16_4d(&tg, a.dout, a.B, a.N, a.h_out, D, kQT) ||
      !encode_tmap_bf16_4d(&tdo, dot, a.B, a.N, n_noise, D, kQT) ||
      !encode_tmap_f32_4d(&tdq, w.dq, a.B, a.N, 2 * a.h, D, kQT))
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(v2_bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_kt = (a.N + kKT - 1) / kKT;
  const int units = a.B * a.h_kv;
  v2_bwd_main_kernel<D><<<n_kt * units, kThreads, kSmemBytes, s>>>(tq, tk, tv, tg, tdo, tdq, a, w);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int sms = a.num_sms > 0 ? a.num_sms : 148;
  const long long work = T * 2 * a.h * (D / 8);
  int grid = static_cast<int>((work + 255) / 256);
  if (grid > 8 * sms) grid = 8 * sms;
  if (grid < 1) grid = 1;
  v2_bwd_finalize_kernel<D><<<grid, 256, 0, s>>>(a, w);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  return cudaSuccess;
}

}  // namespace

size_t v2_bwd_workspace_bytes(int B, int N, int h, int d_model) {
  size_t total = 0;
  carve(nullptr, B, N, h, h, d_model, &total);
  return total;
}

size_t grouped_bwd_workspace_bytes(int B, int N, int h_attn, int h_out, int d_model) {
  size_t total = 0;
  carve(nullptr, B, N, h_attn, h_out, d_model, &total);
  return total;
}

cudaError_t launch_v2_bwd(const V2BwdArgs& a_in, cudaStream_t s) {
  V2BwdArgs a = a_in;
  if (a.ratio < 1) a.ratio = 1;
  if (a.ratio == 1) a.h_out = a.h;
  size_t total = 0;
  const BwdWs w = carve(a.workspace, a.B, a.N, a.h, a.h_out, a.dw ? a.d_model : 0, &total);
  if (total > a.workspace_bytes) return cudaErrorInvalidValue;
  const long long T = static_cast<long long>(a.B) * a.N;
  cudaError_t e;
  if (a.gate == nullptr) {
    GateArgs ga{static_cast<int>(T), a.d_model, a.h_out, a.x, a.d_model, a.w, w.gate, a.status};
    e = launch_gate(ga, s);
    if (e != cudaSuccess) return e;
    a.gate = w.gate;
  }
  float* dz = a.dz ? a.dz : w.dz;

  e = a.d == 128 ? launch_attn<128>(a, w, dz, s) : a.d == 64 ? launch_attn<64>(a, w, dz, s)
                                                              : cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  const int sms = a.num_sms > 0 ? a.num_sms : 148;

  if (a.dx) {
    e = launch_dx(static_cast<int>(T), a.d_model, a.h_out, dz, a.w, a.dx, a.status, s);
    if (e != cudaSuccess) return e;
  }
  if (a.dw) {
    // partial sums per chunk of kDwChunk tokens: on tensor cores
    // (gate_grads.cu) where the shape allows, CUDA cores otherwise
    if (gate_dw_tc_ok(static_cast<int>(T), a.d_model, a.h_out)) {
      e = launch_gate_dw_tc(static_cast<int>(T), a.d_model, a.h_out, kDwChunk, w.chunks, dz, a.x, w.dw_part,
                            a.status, s);
    } else {
      v2_bwd_dw_partial_kernel<<<dim3((a.d_model + kGC - 1) / kGC, w.chunks, (a.h_out + kGP - 1) / kGP), 256, 0,
                                 s>>>(static_cast<int>(T), a.d_model, a.h_out, dz,
                                      static_cast<const __nv_bfloat16*>(a.x), w.dw_part);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const long long n = static_cast<long long>(a.d_model) * a.h_out;
    int g2 = static_cast<int>((n + 255) / 256);
    if (g2 > 4 * sms) g2 = 4 * sms;
    v2_bwd_dw_reduce_kernel<<<g2, 256, 0, s>>>(a.d_model, a.h_out, w.chunks, w.dw_part, a.dw);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace da
