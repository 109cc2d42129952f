// gate_grads.cu — the gate projection's gradients on tcgen05, sm_103a:
// dX = dz W^T and the partial sums of dW = X^T dz for the V2 / grouped gate
// g = sigmoid(X W) ("Differential Transformer V2" (pogovet.com) §1: the gate
// lambda = sigmoid(X W_lambda)), dz being the gradient of the gate logits
// (fp32 [T, h]), X the bf16 [T, d_model] input and W the bf16 [d_model, h]
// projection.
//
// Both contractions have one short dimension (h <= 64 gate heads) and one
// long operand (dX written, X read: 134 MB each at T 16384, d_model 4096),
// so they are bound by memory once the products run on the tensor cores.
// dX:
//   * a CTA owns 128 tokens; dz of those tokens enters the bf16 MMAs as
//     hi + lo, hi = bf16(dz), lo = bf16(dz - hi) — together about 16 bits of
//     dz's mantissa, so the products keep fp32-like accuracy (W is bf16);
//   * per 256-feature tile: D[128 tokens x 256] = hi W^T + lo W^T in TMEM
//     (two accumulators, so the next tile's MMAs run while the epilogue reads
//     this one), W rows staged by TMA (the heads past h read as zero);
//   * the epilogue turns D into bf16 in a 128-byte-swizzled staging tile and
//     one thread stores it with TMA (whole 128-byte row pieces per box row).
// Warps: 0 TMA producer, 1 MMA issuer and TMEM allocation, 2-5 epilogue
// (thread = token row = TMEM lane).
// dW: a CTA owns 128 features and one chunk of tokens (its partial sum is
// added to the others' in a fixed order by v2_bwd_dw_reduce_kernel):
//   * per 64-token stage, X [64 tokens x 128 features] by TMA (A operand,
//     features contiguous: MN-major) and dz of those tokens as hi + lo bf16,
//     written by four warps (B operand, heads contiguous: MN-major, the heads
//     past h zero);
//   * D[128 features x 64 heads] += X^T hi + X^T lo in TMEM; three stages of
//     32 KB, two CTAs per SM.
// Warps: 0 TMA producer, 1 MMA issuer and TMEM allocation, 2-5 dz converter
// and epilogue (thread = feature row = TMEM lane).  Every wait is bounded.
#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace da {
namespace {

constexpr int kDxThreads = 192;
constexpr int kDxN = 256;                  // features per MMA tile
constexpr int kRowB = 128;                 // bytes of one swizzled row: 64 bf16
constexpr int kA = 128 * kRowB;            // 16 KB: 128 tokens x 64 gate heads (hi or lo)
constexpr int kB = kDxN * kRowB;           // 32 KB: 256 features x 64 gate heads
constexpr int kBox = 128 * kRowB;          // 16 KB: one staging box, 128 tokens x 64 features
constexpr int kStg = 4 * kBox;             // 64 KB: a 128 x 256 staging tile
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + 2 * kA;
constexpr int kOffStg = kOffB + 2 * kB;
constexpr int kOffBar = kOffStg + 2 * kStg;  // 229376
constexpr int kDxSmem = kOffBar + 256 + 1024;
constexpr uint32_t kIdescDx = idesc_bf16(128, kDxN, 0);  // both operands K-major

enum { G_AREADY = 0, G_BFULL, G_BFULL1, G_BEMPTY, G_BEMPTY1, G_DFULL, G_DFULL1, G_DFREE, G_DFREE1, G_COUNT };

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * kRowB + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// wait until at most one bulk store group of this thread still reads shared memory
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

__global__ void __launch_bounds__(kDxThreads, 1)
gate_dx_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_dx, int T,
               int d_model, int h, const float* __restrict__ dz, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gen = smem_raw + (sb - raw);
  auto bar = [&](int i) { return sb + kOffBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gen + kOffBar + 128);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * 128;
  const int n_tiles = (d_model + kDxN - 1) / kDxN;
  const int ksteps = (h + 15) / 16;  // gate heads, 16 per MMA

  if (threadIdx.x == 0) {
    mbar_init(bar(G_AREADY), 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(G_BFULL + s), 1);
      mbar_init(bar(G_BEMPTY + s), 1);
      mbar_init(bar(G_DFULL + s), 1);
      mbar_init(bar(G_DFREE + s), 128);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- W tiles (TMA) --------
      prefetch_tmap(&tm_w);
      int issued = 0;
      for (int n = 0; n < n_tiles; ++n) {
        const int st = n & 1;
        if (n >= 2 && !mbar_wait(bar(G_BEMPTY + st), ((n >> 1) - 1) & 1, status, 0x7101)) break;
        mbar_arrive_expect_tx(bar(G_BFULL + st), kB);
        tma_load_4d(sb + kOffB + st * kB, &tm_w, bar(G_BFULL + st), 0, 0, n * kDxN, 0);
        issued = n + 1;
      }
      // every load issued lands before the CTA can leave
      for (int n = issued - 1; n >= 0 && n >= issued - 2; --n) mbar_wait(bar(G_BFULL + (n & 1)), (n >> 1) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuer ---
      bool ok = mbar_wait(bar(G_AREADY), 0, status, 0x7102);
      for (int n = 0; n < n_tiles && ok; ++n) {
        const int st = n & 1;  // W stage and accumulator
        ok = mbar_wait(bar(G_BFULL + st), (n >> 1) & 1, status, 0x7103);
        if (ok && n >= 2) ok = mbar_wait(bar(G_DFREE + st), ((n >> 1) - 1) & 1, status, 0x7104);
        if (!ok) break;
        tc_fence_after();
        const uint32_t bb = sb + kOffB + st * kB;
#pragma unroll 1
        for (int part = 0; part < 2; ++part)  // dz hi, then dz lo
          for (int kk = 0; kk < ksteps; ++kk)
            tc_mma_ss(tmem + st * kDxN, sdesc_sw128(sb + kOffA + part * kA + kk * 32, 16, 1024),
                      sdesc_sw128(bb + kk * 32, 16, 1024), kIdescDx, (part | kk) != 0 ? 1u : 0u);
        tc_commit(bar(G_BEMPTY + st));
        tc_commit(bar(G_DFULL + st));
      }
    }
  } else {
    // -------------------------------------------------------- epilogue -----
    const int q = warp & 3;             // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;      // token within the block
    const int t = t0 + row;
    const bool lead = warp == 2 && lane == 0;  // issues the stores
    // (1) this token's dz as hi + lo bf16 into the A tiles (zero past h / T)
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int p = c * 8 + e;
        v[e] = (t < T && p < h) ? dz[static_cast<int64_t>(t) * h + p] : 0.f;
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        hi[e] = *reinterpret_cast<const uint32_t*>(&hh);
        lo[e] = pack_bf16x2(v[2 * e] - __low2float(hh), v[2 * e + 1] - __high2float(hh));
      }
      *reinterpret_cast<uint4*>(gen + kOffA + sw128(row, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(gen + kOffA + kA + sw128(row, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    fence_proxy_async_smem();  // generic-proxy writes seen by the tensor cores
    mbar_arrive(bar(G_AREADY));
    // (2) each tile: TMEM -> bf16 -> staging -> TMA store.  A failed wait
    //     records its status and the loop carries on without waiting, so
    //     that the four warps reach the same named barriers.
    bool ok = true;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
    for (int n = 0; n < n_tiles; ++n) {
      const int st = n & 1;
      uint8_t* const stg = gen + kOffStg + st * kStg;
      if (n >= 2) {
        if (lead) bulk_wait_read_1();  // tile n - 2's stores have read this buffer
        epi_sync();
      }
      if (ok) ok = mbar_wait(bar(G_DFULL + st), (n >> 1) & 1, status, 0x7105);
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t o[128];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tmem_ld32(t_lane + st * kDxN + half * 128 + k * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[k * 32]));
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c) {  // 8 features per 16-byte chunk
          const uint4 pk = make_uint4(pack_bf16x2(__uint_as_float(o[8 * c]), __uint_as_float(o[8 * c + 1])),
                                      pack_bf16x2(__uint_as_float(o[8 * c + 2]), __uint_as_float(o[8 * c + 3])),
                                      pack_bf16x2(__uint_as_float(o[8 * c + 4]), __uint_as_float(o[8 * c + 5])),
                                      pack_bf16x2(__uint_as_float(o[8 * c + 6]), __uint_as_float(o[8 * c + 7])));
          *reinterpret_cast<uint4*>(stg + (half * 2 + (c >> 3)) * kBox + sw128(row, c & 7)) = pk;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(G_DFREE + st));
      fence_proxy_async_smem();  // the staging tile seen by the TMA unit
      epi_sync();
      if (lead && ok) {
        const uint32_t stg_s = sb + kOffStg + st * kStg;
        for (int box = 0; box < 4; ++box)
          if (n * kDxN + box * 64 < d_model)
            tma_store_4d(&tm_dx, stg_s + box * kBox, n * kDxN + box * 64, 0, t0, 0);
      }
      if (lead) bulk_commit();
    }
    if (lead) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- dW -----
constexpr int kDwThreads = 192;
constexpr int kDwStages = 3;
constexpr int kDwTok = 64;                     // tokens per stage (K)
constexpr int kDwXBox = kDwTok * kRowB;        // 8 KB: 64 tokens x 64 features
constexpr int kDwX = 2 * kDwXBox;              // 16 KB: 64 tokens x 128 features
constexpr int kDwZ = kDwTok * kRowB;           // 8 KB: 64 tokens x 64 heads (hi or lo)
constexpr int kDwStage = kDwX + 2 * kDwZ;      // 32 KB
constexpr int kDwOffBar = kDwStages * kDwStage;
constexpr int kDwSmem = kDwOffBar + 256 + 1024;
// M 128 features, N 64 heads, A (X) and B (dz) both MN-major
constexpr uint32_t kIdescDw = idesc_bf16(128, 64, 1) | (1u << 15);

enum { W_FULL = 0, W_EMPTY = W_FULL + kDwStages, W_ACC = W_EMPTY + kDwStages, W_COUNT };

__global__ void __launch_bounds__(kDwThreads, 2)
gate_dw_kernel(const __grid_constant__ CUtensorMap tm_x, int T, int d_model, int h, int chunk_tokens,
               const float* __restrict__ dz, float* __restrict__ part, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* gen = smem_raw + (sb - raw);
  auto bar = [&](int i) { return sb + kDwOffBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gen + kDwOffBar + 128);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 128;               // first feature
  const int chunk = blockIdx.y;
  const int tbeg = chunk * chunk_tokens, tend = min(T, tbeg + chunk_tokens);
  const int n_st = (tend - tbeg + kDwTok - 1) / kDwTok;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDwStages; ++s) {
      mbar_init(bar(W_FULL + s), 1 + 128);       // the producer's bytes + the converters
      mbar_init(bar(W_EMPTY + s), 1);
    }
    mbar_init(bar(W_ACC), 1);
    fence_mbar_init();
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
      // ------------------------------------------------- X stages (TMA) ----
      prefetch_tmap(&tm_x);
      int issued = 0;
      for (int k = 0; k < n_st; ++k) {
        const int st = k % kDwStages, use = k / kDwStages;
        if (use > 0 && !mbar_wait(bar(W_EMPTY + st), (use - 1) & 1, status, 0x7201)) break;
        mbar_arrive_expect_tx(bar(W_FULL + st), kDwX);
        const uint32_t xs = sb + st * kDwStage;
        tma_load_4d(xs, &tm_x, bar(W_FULL + st), c0, 0, tbeg + k * kDwTok, 0);
        tma_load_4d(xs + kDwXBox, &tm_x, bar(W_FULL + st), c0 + 64, 0, tbeg + k * kDwTok, 0);
        issued = k + 1;
      }
      for (int k = issued - 1; k >= 0 && k >= issued - kDwStages; --k)
        mbar_wait(bar(W_FULL + k % kDwStages), (k / kDwStages) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuer ---
      bool ok = true;
      for (int k = 0; k < n_st && ok; ++k) {
        const int st = k % kDwStages;
        ok = mbar_wait(bar(W_FULL + st), (k / kDwStages) & 1, status, 0x7202);
        if (!ok) break;
        tc_fence_after();
        const uint32_t xs = sb + st * kDwStage, zs = xs + kDwX;
#pragma unroll 1
        for (int part_i = 0; part_i < 2; ++part_i)  // dz hi, then dz lo
#pragma unroll
          for (int kk = 0; kk < kDwTok / 16; ++kk)
            tc_mma_ss(tmem, sdesc_sw128(xs + kk * 2048, kDwXBox, 1024),
                      sdesc_sw128(zs + part_i * kDwZ + kk * 2048, kDwZ, 1024), kIdescDw,
                      (k | part_i | kk) != 0 ? 1u : 0u);
        tc_commit(bar(W_EMPTY + st));
      }
      tc_commit(bar(W_ACC));  // also on the way out: every MMA issued completes first
    }
  } else {
    // ------------------------------------------ dz converter, epilogue -----
    const int q = warp & 3;
    const int r = q * 32 + lane;                 // 0..127
    const int tok = r >> 1, half = r & 1;        // token of the stage; heads 32 half ..
    // this thread's 32 heads of its token, loaded one stage ahead (float4:
    // h % 8 == 0, so a group of four heads is all valid or all past h)
    auto load = [&](int k, float4 (&v)[8]) {
      const int t = tbeg + k * kDwTok + tok;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const int p = half * 32 + g * 4;
        v[g] = (k < n_st && t < tend && p < h) ? *reinterpret_cast<const float4*>(dz + static_cast<int64_t>(t) * h + p)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    float4 nxt[8];
    load(0, nxt);
    bool ok = true;
#pragma unroll 1
    for (int k = 0; k < n_st; ++k) {
      const int st = k % kDwStages, use = k / kDwStages;
      float4 cur[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) cur[g] = nxt[g];
      load(k + 1, nxt);
      if (ok && use > 0) ok = mbar_wait(bar(W_EMPTY + st), (use - 1) & 1, status, 0x7203);
      uint8_t* const zs = gen + st * kDwStage + kDwX;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {           // 16-byte chunks of 8 heads
        const float v[8] = {cur[2 * cc].x, cur[2 * cc].y, cur[2 * cc].z, cur[2 * cc].w,
                            cur[2 * cc + 1].x, cur[2 * cc + 1].y, cur[2 * cc + 1].z, cur[2 * cc + 1].w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 hh = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
          hi[e] = *reinterpret_cast<const uint32_t*>(&hh);
          lo[e] = pack_bf16x2(v[2 * e] - __low2float(hh), v[2 * e + 1] - __high2float(hh));
        }
        const int c = half * 4 + cc;
        *reinterpret_cast<uint4*>(zs + sw128(tok, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(zs + kDwZ + sw128(tok, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(W_FULL + st));
    }
    // the partial sums of this CTA's 128 features: thread = feature row
    if (ok) ok = mbar_wait(bar(W_ACC), 0, status, 0x7204);
    tc_fence_after();
    uint32_t o[64];
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    tmem_ld32(t_lane, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
    tmem_ld32(t_lane + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
    tmem_ld_wait();
    const int c = c0 + q * 32 + lane;
    if (ok && c < d_model) {
      float* dst = part + (static_cast<int64_t>(chunk) * d_model + c) * h;
#pragma unroll
      for (int p = 0; p < 64; ++p)
        if (p < h) dst[p] = __uint_as_float(o[p]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 64);
}

}  // namespace

bool gate_dw_tc_ok(int T, int d_model, int h) {
  return T >= 64 && h > 0 && h <= 64 && h % 8 == 0 && d_model % 128 == 0;
}

cudaError_t launch_gate_dw_tc(int T, int d_model, int h, int chunk_tokens, int chunks, const float* dz, const void* X,
                              float* part, uint32_t* status, cudaStream_t s) {
  if (!gate_dw_tc_ok(T, d_model, h) || chunk_tokens % kDwTok) return cudaErrorInvalidValue;
  CUtensorMap tx;
  const da_t4 xt{const_cast<void*>(X), 0, d_model, 0};
  if (!encode_tmap_bf16_4d(&tx, xt, 1, T, 1, d_model, kDwTok)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gate_dw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDwSmem);
  if (e != cudaSuccess) return e;
  gate_dw_kernel<<<dim3(d_model / 128, chunks), kDwThreads, kDwSmem, s>>>(tx, T, d_model, h, chunk_tokens, dz, part,
                                                                        status);
  return cudaGetLastError();
}

bool gate_dx_tc_ok(int T, int d_model, int h) {
  return T >= 128 && h > 0 && h <= 64 && h % 8 == 0 && d_model % 64 == 0;
}

cudaError_t launch_gate_dx_tc(int T, int d_model, int h, const float* dz, const void* W, void* dx, uint32_t* status,
                              cudaStream_t s) {
  if (!gate_dx_tc_ok(T, d_model, h)) return cudaErrorInvalidValue;
  CUtensorMap tw, tdx;
  const da_t4 wt{const_cast<void*>(W), 0, h, 0};
  const da_t4 xt{dx, 0, d_model, 0};
  if (!encode_tmap_bf16_4d(&tw, wt, 1, d_model, 1, h, kDxN) || !encode_tmap_bf16_4d(&tdx, xt, 1, T, 1, d_model, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gate_dx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDxSmem);
  if (e != cudaSuccess) return e;
  gate_dx_kernel<<<(T + 127) / 128, kDxThreads, kDxSmem, s>>>(tw, tdx, T, d_model, h, dz, status);
  return cudaGetLastError();
}

}  // namespace da
