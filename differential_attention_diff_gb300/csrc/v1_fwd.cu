// v1_fwd.cu — V1 differential attention forward (bf16) on tcgen05 + TMEM + TMA
// with 2-CTA clusters, sm_103a.
//
// "Differential Transformer | ICLR 2025 Oral" (dainus.ai), "Differential
// Attention: 빼기의 힘":
//     O = (softmax(s Q1 K1^T) - lambda softmax(s Q2 K2^T)) V
// "Differential Transformer V2" (pogovet.com), §1: lambda is one scalar per
// layer from dot products of four learnable vectors plus the per-layer init;
// the V head dim is twice the Q/K head dim; per-head RMS normalisation after
// the subtraction, then the per-layer scale (read as 1 - lambda_init).
//
// One stream per CTA.  A stream needs 2 x 128 TMEM columns of scores (double
// buffered, so the next tile's Q K^T runs while the softmax works) plus 256
// columns for its O accumulator (d_v = 256): the whole 512-column TMEM of an
// SM.  So a work item (batch, head, 128 query rows) runs on a cluster of two
// CTAs: rank 0 computes stream 1, rank 1 stream 2, each from its own Q and K
// loads; V, which both streams multiply, is read once per pair: each CTA
// loads half of every V tile's column boxes with cluster multicast, into
// both CTAs' shared memory, and a V stage is refilled only once both CTAs'
// P.V MMAs are done with it (their commits arrive on both CTAs' barriers).
//
// The epilogue runs in warps of its own, under the next item's main loop.
// Shared memory is full with the Q tile and the K and V rings, so the
// epilogue keeps nothing there: each CTA keeps half of the 256 output
// columns; it writes the other half of its O/l to its exchange slot in the
// workspace (64 KB, which stays in L2) and tells the partner with a release
// arrive at cluster scope; it reads the partner's slot for its own half,
// forms O = O1/l1 - lambda O2/l2, swaps the per-row partial sums of squares
// through distributed shared memory (asynchronous 4-byte stores counted on
// an mbarrier), and writes Y = (1 - lambda_init) O / sqrt(mean O^2 + eps)
// straight from registers.  The O accumulator is released to the next
// item's first P.V as soon as the epilogue has read it out of TMEM.  Every
// hand-off is an mbarrier with a bounded wait.
//
//   TMEM: [0,128) S / P buffer 0, [128,256) S / P buffer 1, [256,256+DV) O.
//   SMEM: Q (32 KB), K ring 2 x 32 KB, V ring 2 x 64 KB (128-byte swizzle),
//   for head dims (128, 256); half of each for (64, 128).
//   warps 0-7: softmax, two warpgroups, each taking 64 key columns of every
//   tile (softmax.cuh; thread = query row = TMEM lane); warps 8-11:
//   epilogue (thread = query row); warps 12 and 14: TMA producers (Q and K;
//   V); warp 13: MMA issuer (one lane); warp 15 idle (it completes the
//   fourth warpgroup, whose registers go to the epilogue).
#include "kernels.h"
#include "softmax.cuh"
#include "tma.cuh"

namespace da {
namespace {

constexpr int kBM = 128, kBN = 128;
constexpr int kThreads = 512;
// registers per thread after the split: the epilogue warpgroup takes what
// the producer warpgroup gives up (launch: 512 x 128; after: 128 x 48 +
// 256 x 128 + 128 x 208, the same total)
constexpr int kRegsLow = 48, kRegsEpi = 208;
constexpr int kBox = 128 * 128;  // one 64-column box of 128 rows (bf16)
// Tiles for head dims (DQK, DV = 2 DQK) = (128, 256) or (64, 128), in boxes:
//   Q at 0 (DQK/64), K ring [stage][DQK/64] after it, V ring [stage][DV/64]
//   after that.  The barrier block sits after the largest layout.
constexpr int kOffBar = 14 * kBox;            // 229376
constexpr int kSmemBytes = kOffBar + 2048 + 1024;  // 232448: the per-block limit
// workspace: the work counter, then one exchange slot per CTA of
// 128 rows x 128 fp32 (the half of O/l its partner finishes)
constexpr size_t kXchgOff = 256;
constexpr size_t kXchgBytes = 128 * 128 * 4;

// K stages land per 64-column box ([stage][box]) and V stages per 64-key half
// ([stage][half]), so that a tile's first MMAs start before the rest of it
// has arrived
enum {
  B_QFULL = 0, B_QEMPTY, B_KFULL, B_KEMPTY = B_KFULL + 4, B_VFULL = B_KEMPTY + 2, B_VEMPTY = B_VFULL + 4,
  B_SFULL = B_VEMPTY + 2, B_PFULL = B_SFULL + 2, B_ORDY = B_PFULL + 2, B_ODONE, B_EPI, B_OFREE, B_XRDY,
  B_SSQ, B_SSQ1, B_SCHF, B_SCHE = B_SCHF + 4, B_COUNT = B_SCHE + 4
};
static_assert(B_COUNT * 8 <= 320, "barriers end where the TMEM slot begins");

constexpr uint32_t kIdescS = idesc_bf16(128, 128, 0);

struct Shared {
  uint32_t base;
  uint8_t* gen;
  __device__ uint32_t bar(int i) const { return base + kOffBar + 8 * i; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(gen + kOffBar + 320); }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(gen + kOffBar + 328);
  }
  __device__ float* lam() const { return reinterpret_cast<float*>(gen + kOffBar + 332); }
  // ring of the next work items (4 slots), written by rank 0's producer
  __device__ volatile int* ring() const { return reinterpret_cast<volatile int*>(gen + kOffBar + 336); }
  __device__ uint32_t ring_s(int slot) const { return base + kOffBar + 336 + 4 * slot; }
  // softmax -> epilogue hand-off of one item: its index, and each row's two
  // half sums of l, float[2][128] (on the rare tile that raises a row's max,
  // the softmax warpgroups swap their half maxima through the same slots)
  __device__ volatile int* epi_item() const { return reinterpret_cast<volatile int*>(gen + kOffBar + 352); }
  __device__ volatile float* epi_l() const { return reinterpret_cast<volatile float*>(gen + kOffBar + 1024); }
  // the partner's per-row partial sums of squares, float[128]: one slot
  // serves every item, since the partner sends an item's sums only after it
  // has my slot row of that item, which I write after reading its last sums
  __device__ uint32_t ssq_rx() const { return base + kOffBar + 512; }
  __device__ float* ssq_rx_ptr() const { return reinterpret_cast<float*>(gen + kOffBar + 512); }
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

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

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void remote_arrive(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
// four values of another SM's exchange slot, read at L2 (never a stale L1
// line of an earlier item)
__device__ __forceinline__ float4 ld_cg_f32x4(const float4* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// 4 bytes into a cluster peer's shared memory, completion counted in bytes on
// the peer's mbarrier
__device__ __forceinline__ void st_async_f32(uint32_t dst_cluster, float v, uint32_t bar_cluster) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst_cluster),
               "r"(__float_as_uint(v)), "r"(bar_cluster)
               : "memory");
}
template <int kRegs>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <int kRegs>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
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

struct Item {
  int b, h, mt, n_kv;
};
// Items are taken in blocks of `ub` (batch, head) units whose K1, K2 and V
// fit in L2 together; inside a block, heaviest causal rows first.
__device__ __forceinline__ Item item_of(int i, int units, int H, int n_mtiles, int ub, bool causal) {
  const int per_blk = n_mtiles * ub;
  const int blk = i / per_blk, r = i - blk * per_blk;
  const int bsize = min(ub, units - blk * ub);
  Item it;
  it.mt = n_mtiles - 1 - r / bsize;
  const int u = blk * ub + r % bsize;
  it.b = u / H;
  it.h = u % H;
  it.n_kv = causal ? it.mt + 1 : n_mtiles;  // causal: key tiles 0 .. mt; else all
  return it;
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
v1_fwd_kernel(const __grid_constant__ CUtensorMap tm_q1, const __grid_constant__ CUtensorMap tm_q2,
              const __grid_constant__ CUtensorMap tm_k1, const __grid_constant__ CUtensorMap tm_k2,
              const __grid_constant__ CUtensorMap tm_v, V1FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Shared sh;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t al = (raw + 1023u) & ~1023u;
    sh.base = al;
    sh.gen = smem_raw + (al - raw);
  }
  constexpr int kDv = DV;
  constexpr int kNQ = DQK / 64, kNV = DV / 64;  // 64-column boxes per tile row
  constexpr int kOffQ = 0, kOffK = kNQ * kBox, kOffV = 3 * kNQ * kBox;
  constexpr int kHalf = DV / 2;                 // output columns each CTA finishes
  constexpr uint32_t kIdescPV = idesc_bf16(128, DV, 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();         // 0: stream 1, 1: stream 2
  const uint32_t partner = rank ^ 1u;
  const int n_mtiles = (a.N + kBM - 1) / kBM;
  const int units = a.B * a.H;
  const int n_items = n_mtiles * units;
  const bool causal = a.causal != 0;
  // units per L2 block: K1 + K2 + V of one (batch, head) is N (2 DQK + DV) * 2 bytes
  const int ub = max(1, min(units, static_cast<int>((48ll << 20) /
                                                    (static_cast<long long>(a.N) * (2 * DQK + DV) * 2))));
  const CUtensorMap* tq = rank == 0 ? &tm_q1 : &tm_q2;
  const CUtensorMap* tk = rank == 0 ? &tm_k1 : &tm_k2;

  if (threadIdx.x == 0) {
    mbar_init(sh.bar(B_QFULL), 1);
    mbar_init(sh.bar(B_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(sh.bar(B_KFULL + 2 * s), 1);
      mbar_init(sh.bar(B_KFULL + 2 * s + 1), 1);
      mbar_init(sh.bar(B_KEMPTY + s), 1);
      mbar_init(sh.bar(B_VFULL + 2 * s), 1);
      mbar_init(sh.bar(B_VFULL + 2 * s + 1), 1);
      mbar_init(sh.bar(B_VEMPTY + s), 2);  // both CTAs' P.V commits
      mbar_init(sh.bar(B_SFULL + s), 1);
      mbar_init(sh.bar(B_PFULL + s), 256);
    }
    mbar_init(sh.bar(B_ORDY), 1);
    mbar_init(sh.bar(B_ODONE), 1);
    mbar_init(sh.bar(B_EPI), 256);    // softmax threads: item handed to the epilogue
    mbar_init(sh.bar(B_OFREE), 128);  // epilogue rows: O read out of TMEM
    mbar_init(sh.bar(B_XRDY), 128);   // the partner's epilogue rows: its slot is written
    mbar_init(sh.bar(B_SSQ), 1);      // + 512 bytes of the partner's partial sums
    mbar_init(sh.bar(B_SSQ1), 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(sh.bar(B_SCHF + q), 1);
      mbar_init(sh.bar(B_SCHE + q), 2);  // one epilogue thread of each CTA
    }
    *sh.abort_flag() = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init
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
    if (lane == 0) {
      const float lam = expf(d1) - expf(d2) + a.lambda_init;
      *sh.lam() = lam;
      if (a.lambda_out && blockIdx.x == 0) *a.lambda_out = lam;
    }
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(sh.tmem_slot()), 512);
    tmem_relinquish();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tmap(tq);
    prefetch_tmap(tk);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the partner's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot();

  // ---- dynamic work distribution ------------------------------------------
  // Rank 0's producer takes item indices from a global counter (zeroed by the
  // host before the launch; heaviest items come first in index order) and
  // publishes them to a 4-slot ring in both CTAs, item k + 1 while it loads
  // item k's first key tiles (so that neither the atomic nor the arrives sit
  // between two items); the producer, MMA and softmax roles of both CTAs
  // read the same sequence (the epilogue warps get each item from the
  // softmax warps).  Index >= n_items ends the sequence.  A slot is released
  // in each CTA by one epilogue thread once it has the item, by which time
  // every reader in that CTA has read it: an arrive on the other CTA's
  // barrier with a cluster-scope release costs the arriving thread about
  // 0.8 us, which the producer, MMA and softmax roles would otherwise pay at
  // every item start.
  int* counter = static_cast<int*>(a.workspace);
  auto publish = [&](int k) -> int {  // rank 0 producer only
    const int slot = k & 3;
    if (k >= 4 && !wait_bar(sh, sh.bar(B_SCHE + slot), ((k >> 2) - 1) & 1, a.status, 0x3008)) return -1;
    const int idx = atomicAdd(counter, 1);
    sh.ring()[slot] = idx;
    st_cluster_s32(map_to_rank(sh.ring_s(slot), partner), idx);
    mbar_arrive(sh.bar(B_SCHF + slot));
    remote_arrive(map_to_rank(sh.bar(B_SCHF + slot), partner));
    return idx;
  };
  // consumers: the k-th item index (-1 on timeout)
  auto release = [&](int k) {
    const int slot = k & 3;
    if (rank == 0) mbar_arrive(sh.bar(B_SCHE + slot));
    else remote_arrive(map_to_rank(sh.bar(B_SCHE + slot), 0));
  };
  auto consume = [&](int k) -> int {
    const int slot = k & 3;
    if (!wait_bar<true>(sh, sh.bar(B_SCHF + slot), (k >> 2) & 1, a.status, 0x3009)) return -1;
    return sh.ring()[slot];
  };

  if (warp >= 12) {
    regs_dec<kRegsLow>();
    if (warp == 12 || warp == 14) {
      // ----------------------------------------------------- TMA producers --
      // warp 12: the Q and K tiles (and, in rank 0, the work ring); warp 14:
      // the V tiles.  Two threads, so that a K load waits only for its own
      // ring stage, never behind a V stage that a P.V still reads.
      if (lane == 0) {
        const bool qk = warp == 12;
        int kv = 0;
        bool ok = true;
        int next = (qk && rank == 0) ? publish(0) : 0;
        for (int it = 0; ok; ++it) {
          const int i = (qk && rank == 0) ? next : consume(it);
          if (i < 0) { ok = false; break; }
          if (i >= n_items) break;
          const Item w = item_of(i, units, a.H, n_mtiles, ub, causal);
          if (qk) {
            if (it > 0 && !wait_bar(sh, sh.bar(B_QEMPTY), (it - 1) & 1, a.status, 0x3001)) { ok = false; break; }
            mbar_arrive_expect_tx(sh.bar(B_QFULL), kNQ * kBox);
            for (int box = 0; box < kNQ; ++box)
              tma_load_4d(sh.base + kOffQ + box * kBox, tq, sh.bar(B_QFULL), box * 64, w.h, w.mt * kBM, w.b);
          }
          for (int j = 0; j < w.n_kv; ++j, ++kv) {
            const int st = kv & 1, use = kv >> 1;
            if (qk) {
              if (use > 0 && !wait_bar(sh, sh.bar(B_KEMPTY + st), (use - 1) & 1, a.status, 0x3002)) { ok = false; break; }
              for (int box = 0; box < kNQ; ++box) {
                mbar_arrive_expect_tx(sh.bar(B_KFULL + 2 * st + box), kBox);
                tma_load_4d(sh.base + kOffK + (st * kNQ + box) * kBox, tk, sh.bar(B_KFULL + 2 * st + box), box * 64,
                            w.h, j * kBN, w.b);
              }
              if (rank == 0 && j == min(1, w.n_kv - 1)) next = publish(it + 1);
            } else {
              if (use > 0 && !wait_bar(sh, sh.bar(B_VEMPTY + st), (use - 1) & 1, a.status, 0x3003)) { ok = false; break; }
              // each 64-key half of the tile lands whole here: this CTA's
              // column boxes and the partner's (64-row boxes: the second
              // half sits 8 KB into each 128-row box, the swizzle unchanged)
              for (int half = 0; half < 2; ++half) {
                mbar_arrive_expect_tx(sh.bar(B_VFULL + 2 * st + half), kNV * (kBox / 2));
                for (int box = static_cast<int>(rank) * (kNV / 2); box < (static_cast<int>(rank) + 1) * (kNV / 2);
                     ++box)
                  tma_load_4d_mc(sh.base + kOffV + (st * kNV + box) * kBox + half * (kBox / 2), &tm_v,
                                 sh.bar(B_VFULL + 2 * st + half), box * 64, w.h, j * kBN + half * 64, w.b, 3);
              }
            }
          }
        }
        if (!ok) {
          // bounded drain of the loads that may still be in flight
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 200000000ull) {
          }
        }
      }
    } else if (warp == 13) {
      // ------------------------------------------------------- MMA issuer ---
      if (lane == 0) {
        int kv = 0, it = 0;
        bool ok = true;
        const uint32_t t_o = tmem + 256;
        // S of global tile g into buffer g & 1, each 64-column box of K as
        // soon as it has landed (false on a failed wait)
        auto issue_s = [&](int g) -> bool {
          const int st = g & 1;
          const uint32_t kb = sh.base + kOffK + st * kNQ * kBox;
          const uint32_t qa = sh.base + kOffQ;
  #pragma unroll
          for (int box = 0; box < kNQ; ++box) {
            if (!wait_bar(sh, sh.bar(B_KFULL + 2 * st + box), (g >> 1) & 1, a.status, 0x3102)) return false;
            tc_fence_after();
  #pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
              const uint32_t off = box * kBox + kq * 32;
              tc_mma_ss(tmem + st * 128, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                        kIdescS, (box | kq) != 0 ? 1u : 0u);
            }
          }
          return true;
        };
        for (;; ++it) {
          const int i = consume(it);
          if (i < 0) { ok = false; break; }
          if (i >= n_items) break;
          const Item w = item_of(i, units, a.H, n_mtiles, ub, causal);
          const int n = w.n_kv;
          if (!wait_bar(sh, sh.bar(B_QFULL), it & 1, a.status, 0x3101)) { ok = false; break; }
          tc_fence_after();
          for (int j = 0; j < 2 && j < n; ++j) {
            if (!issue_s(kv + j)) { ok = false; break; }
            tc_commit(sh.bar(B_KEMPTY + ((kv + j) & 1)));
            tc_commit(sh.bar(B_SFULL + ((kv + j) & 1)));
            if (j == n - 1) tc_commit(sh.bar(B_QEMPTY));
          }
          if (!ok) break;
          for (int j = 0; j < n; ++j) {
            const int g = kv + j, st = g & 1;
            // the first P.V overwrites O: the previous item's epilogue has read it
            if (j == 0 && it > 0 && !wait_bar(sh, sh.bar(B_OFREE), (it - 1) & 1, a.status, 0x3105)) {
              ok = false;
              break;
            }
            if (!wait_bar(sh, sh.bar(B_PFULL + st), (g >> 1) & 1, a.status, 0x3103)) { ok = false; break; }
            const uint32_t vb = sh.base + kOffV + st * kNV * kBox;
            // each 64-key half of V as soon as it has landed; P of keys
            // 64 h .. 64 h + 63 sits at columns 64 h .. of the buffer
  #pragma unroll
            for (int half = 0; half < 2 && ok; ++half) {
              if (!wait_bar(sh, sh.bar(B_VFULL + 2 * st + half), (g >> 1) & 1, a.status, 0x3104)) {
                ok = false;
                break;
              }
              tc_fence_after();
  #pragma unroll
              for (int kq = 0; kq < 4; ++kq) {
                const int kk = half * 4 + kq;
                tc_mma_ts(t_o, tmem + st * 128 + half * 64 + kq * 8, sdesc_sw128(vb + kk * 2048, kBox, 1024),
                          kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
              }
            }
            if (!ok) break;
            tc_commit_mc(sh.bar(B_VEMPTY + st), 3);  // the stage is free in both CTAs
            tc_commit(sh.bar(B_ODONE));
            if (j + 2 < n) {
              if (!issue_s(g + 2)) { ok = false; break; }
              tc_commit(sh.bar(B_KEMPTY + st));
              tc_commit(sh.bar(B_SFULL + st));
              if (j + 2 == n - 1) tc_commit(sh.bar(B_QEMPTY));
            }
          }
          if (!ok) break;
          tc_commit(sh.bar(B_ORDY));
          kv += n;
        }
      }
    }
    // warp 15: idle (it completes the producer warpgroup)
  } else if (warp < 8) {
    // ------------------------------------------------------- softmax ------
    // Both warpgroups work on every tile: warpgroup wg takes key columns
    // [64 wg, 64 wg + 64) (thread = query row = TMEM lane) and writes its P
    // as bf16 pairs over the first 32 of those columns, so a tile's
    // exponentials run on eight warps.  The halves of a row share one running
    // max: on a row's first tile both read the whole row and take the same
    // max (a barrier keeps either from writing P over scores the other still
    // reads); later tiles keep that stale max, and on the rare tile whose sum
    // leaves the guard in some half (a barrier reduction over both
    // warpgroups decides) both halves recompute against a max raised over the
    // tile, swapped through shared memory.  Named barrier 1 (these 256
    // threads) is reached by both warpgroups in the same sequence: a failed
    // wait only clears `ok`, and every stop is decided by a barrier reduction.
    const int wg = warp >> 2, q4 = warp & 3;
    const int row = q4 * 32 + lane;  // query row within the item = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int c0 = wg * 64;          // first key column of this half
    const uint32_t t_oh = tmem + lane_off + 256 + wg * kHalf;  // this half's O columns (rescale)
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    float* lse = rank == 0 ? a.lse1 : a.lse2;
    volatile float* xl = sh.epi_l();  // [half][row]
    int kv = 0;
    bool ok = true;
    for (int it = 0;; ++it) {
      const int i = consume(it);
      if (named_red_or_256(i < 0 || !ok)) break;
      // (the hand-off slots are free once the epilogue warps have taken the
      // previous item: they read them before they release O)
      if (i >= n_items) {
        if (it > 0 && !wait_bar(sh, sh.bar(B_OFREE), (it - 1) & 1, a.status, 0x3209)) break;
        if (threadIdx.x == 0) *sh.epi_item() = n_items;  // end of the sequence
        mbar_arrive(sh.bar(B_EPI));
        break;
      }
      const Item w = item_of(i, units, a.H, n_mtiles, ub, causal);
      float m_run = -INFINITY, l_half = 0.f;
      for (int j = 0; j < w.n_kv; ++j) {
        const int g = kv + j;
        const uint32_t t_s = tmem + lane_off + (g & 1) * 128;
        if (!wait_bar(sh, sh.bar(B_SFULL + (g & 1)), (g >> 1) & 1, a.status, 0x3201)) ok = false;
        tc_fence_after();
        // masked columns: keys after the query (causal diagonal tile), or
        // keys >= N (ragged last tile without the causal mask)
        const bool masked = causal ? j == w.mt : (j == w.n_kv - 1 && (a.N % kBN) != 0);
        const int lim = causal ? row : a.N - 1 - j * kBN;
        uint32_t sv[64];
        tmem_ld32(t_s + c0, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(t_s + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        if (j == 0) {
          // the row max over both halves (the same value in both warpgroups)
          const int o0 = c0 ^ 64;
          uint32_t ov[32];
          tmem_ld32(t_s + o0, ov);
          tmem_ld_wait();
          float mx = masked ? half_max<true>(sv, c0, lim) : half_max<false>(sv, c0, lim);
          mx = masked ? chunk_max<true>(ov, o0, lim, mx) : chunk_max<false>(ov, o0, lim, mx);
          tmem_ld32(t_s + o0 + 32, ov);
          tmem_ld_wait();
          mx = masked ? chunk_max<true>(ov, o0 + 32, lim, mx) : chunk_max<false>(ov, o0 + 32, lim, mx);
          m_run = mx * sl2;
          named_sync_256();  // both halves have read the row
          l_half = masked ? exp_half<true>(sv, c0, lim, sl2x2, m_run, t_s + c0)
                          : exp_half<false>(sv, c0, lim, sl2x2, m_run, t_s + c0);
        } else {
          tmem_ld_wait();
          float lsum = masked ? exp_half<true>(sv, c0, lim, sl2x2, m_run, t_s + c0)
                              : exp_half<false>(sv, c0, lim, sl2x2, m_run, t_s + c0);
          if (named_red_or_256(!(lsum <= kSumGuard))) {
            // rare: some row's half left the guard.  Both halves of every row
            // recompute against a max raised over this tile; the half maxima
            // go through the hand-off slots, which the epilogue has left once
            // it released the previous item's O
            if (it > 0 && !wait_bar(sh, sh.bar(B_OFREE), (it - 1) & 1, a.status, 0x320b)) ok = false;
            const float hm = masked ? half_max<true>(sv, c0, lim) : half_max<false>(sv, c0, lim);
            xl[wg * 128 + row] = hm;
            named_sync_256();
            const float m_new = fmaxf(m_run, fmaxf(hm, xl[(wg ^ 1) * 128 + row]) * sl2);
            const float alpha = fast_exp2(m_run - m_new);
            m_run = m_new;
            lsum = masked ? exp_half<true>(sv, c0, lim, sl2x2, m_new, t_s + c0)
                          : exp_half<false>(sv, c0, lim, sl2x2, m_new, t_s + c0);
            l_half = l_half * alpha + lsum;
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
              // PV(g - 1) may still run: wait for it before rescaling this
              // half's columns of O
              if (!wait_bar(sh, sh.bar(B_ODONE), (g - 1) & 1, a.status, 0x3202)) ok = false;
              tc_fence_after();
#pragma unroll 1
              for (int c = 0; c < kHalf / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(t_oh + c * 32, o);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st32(t_oh + c * 32, o);
              }
            }
            named_sync_256();  // both halves have read the swapped maxima
          } else {
            l_half += lsum;
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(sh.bar(B_PFULL + (g & 1)));
      }
      kv += w.n_kv;
      // hand the item and the row's half sums to the epilogue warps
      if (it > 0 && !wait_bar(sh, sh.bar(B_OFREE), (it - 1) & 1, a.status, 0x320a)) ok = false;
      xl[wg * 128 + row] = l_half;
      named_sync_256();
      if (wg == 0) {
        const int n = w.mt * kBM + row;
        const float l_run = xl[row] + xl[128 + row];
        if (lse && n < a.N)
          lse[(static_cast<int64_t>(w.b) * a.H + w.h) * a.N + n] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      }
      if (threadIdx.x == 0) *sh.epi_item() = i;
      mbar_arrive(sh.bar(B_EPI));
    }
  } else {
    // ------------------------------------------------------ epilogue ------
    regs_inc<kRegsEpi>();
    const int q = warp - 8;
    const int row = q * 32 + lane;  // query row = TMEM lane of this warp's quadrant
    const uint32_t t_o = tmem + (static_cast<uint32_t>(q * 32) << 16) + 256;
    const float lam = *sh.lam();
    const float cscale = 1.f - a.lambda_init;
    const int give = (1 - static_cast<int>(rank)) * kHalf, keep = static_cast<int>(rank) * kHalf;
    // exchange slots: 128 rows x kHalf fp32 (O/l of the columns the partner
    // finishes), stored as float4 groups of four columns, group-major, so
    // that one 16-byte store per lane writes 512 contiguous bytes per warp
    float* xchg = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + kXchgOff);
    const size_t cl = blockIdx.x >> 1;
    // (columns 4k .. 4k + 3 of a row at float4 [k * 128 + row])
    float4* my_x = reinterpret_cast<float4*>(xchg + (cl * 2 + rank) * 128 * kHalf) + row;
    const float4* partner_x = reinterpret_cast<const float4*>(xchg + (cl * 2 + partner) * 128 * kHalf) + row;
    const uint32_t partner_xrdy = map_to_rank(sh.bar(B_XRDY), partner);
    const uint32_t partner_ssq_bar0 = map_to_rank(sh.bar(B_SSQ), partner);
    const uint32_t partner_ssq_bar1 = map_to_rank(sh.bar(B_SSQ1), partner);
    const uint32_t partner_ssq_slot = map_to_rank(sh.ssq_rx() + row * 4, partner);
    const bool want_o2 = a.o2.ptr != nullptr;
    __nv_bfloat16* const yb = static_cast<__nv_bfloat16*>(a.out.ptr);
    __nv_bfloat16* const o2b = static_cast<__nv_bfloat16*>(a.o2.ptr);
    // bf16 of 8 values, 16 bytes
    auto pack8 = [](const float* v) {
      uint4 pk;
      pk.x = pack_bf16x2(v[0], v[1]);
      pk.y = pack_bf16x2(v[2], v[3]);
      pk.z = pack_bf16x2(v[4], v[5]);
      pk.w = pack_bf16x2(v[6], v[7]);
      return pk;
    };
    for (int it = 0;; ++it) {
      if (!wait_bar(sh, sh.bar(B_EPI), it & 1, a.status, 0x3203)) break;
      const int i = *sh.epi_item();
      const float l_run = sh.epi_l()[row] + sh.epi_l()[128 + row];
      if (i >= n_items) break;
      const Item w = item_of(i, units, a.H, n_mtiles, ub, causal);
      if (!wait_bar(sh, sh.bar(B_ORDY), it & 1, a.status, 0x3204)) break;
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      // (1) the partner's half of my O/l into my exchange slot
#pragma unroll 1
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_o + give + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e)
          my_x[(c * 8 + e) * 128] = make_float4(__uint_as_float(o[4 * e]) * inv_l, __uint_as_float(o[4 * e + 1]) * inv_l,
                                                __uint_as_float(o[4 * e + 2]) * inv_l, __uint_as_float(o[4 * e + 3]) * inv_l);
      }
      // (2) my own half of O/l into registers
      float dvals[kHalf];
#pragma unroll
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_o + keep + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) dvals[c * 32 + e] = __uint_as_float(o[e]) * inv_l;
      }
      // O has been read: the next item's first P.V may overwrite it; my slot
      // row is written: release it to the partner (cluster scope orders the
      // slot stores before the arrive)
      tc_fence_before();
      mbar_arrive(sh.bar(B_OFREE));
      remote_arrive(partner_xrdy);
      if (q == 0 && lane == 0) release(it);  // the item's ring slot: every reader in this CTA has read it
      const int n = w.mt * kBM + row;
      const bool live = n < a.N;
      const int64_t yrow = static_cast<int64_t>(w.b) * a.out.sb + static_cast<int64_t>(n) * a.out.sn +
                           static_cast<int64_t>(w.h) * a.out.sh + keep;
      const int64_t o2row = static_cast<int64_t>(w.b) * a.o2.sb + static_cast<int64_t>(n) * a.o2.sn +
                            static_cast<int64_t>(w.h) * a.o2.sh + keep;
      if (want_o2 && rank == 1 && live) {
        // O2 / l2 of my columns: my own stream
#pragma unroll
        for (int e = 0; e < kHalf; e += 8) *reinterpret_cast<uint4*>(o2b + o2row + e) = pack8(&dvals[e]);
      }
      // (3) the partner's half of its O/l for my columns
      if (!wait_bar<true>(sh, sh.bar(B_XRDY), it & 1, a.status, 0x3205)) break;
      float ssq = 0.f;
#pragma unroll
      for (int c = 0; c < kHalf / 32; ++c) {
        float oth[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) *reinterpret_cast<float4*>(&oth[4 * e]) = ld_cg_f32x4(partner_x + (c * 8 + e) * 128);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float own = dvals[c * 32 + e];
          const float a1 = rank == 0 ? own : oth[e];
          const float a2 = rank == 0 ? oth[e] : own;
          const float dd = __fsub_rn(a1, __fmul_rn(lam, a2));
          dvals[c * 32 + e] = dd;
          ssq = fmaf(dd, dd, ssq);
        }
      }
      if (want_o2 && rank == 0 && live) {
        // O2 / l2 of my columns: received
#pragma unroll 1
        for (int e = 0; e < kHalf; e += 8) {
          float v[8];
          *reinterpret_cast<float4*>(&v[0]) = ld_cg_f32x4(partner_x + (e / 4) * 128);
          *reinterpret_cast<float4*>(&v[4]) = ld_cg_f32x4(partner_x + (e / 4 + 1) * 128);
          *reinterpret_cast<uint4*>(o2b + o2row + e) = pack8(v);
        }
      }
      // (4) swap the per-row partial sums: one asynchronous 4-byte store per
      //     row into the partner's slot of this item's parity, its bytes
      //     counted on the partner's barrier of that parity (one local arrive
      //     with the expected 512 bytes per phase).  The partner sends its
      //     sums only after it has read my slot, so once they are here my
      //     slot may take the next item.
      const int sp = it & 1;
      if (row == 0) mbar_arrive_expect_tx(sh.bar(B_SSQ + sp), 128 * 4);
      st_async_f32(partner_ssq_slot, ssq, sp ? partner_ssq_bar1 : partner_ssq_bar0);
      if (!wait_bar<true>(sh, sh.bar(B_SSQ + sp), (it >> 1) & 1, a.status, 0x3206)) {
        // abort path: the partner's asynchronous stores into this CTA's
        // shared memory may still be in flight; give them a short, bounded
        // time to land before this CTA can leave (barrier.cluster does not
        // wait for them)
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000000ull && !try_wait_cluster(sh.bar(B_SSQ + sp), (it >> 1) & 1)) {
        }
        break;
      }
      const float other_ssq = sh.ssq_rx_ptr()[row];
      const float tot = rank == 0 ? ssq + other_ssq : other_ssq + ssq;
      const float rstd = 1.f / sqrtf(tot * (1.f / kDv) + a.rms_eps);
      const float cs = cscale * rstd;
      // (5) Y = (1 - lambda_init) w O / rms on my columns, straight to HBM
      if (live) {
        if (a.rms_weight) {
          const float* wk = a.rms_weight + keep;
#pragma unroll
          for (int e = 0; e < kHalf; ++e) dvals[e] = __fmul_rn(__fmul_rn(dvals[e], cs), __ldg(wk + e));
        } else {
#pragma unroll
          for (int e = 0; e < kHalf; ++e) dvals[e] = __fmul_rn(dvals[e], cs);
        }
#pragma unroll
        for (int e = 0; e < kHalf; e += 8) *reinterpret_cast<uint4*>(yb + yrow + e) = pack8(&dvals[e]);
        if (rank == 0 && a.rstd) a.rstd[(static_cast<int64_t>(w.b) * a.H + w.h) * a.N + n] = rstd;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its partner may still address its shared memory
  tc_fence_after();
  if (warp == 13) tmem_dealloc(tmem, 512);
}

}  // namespace

// the work counter of the dynamic schedule and one exchange slot per CTA
size_t v1_fwd_workspace_bytes(int num_sms) {
  const int sms = num_sms > 0 ? num_sms : 152;
  return kXchgOff + static_cast<size_t>(sms / 2) * 2 * kXchgBytes;
}

namespace {

template <int DQK, int DV>
cudaError_t launch_dims(const V1FwdArgs& a, cudaStream_t s) {
  constexpr int kDqk = DQK, kDv = DV;
  CUtensorMap tq1, tq2, tk1, tk2, tv;
  if (!encode_tmap_bf16_4d(&tq1, a.q1, a.B, a.N, a.H, kDqk, kBM) ||
      !encode_tmap_bf16_4d(&tq2, a.q2, a.B, a.N, a.H, kDqk, kBM) ||
      !encode_tmap_bf16_4d(&tk1, a.k1, a.B, a.N, a.H, kDqk, kBN) ||
      !encode_tmap_bf16_4d(&tk2, a.k2, a.B, a.N, a.H, kDqk, kBN) ||
      !encode_tmap_bf16_4d(&tv, a.v, a.B, a.N, a.H, kDv, kBN / 2))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(v1_fwd_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_items = ((a.N + kBM - 1) / kBM) * a.B * a.H;
  const int sms = a.num_sms > 0 ? a.num_sms : 152;
  // clusters of two CTAs; as many as fit at once (one CTA per SM), and no
  // more than the workspace has exchange slots for
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = 0;
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  e = cudaOccupancyMaxActiveClusters(&max_clusters, v1_fwd_kernel<DQK, DV>, &cfg);
  if (e != cudaSuccess || max_clusters <= 0) max_clusters = sms / 2;
  int clusters = max_clusters;
  if (clusters > sms / 2) clusters = sms / 2;
  if (clusters > n_items) clusters = n_items;
  if (clusters <= 0) return cudaErrorInvalidValue;
  if (a.workspace_bytes < kXchgOff + static_cast<size_t>(clusters) * 2 * kXchgBytes) return cudaErrorInvalidValue;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  e = cudaMemsetAsync(a.workspace, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, v1_fwd_kernel<DQK, DV>, tq1, tq2, tk1, tk2, tv, a);
}

}  // namespace

cudaError_t launch_v1_fwd(const V1FwdArgs& a, cudaStream_t s) {
  if (a.d_qk == 128 && a.d_v == 256) return launch_dims<128, 256>(a, s);
  if (a.d_qk == 64 && a.d_v == 128) return launch_dims<64, 128>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace da
