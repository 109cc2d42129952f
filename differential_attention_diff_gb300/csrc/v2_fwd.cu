// v2_fwd.cu — V2 differential attention forward on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), sm_103a.
//
// "Differential Transformer V2" (pogovet.com), §1 and the one-line summary:
// one causal GQA attention over 2h query heads; heads 2p and 2p+1 share one
// K/V head (same group) and are combined per token as
//     out[t, p] = O[t, 2p] - gate[t, p] * O[t, 2p + 1].
//
// One CTA (persistent, one per SM) owns a work item = (batch, pair p, 128
// query rows) at a time, heaviest causal rows first, dealt in a snake order.  Both heads of the pair
// are computed side by side against the same K/V tiles, each tile fetched
// once by TMA for the two heads:
//
//   TMEM (512 columns x 128 lanes, lane = query row):
//     [  0,128) S_even (fp32 scores) / P_even (bf16, first 64 columns)
//     [128,256) S_odd / P_odd
//     [256,384) O_even accumulator     [384,512) O_odd accumulator
//     (head dim D = 64 or 128: the first D columns of each O region)
//   Shared memory: Q_even, Q_odd (2 x D/64 boxes), K and V rings of 2 stages
//   (2 x 2 x D/64 boxes), all in 128-byte-swizzled 64-column boxes of 128
//   rows (16 KB each).
//
//   warp 8 (one lane): TMA producer — Q of the item, then K_j, V_j per tile.
//   warp 9 (one lane): MMA issuer — S = Q K^T (SS form) and O += P V (P read
//     from TMEM, V from shared memory), interleaving the two heads so that
//     one head's softmax overlaps the other head's MMAs.
//   warps 0-7: softmax of every tile of both heads, split by key columns:
//     warpgroup 0 takes keys 0-63 of the tile, warpgroup 1 keys 64-127 (one
//     thread per query row and half), so a head's tile is done by eight warps
//     and its next P.V and S MMAs start sooner (the per-head chain softmax ->
//     P.V -> next S bounds the loop).  Online softmax per tile (the row max
//     of the first tile, shared by the two halves; a guarded stale max
//     afterwards), P written back to TMEM as bf16 over the columns each half
//     read, O rescaled in TMEM on the rare tiles that raise the max.  The
//     same threads run the epilogue (each warpgroup half of the D features):
//     O_even / l_even - gate * O_odd / l_odd, bf16 store, optional
//     log-sum-exp and per-head outputs (the backward's saves).  With no
//     output tensor the kernel writes only the per-head outputs (the
//     attention part of grouped differential attention, whose groups span
//     more than a pair).
//
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records
// DA_ERR_TIMEOUT in the status word, raises a shared abort flag so the other
// roles leave too, drains its TMA loads and frees TMEM before returning.
#include "kernels.h"
#include "softmax.cuh"
#include "tma.cuh"

namespace da {
namespace {

constexpr int kBM = 128;   // query rows per item
constexpr int kBN = 128;   // keys per tile
constexpr int kThreads = 320;
constexpr int kBox = 128 * 128;            // bytes of one 64-column box of 128 rows
// Tiles for head dim D (64 or 128) take D / 64 boxes per 128-row tile:
//   Q [head][box] at 0, K [stage][box] at 2 D/64 boxes, V [stage][box] at
//   4 D/64 boxes.  The barrier block sits after the largest (D = 128) layout.
constexpr int kOffBar = 12 * kBox;         // 196608
constexpr int kSmemBytes = kOffBar + 8192 + 1024;  // + barriers/exchange + alignment slack

// barrier indices (8 bytes each)
enum {
  B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_VFULL = 4, B_KVEMPTY = 6, B_SFULL = 8,
  B_PFULL = 10, B_ORDY = 12, B_EPI = 13, B_COUNT = 14
};

constexpr uint32_t kIdescS = idesc_bf16(128, 128, 0);   // Q (K-major) x K (K-major)

struct Shared {
  uint32_t base;  // 1024-aligned shared address of the tile region
  uint8_t* gen;   // same, generic pointer
  __device__ uint32_t bar(int i) const { return base + kOffBar + 8 * i; }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(gen + kOffBar + 128); }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(gen + kOffBar + 192);
  }
  // per-row partial sums [head][half][128] and half maxima [head][half][128]
  __device__ float* lx() const { return reinterpret_cast<float*>(gen + kOffBar + 256); }
  __device__ float* xm() const { return reinterpret_cast<float*>(gen + kOffBar + 256 + 2048); }
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait that also gives up when another role raised the abort flag.
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

struct Item {
  int b, p, mt, n_kv;
};

__device__ __forceinline__ Item item_of(int i, int units, int h, int n_mtiles, bool causal) {
  Item it;
  it.mt = n_mtiles - 1 - i / units;
  const int u = i % units;
  it.b = u / h;
  it.p = u % h;
  it.n_kv = causal ? it.mt + 1 : n_mtiles;  // causal: key tiles 0 .. mt; else all
  return it;
}

// The k-th item of this CTA: rounds of gridDim.x items taken heaviest first,
// every other round in reverse CTA order (a snake), so that no CTA draws the
// largest item of every round (1.03-1.09x -> 1.00x the ideal makespan for
// causal item sizes).  Increasing in k, so a CTA stops at its first index
// past the end.
__device__ __forceinline__ int sched(int k) {
  return k * static_cast<int>(gridDim.x) +
         ((k & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
v2_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, V2FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Shared sh;
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t aligned = (raw + 1023u) & ~1023u;
    sh.base = aligned;
    sh.gen = smem_raw + (aligned - raw);
  }
  constexpr int kNB = D / 64;                 // 64-column boxes per tile row
  constexpr int kOffQ = 0, kOffK = 2 * kNB * kBox, kOffV = 4 * kNB * kBox;
  constexpr uint32_t kIdescPV = idesc_bf16(128, D, 1);  // P (TMEM) x V (MN-major)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (2 * a.h) / a.h_kv;
  const int n_mtiles = (a.N + kBM - 1) / kBM;
  const int units = a.B * a.h;
  const int n_items = n_mtiles * units;
  const bool causal = a.causal != 0;

  if (threadIdx.x == 0) {
    mbar_init(sh.bar(B_QFULL), 1);
    mbar_init(sh.bar(B_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(sh.bar(B_KFULL + s), 1);
      mbar_init(sh.bar(B_VFULL + s), 1);
      mbar_init(sh.bar(B_KVEMPTY + s), 1);
      mbar_init(sh.bar(B_SFULL + s), 1);
      mbar_init(sh.bar(B_PFULL + s), 256);  // both warpgroups write P of every tile
    }
    mbar_init(sh.bar(B_ORDY), 1);
    mbar_init(sh.bar(B_EPI), 256);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot();

  if (warp == 8) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int kv_it = 0, it = 0;
      int last_kv = -1;  // last K/V tile issued (for the drain on error)
      bool ok = true;
      for (int i = sched(0); i < n_items && ok; ++it, i = sched(it)) {
        const Item w = item_of(i, units, a.h, n_mtiles, causal);
        const int g = (2 * w.p) / G;
        if (it > 0 && !wait_bar(sh, sh.bar(B_QEMPTY), (it - 1) & 1, a.status, 0x2001)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(sh.bar(B_QFULL), 2 * kNB * kBox);
        for (int hh = 0; hh < 2; ++hh)
          for (int box = 0; box < kNB; ++box)
            tma_load_4d(sh.base + kOffQ + (hh * kNB + box) * kBox, &tm_q, sh.bar(B_QFULL), box * 64,
                        2 * w.p + hh, w.mt * kBM, w.b);
        for (int j = 0; j < w.n_kv; ++j, ++kv_it) {
          const int st = kv_it & 1, use = kv_it >> 1;
          if (use > 0 && !wait_bar(sh, sh.bar(B_KVEMPTY + st), (use - 1) & 1, a.status, 0x2002)) {
            ok = false;
            break;
          }
          // (test hook: the first CTA leaves its first K tile unloaded, so
          // the MMA issuer's bounded wait for it expires)
          if (!(a.fault && blockIdx.x == 0 && kv_it == 0)) {
            mbar_arrive_expect_tx(sh.bar(B_KFULL + st), kNB * kBox);
            for (int box = 0; box < kNB; ++box)
              tma_load_4d(sh.base + kOffK + (st * kNB + box) * kBox, &tm_k, sh.bar(B_KFULL + st),
                          box * 64, g, j * kBN, w.b);
          }
          mbar_arrive_expect_tx(sh.bar(B_VFULL + st), kNB * kBox);
          for (int box = 0; box < kNB; ++box)
            tma_load_4d(sh.base + kOffV + (st * kNB + box) * kBox, &tm_v, sh.bar(B_VFULL + st),
                        box * 64, g, j * kBN, w.b);
          last_kv = kv_it;
        }
      }
      if (!ok && last_kv >= 0) {
        // drain: give the loads already issued (bounded) time to land
        for (int kv = last_kv; kv >= 0 && kv > last_kv - 2; --kv) {
          const uint32_t par = (kv >> 1) & 1;
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 200000000ull &&
                 !(mbar_try_wait(sh.bar(B_KFULL + (kv & 1)), par) &&
                   mbar_try_wait(sh.bar(B_VFULL + (kv & 1)), par))) {
          }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      int kv_it = 0, it = 0, pc = 0;
      bool ok = true;
      const uint32_t t_s[2] = {tmem + 0, tmem + 128};
      const uint32_t t_o[2] = {tmem + 256, tmem + 384};  // D <= 128 columns each
      auto issue_s = [&](int hh, int st) {
        const uint32_t qa = sh.base + kOffQ + hh * kNB * kBox;
        const uint32_t kb = sh.base + kOffK + st * kNB * kBox;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          tc_mma_ss(t_s[hh], sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                    kIdescS, kk > 0);
        }
      };
      auto issue_pv = [&](int hh, int st, bool acc) {
        const uint32_t vb = sh.base + kOffV + st * kNB * kBox;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // P of keys 0-63 in columns 0-31 of the S buffer, keys 64-127 in 64-95
          tc_mma_ts(t_o[hh], t_s[hh] + kk * 8 + (kk >= 4 ? 32 : 0), sdesc_sw128(vb + kk * 2048, kBox, 1024), kIdescPV,
                    (acc || kk > 0) ? 1u : 0u);
        }
      };
      for (int i = sched(0); i < n_items && ok; ++it, i = sched(it)) {
        const Item w = item_of(i, units, a.h, n_mtiles, causal);
        if (!wait_bar(sh, sh.bar(B_QFULL), it & 1, a.status, 0x2101)) { ok = false; break; }
        tc_fence_after();
        {
          const int st = kv_it & 1;
          if (!wait_bar(sh, sh.bar(B_KFULL + st), (kv_it >> 1) & 1, a.status, 0x2102)) { ok = false; break; }
          tc_fence_after();
          issue_s(0, st);
          tc_commit(sh.bar(B_SFULL + 0));
          issue_s(1, st);
          tc_commit(sh.bar(B_SFULL + 1));
          if (w.n_kv == 1) tc_commit(sh.bar(B_QEMPTY));
        }
        for (int j = 0; j < w.n_kv; ++j) {
          const int cur = kv_it + j, st = cur & 1;
          const int nxt = cur + 1, st2 = nxt & 1;
          const bool more = j + 1 < w.n_kv;
          if (!wait_bar(sh, sh.bar(B_PFULL + 0), pc & 1, a.status, 0x2103)) { ok = false; break; }
          if (!wait_bar(sh, sh.bar(B_VFULL + st), (cur >> 1) & 1, a.status, 0x2104)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, st, j > 0);
          if (more) {
            if (!wait_bar(sh, sh.bar(B_KFULL + st2), (nxt >> 1) & 1, a.status, 0x2105)) { ok = false; break; }
            tc_fence_after();
            issue_s(0, st2);
            tc_commit(sh.bar(B_SFULL + 0));
          }
          if (!wait_bar(sh, sh.bar(B_PFULL + 1), pc & 1, a.status, 0x2106)) { ok = false; break; }
          tc_fence_after();
          issue_pv(1, st, j > 0);
          tc_commit(sh.bar(B_KVEMPTY + st));
          if (more) {
            issue_s(1, st2);
            tc_commit(sh.bar(B_SFULL + 1));
            if (j + 2 == w.n_kv) tc_commit(sh.bar(B_QEMPTY));
          }
          ++pc;
        }
        if (!ok) break;
        tc_commit(sh.bar(B_ORDY));
        kv_it += w.n_kv;
      }
    }
  } else {
    // --------------------------------------------- softmax + epilogue -----
    // Both warpgroups work on every tile of both heads: warpgroup wg takes
    // key columns [64 wg, 64 wg + 64) of the tile (thread = query row = TMEM
    // lane), so a tile's exponentials run on eight warps and the head's next
    // P.V / S MMAs start sooner.  The two halves of a row share one running
    // max: exchanged on a row's first tile, and re-exchanged on the rare tile
    // whose sum overflows the stale-max guard in either half (a CTA-wide
    // barrier reduction decides).  Named barrier 1 (these 256 threads) is
    // reached by both warpgroups in the same sequence (it depends only on
    // the item, the tile and that reduction); every stop is decided by a
    // barrier reduction, so neither leaves while the other waits.
    const int wg = warp >> 2;             // key-column half of the tile
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;       // query row within the item = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    const int c0 = wg * 64;               // first key column of this half
    int it = 0, sc = 0, ec = 0;
    bool ok = true;
    // bounded 256-thread sync of the two softmax warpgroups
    auto epi_sync = [&](uint32_t site) -> bool {
      mbar_arrive(sh.bar(B_EPI));
      const bool r = wait_bar(sh, sh.bar(B_EPI), ec & 1, a.status, site);
      ++ec;
      return r;
    };
    float* xm = sh.xm();  // [head][half][row] half maxima
    for (int i = sched(0); i < n_items; ++it, i = sched(it)) {
      const Item w = item_of(i, units, a.h, n_mtiles, causal);
      float m_run[2] = {-INFINITY, -INFINITY}, l_half[2] = {0.f, 0.f};
      bool stop = false;
      for (int j = 0; j < w.n_kv && !stop; ++j, ++sc) {
        // masked columns: keys after the query (causal diagonal tile), or
        // keys >= N (ragged last tile without the causal mask)
        const bool masked = causal ? j == w.mt : (j == w.n_kv - 1 && (a.N % kBN) != 0);
        const int lim = causal ? row : a.N - 1 - j * kBN;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          // a failed wait does not leave here: the named-barrier sequence
          // below is the same for both warpgroups, and the stop is decided
          // together after the tile
          if (!wait_bar(sh, sh.bar(B_SFULL + hh), sc & 1, a.status, 0x2201 + hh)) ok = false;
          tc_fence_after();
          const uint32_t t_s = tmem + lane_off + hh * 128 + c0;
          uint32_t sv[64];
          tmem_ld32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
          tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
          tmem_ld_wait();
          if (j == 0) {
            const float hm = masked ? half_max<true>(sv, c0, lim) : half_max<false>(sv, c0, lim);
            xm[(hh * 2 + wg) * 128 + row] = hm;
            named_sync_256();
            m_run[hh] = fmaxf(hm, xm[(hh * 2 + (wg ^ 1)) * 128 + row]) * sl2;
            l_half[hh] = masked ? exp_half<true>(sv, c0, lim, sl2x2, m_run[hh], t_s)
                                : exp_half<false>(sv, c0, lim, sl2x2, m_run[hh], t_s);
          } else {
            float lsum = masked ? exp_half<true>(sv, c0, lim, sl2x2, m_run[hh], t_s)
                                : exp_half<false>(sv, c0, lim, sl2x2, m_run[hh], t_s);
            if (named_red_or_256(!(lsum <= kSumGuard))) {
              // rare: some row's half left the guard; both halves of every
              // row recompute against a max raised over this tile, and O is
              // rescaled (O is stable here: the commit that signalled S(j)
              // covers PV(j - 1))
              const float hm = masked ? half_max<true>(sv, c0, lim) : half_max<false>(sv, c0, lim);
              xm[(hh * 2 + wg) * 128 + row] = hm;
              named_sync_256();
              const float m_new = fmaxf(m_run[hh], fmaxf(hm, xm[(hh * 2 + (wg ^ 1)) * 128 + row]) * sl2);
              const float alpha = fast_exp2(m_run[hh] - m_new);
              m_run[hh] = m_new;
              lsum = masked ? exp_half<true>(sv, c0, lim, sl2x2, m_new, t_s)
                            : exp_half<false>(sv, c0, lim, sl2x2, m_new, t_s);
              l_half[hh] = l_half[hh] * alpha + lsum;
              if (__any_sync(0xffffffffu, alpha != 1.f)) {
                // this half's D / 2 columns of the head's O
                const uint32_t t_o = tmem + lane_off + 256 + hh * 128 + wg * (D / 2);
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                  uint32_t o[32];
                  tmem_ld32(t_o + c * 32, o);
                  tmem_ld_wait();
#pragma unroll
                  for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                  tmem_st32(t_o + c * 32, o);
                }
              }
            } else {
              l_half[hh] += lsum;
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(sh.bar(B_PFULL + hh));
        }
        stop = named_red_or_256(!ok || *sh.abort_flag());
      }
      if (stop) break;
      // ----------------------------------------------------- epilogue ----
      bool eok = wait_bar(sh, sh.bar(B_ORDY), it & 1, a.status, 0x2203);
      if (eok) {
        tc_fence_after();
        sh.lx()[(0 * 2 + wg) * 128 + row] = l_half[0];
        sh.lx()[(1 * 2 + wg) * 128 + row] = l_half[1];
        eok = epi_sync(0x2204);
      }
      if (eok) {
        const int n = w.mt * kBM + row;
        // l of each head: the two column halves' partial sums, in a fixed order
        const float le = sh.lx()[0 * 128 + row] + sh.lx()[1 * 128 + row];
        const float lo = sh.lx()[2 * 128 + row] + sh.lx()[3 * 128 + row];
        // each warpgroup writes half of the D features of the row
        constexpr int kHalf = D / 2, kNC = kHalf / 32;
        uint32_t oe[kNC][32], oo[kNC][32];
#pragma unroll
        for (int c = 0; c < kNC; ++c) {
          tmem_ld32(tmem + lane_off + 256 + wg * kHalf + c * 32, oe[c]);
          tmem_ld32(tmem + lane_off + 384 + wg * kHalf + c * 32, oo[c]);
        }
        tmem_ld_wait();
        if (n < a.N) {
          const float ie = 1.f / le;
          if (a.out.ptr) {
            const float gte = a.gate[(static_cast<int64_t>(w.b) * a.N + n) * a.h + w.p];
            const float io = gte / lo;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out.ptr) + w.b * a.out.sb +
                                 static_cast<int64_t>(n) * a.out.sn + w.p * a.out.sh + wg * kHalf;
            // both products rounded separately (no FMA contraction), so equal
            // even and odd outputs with gate 1 cancel exactly
            auto diff = [&](uint32_t xe, uint32_t xo) {
              return __fsub_rn(__fmul_rn(__uint_as_float(xe), ie), __fmul_rn(__uint_as_float(xo), io));
            };
#pragma unroll
            for (int c = 0; c < kNC; ++c) {
#pragma unroll
              for (int e = 0; e < 32; e += 8) {
                uint4 v;
                v.x = pack_bf16x2(diff(oe[c][e], oo[c][e]), diff(oe[c][e + 1], oo[c][e + 1]));
                v.y = pack_bf16x2(diff(oe[c][e + 2], oo[c][e + 2]), diff(oe[c][e + 3], oo[c][e + 3]));
                v.z = pack_bf16x2(diff(oe[c][e + 4], oo[c][e + 4]), diff(oe[c][e + 5], oo[c][e + 5]));
                v.w = pack_bf16x2(diff(oe[c][e + 6], oo[c][e + 6]), diff(oe[c][e + 7], oo[c][e + 7]));
                *reinterpret_cast<uint4*>(dst + c * 32 + e) = v;
              }
            }
          }
          if (a.o_heads.ptr) {
            // the saves for the backward: each head's normalised output
            const float inv_o = 1.f / lo;
            __nv_bfloat16* he = static_cast<__nv_bfloat16*>(a.o_heads.ptr) + w.b * a.o_heads.sb +
                                static_cast<int64_t>(n) * a.o_heads.sn + 2 * w.p * a.o_heads.sh + wg * kHalf;
            __nv_bfloat16* ho = he + a.o_heads.sh;
#pragma unroll
            for (int c = 0; c < kNC; ++c) {
#pragma unroll
              for (int e = 0; e < 32; e += 8) {
                uint4 ve, vo;
                ve.x = pack_bf16x2(__uint_as_float(oe[c][e]) * ie, __uint_as_float(oe[c][e + 1]) * ie);
                ve.y = pack_bf16x2(__uint_as_float(oe[c][e + 2]) * ie, __uint_as_float(oe[c][e + 3]) * ie);
                ve.z = pack_bf16x2(__uint_as_float(oe[c][e + 4]) * ie, __uint_as_float(oe[c][e + 5]) * ie);
                ve.w = pack_bf16x2(__uint_as_float(oe[c][e + 6]) * ie, __uint_as_float(oe[c][e + 7]) * ie);
                vo.x = pack_bf16x2(__uint_as_float(oo[c][e]) * inv_o, __uint_as_float(oo[c][e + 1]) * inv_o);
                vo.y = pack_bf16x2(__uint_as_float(oo[c][e + 2]) * inv_o, __uint_as_float(oo[c][e + 3]) * inv_o);
                vo.z = pack_bf16x2(__uint_as_float(oo[c][e + 4]) * inv_o, __uint_as_float(oo[c][e + 5]) * inv_o);
                vo.w = pack_bf16x2(__uint_as_float(oo[c][e + 6]) * inv_o, __uint_as_float(oo[c][e + 7]) * inv_o);
                *reinterpret_cast<uint4*>(he + c * 32 + e) = ve;
                *reinterpret_cast<uint4*>(ho + c * 32 + e) = vo;
              }
            }
          }
          if (a.lse) {
            // natural-log LSE of head 2p + wg: (m + log2 l) * ln 2
            a.lse[(static_cast<int64_t>(w.b) * 2 * a.h + 2 * w.p + wg) * a.N + n] =
                (m_run[wg] + __log2f(wg == 0 ? le : lo)) * 0.69314718055994531f;
          }
        }

        tc_fence_before();
        eok = epi_sync(0x2205);
      }
      if (!eok) ok = false;
      if (named_red_or_256(!ok || *sh.abort_flag())) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

template <int D>
cudaError_t launch_d(const V2FwdArgs& a, cudaStream_t s) {
  CUtensorMap tq, tk, tv;
  if (!encode_tmap_bf16_4d(&tq, a.q, a.B, a.N, 2 * a.h, D, kBM)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16_4d(&tk, a.k, a.B, a.N, a.h_kv, D, kBN)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16_4d(&tv, a.v, a.B, a.N, a.h_kv, D, kBN)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(v2_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_items = ((a.N + kBM - 1) / kBM) * a.B * a.h;
  int grid = a.num_sms > 0 ? a.num_sms : 148;
  if (grid > n_items) grid = n_items;
  if (grid <= 0) return cudaSuccess;
  v2_fwd_kernel<D><<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_v2_fwd(const V2FwdArgs& a, cudaStream_t s) {
  if (a.d == 128) return launch_d<128>(a, s);
  if (a.d == 64) return launch_d<64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace da
