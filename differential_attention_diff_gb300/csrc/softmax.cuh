// softmax.cuh — the per-row, per-tile online softmax shared by the tcgen05
// attention kernels (thread = query row = TMEM lane, 128 keys per tile).
//
// For a row of 128 fp32 scores S (in TMEM) it writes P = exp2(S*scale*log2e
// - m) as bf16 pairs into the first 64 columns of the same TMEM region (the A
// operand of the P.V MMA) and keeps the running max m and sum l.
//
// Instruction economy (the softmax warps are issue-bound, not exp-bound):
//  * the row max is taken only on the first tile of a row; later tiles reuse
//    that (stale) max and only check that the tile's sum stays finite and
//    below 2^64 — bf16 P and the fp32 accumulators keep full relative
//    precision for any magnitude below that, and the common case then skips
//    the 127 max operations per tile;  when the guard trips (scores far
//    above every earlier one) the warp recomputes the tile against the new
//    max and reports the rescale factor for O and l;
//  * masking (key > query) only on the diagonal tile, or (not causal) only
//    on a ragged last key tile (key >= N);
//  * scale-and-subtract and the row sum use packed f32x2 FMA / add;
//  * the score chunks are loaded from TMEM in two halves so that the second
//    half's load overlaps the first half's exponentials.
#pragma once

#include "tma.cuh"

namespace da {

constexpr float kSumGuard = 18446744073709551616.0f;  // 2^64

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) |
         (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// exp2 of 32 scores (one TMEM chunk starting at key col0) against max m
// (negm2 = {-m, -m}), columns past lim zeroed when kMask; writes 16 bf16x2
// words to TMEM at t_p; returns the pairwise partial sums.
template <bool kMask>
__device__ __forceinline__ uint64_t exp_chunk(const uint32_t* s, int col0, int lim, uint64_t sl2x2,
                                              uint64_t negm2, uint32_t t_p) {
  uint32_t pk[16];
  uint64_t acc = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint64_t x = fma_f32x2(static_cast<uint64_t>(s[2 * e]) |
                                     (static_cast<uint64_t>(s[2 * e + 1]) << 32),
                                 sl2x2, negm2);
    float p0 = fast_exp2(f2_lo(x));
    float p1 = fast_exp2(f2_hi(x));
    if (kMask) {
      if (col0 + 2 * e > lim) p0 = 0.f;
      if (col0 + 2 * e + 1 > lim) p1 = 0.f;
    }
    acc = add_f32x2(acc, f2(p0, p1));
    pk[e] = pack_bf16x2(p0, p1);
  }
  tmem_st16(t_p, pk);
  return acc;
}

template <bool kMask>
__device__ __forceinline__ float exp_row(const uint32_t (&s)[128], int lim, uint64_t sl2x2,
                                         float m, uint32_t t_s) {
  const uint64_t negm2 = f2(-m, -m);
  uint64_t a0 = exp_chunk<kMask>(s, 0, lim, sl2x2, negm2, t_s);
  uint64_t a1 = exp_chunk<kMask>(s + 32, 32, lim, sl2x2, negm2, t_s + 16);
  uint64_t a2 = exp_chunk<kMask>(s + 64, 64, lim, sl2x2, negm2, t_s + 32);
  uint64_t a3 = exp_chunk<kMask>(s + 96, 96, lim, sl2x2, negm2, t_s + 48);
  const uint64_t t = add_f32x2(add_f32x2(a0, a1), add_f32x2(a2, a3));
  return f2_lo(t) + f2_hi(t);
}

template <bool kMask>
__device__ __forceinline__ float row_max(const uint32_t (&s)[128], int lim) {
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < 128; ++e) {
    const float v = __uint_as_float(s[e]);
    if (!kMask || e <= lim) mx = fmaxf(mx, v);
  }
  return mx;
}

// One tile of one row.  t_s: TMEM address of the row's 128 scores (lane
// offset included).  With `masked`, key columns past `lim` are excluded: lim
// is the query row within the tile on a causal diagonal tile, or the last
// valid key column of a ragged final tile when attention is not causal.
// Updates (m_run, l_run); returns the factor the row's O accumulator must be
// multiplied by before the next P.V (1 = unchanged; the first tile returns 0:
// O has no content yet).  Warp-uniform control flow: `first` and `masked` are
// the same for the whole warp.
__device__ __forceinline__ float softmax_tile(uint32_t t_s, int lim, bool first, bool masked,
                                              float sl2, float& m_run, float& l_run) {
  uint32_t s[128];
  const uint64_t sl2x2 = f2(sl2, sl2);
  if (first) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
    tmem_ld_wait();
    const float mx = masked ? row_max<true>(s, lim) : row_max<false>(s, lim);
    m_run = mx * sl2;
    l_run = masked ? exp_row<true>(s, lim, sl2x2, m_run, t_s) : exp_row<false>(s, lim, sl2x2, m_run, t_s);
    return 0.f;
  }
  // two-phase load: chunks 0-1, then 2-3 in flight while 0-1 are processed
  tmem_ld32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
  tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
  tmem_ld_wait();
  tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
  tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
  const uint64_t negm2 = f2(-m_run, -m_run);
  uint64_t a0, a1, a2, a3;
  if (masked) {
    a0 = exp_chunk<true>(s, 0, lim, sl2x2, negm2, t_s);
    a1 = exp_chunk<true>(s + 32, 32, lim, sl2x2, negm2, t_s + 16);
    tmem_ld_wait();
    a2 = exp_chunk<true>(s + 64, 64, lim, sl2x2, negm2, t_s + 32);
    a3 = exp_chunk<true>(s + 96, 96, lim, sl2x2, negm2, t_s + 48);
  } else {
    a0 = exp_chunk<false>(s, 0, lim, sl2x2, negm2, t_s);
    a1 = exp_chunk<false>(s + 32, 32, lim, sl2x2, negm2, t_s + 16);
    tmem_ld_wait();
    a2 = exp_chunk<false>(s + 64, 64, lim, sl2x2, negm2, t_s + 32);
    a3 = exp_chunk<false>(s + 96, 96, lim, sl2x2, negm2, t_s + 48);
  }
  const uint64_t t = add_f32x2(add_f32x2(a0, a1), add_f32x2(a2, a3));
  float lsum = f2_lo(t) + f2_hi(t);
  const bool over = !(lsum <= kSumGuard);
  if (__any_sync(0xffffffffu, over)) {
    // rare: recompute the tile against a raised max (whole warp, since the
    // TMEM stores are warp-collective; rows that did not trip keep theirs)
    float m_new = m_run;
    if (over) m_new = fmaxf(m_run, (masked ? row_max<true>(s, lim) : row_max<false>(s, lim)) * sl2);
    const float alpha = fast_exp2(m_run - m_new);
    m_run = m_new;
    lsum = masked ? exp_row<true>(s, lim, sl2x2, m_run, t_s) : exp_row<false>(s, lim, sl2x2, m_run, t_s);
    l_run = l_run * alpha + lsum;
    return alpha;
  }
  l_run += lsum;
  return 1.f;
}

// ---- the softmax of one half row (64 key columns) --------------------------
// Max over the valid columns of this half (key column c0 + e <= lim when
// masked; -inf when none is valid).
template <bool kMask>
__device__ __forceinline__ float half_max(const uint32_t (&s)[64], int c0, int lim) {
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < 64; ++e)
    if (!kMask || c0 + e <= lim) mx = fmaxf(mx, __uint_as_float(s[e]));
  return mx;
}
// The same over 32 scores starting at key column c0, folded into mx.
template <bool kMask>
__device__ __forceinline__ float chunk_max(const uint32_t (&s)[32], int c0, int lim, float mx) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (!kMask || c0 + e <= lim) mx = fmaxf(mx, __uint_as_float(s[e]));
  return mx;
}
// exp2(S scale log2e - m) of the 64 scores, written as bf16 pairs over the
// first 32 of those columns (t_p); returns their sum.
template <bool kMask>
__device__ __forceinline__ float exp_half(const uint32_t (&s)[64], int c0, int lim, uint64_t sl2x2,
                                          float m, uint32_t t_p) {
  const uint64_t negm2 = f2(-m, -m);
  const uint64_t a0 = exp_chunk<kMask>(s, c0, lim, sl2x2, negm2, t_p);
  const uint64_t a1 = exp_chunk<kMask>(s + 32, c0 + 32, lim, sl2x2, negm2, t_p + 16);
  const uint64_t t = add_f32x2(a0, a1);
  return f2_lo(t) + f2_hi(t);
}
// Named barrier 1 over 256 softmax threads (warps 0-7, two warpgroups that
// split each tile's key columns): a plain sync, and a sync that returns
// whether any of them passed `pred`.
__device__ __forceinline__ void named_sync_256() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}
__device__ __forceinline__ bool named_red_or_256(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

}  // namespace da
