// grouped.cu — the combination step of grouped differential attention.
//
// "Differential Transformer | ICLR 2025 Oral" (dainus.ai), "같은 문제, 다른
// 접근": a follow-up gives signal-extracting heads and noise-controlling heads
// an uneven share, 3:1 or 4:1.  Read in the V2 form ("Differential Transformer
// V2", pogovet.com, §1): query heads come in groups of `ratio` signal heads
// followed by one noise head (all in one K/V group), and
//   out[t, g r + i] = O[t, g (r+1) + i] - gate[t, g r + i] * O[t, g (r+1) + r].
// The per-head outputs O come from the V2 attention kernel run without its
// pair combination (a group spans more heads than a pair, and one SM's TMEM
// holds two heads' scores and accumulators); this HBM-bound kernel then reads
// each signal row and its group's noise row once per output and writes out.
#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

// One CTA per token (b, n): its threads walk the token's h * d / 8 groups of
// 8 features (output head p, features c8 .. c8 + 7), so the token's per-head
// row block is read with coalesced 16-byte loads (each noise row serves its
// `ratio` signal rows from L1) and the index arithmetic is per token.
__global__ void __launch_bounds__(256)
grouped_combine_kernel(GroupedArgs a) {
  const int nc = a.d / 8;
  const int work = a.h * nc;
  for (long long tok = blockIdx.x; tok < static_cast<long long>(a.B) * a.N; tok += gridDim.x) {
    const int n = static_cast<int>(tok % a.N), b = static_cast<int>(tok / a.N);
    const __nv_bfloat16* base = static_cast<const __nv_bfloat16*>(a.o_heads.ptr) + b * a.o_heads.sb +
                                static_cast<int64_t>(n) * a.o_heads.sn;
    const float* gt_row = a.gate + tok * a.h;
    __nv_bfloat16* dst_row = static_cast<__nv_bfloat16*>(a.out.ptr) + b * a.out.sb +
                             static_cast<int64_t>(n) * a.out.sn;
    for (int idx = threadIdx.x; idx < work; idx += blockDim.x) {
      const int p = idx / nc, c8 = (idx - p * nc) * 8;
      const int g = p / a.ratio, i = p - g * a.ratio;
      const uint4 sv =
          *reinterpret_cast<const uint4*>(base + static_cast<int64_t>(g * (a.ratio + 1) + i) * a.o_heads.sh + c8);
      const uint4 nv = *reinterpret_cast<const uint4*>(
          base + static_cast<int64_t>(g * (a.ratio + 1) + a.ratio) * a.o_heads.sh + c8);
      const float gt = gt_row[p];
      const __nv_bfloat162* s2 = reinterpret_cast<const __nv_bfloat162*>(&sv);
      const __nv_bfloat162* n2 = reinterpret_cast<const __nv_bfloat162*>(&nv);
      uint32_t r[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // both terms rounded on their own: equal signal and noise rows with
        // gate 1 give exactly zero
        const float lo = __fsub_rn(__low2float(s2[e]), __fmul_rn(gt, __low2float(n2[e])));
        const float hi = __fsub_rn(__high2float(s2[e]), __fmul_rn(gt, __high2float(n2[e])));
        r[e] = pack_bf16x2(lo, hi);
      }
      *reinterpret_cast<uint4*>(dst_row + static_cast<int64_t>(p) * a.out.sh + c8) = make_uint4(r[0], r[1], r[2], r[3]);
    }
  }
}

}  // namespace

cudaError_t launch_grouped_combine(const GroupedArgs& a, cudaStream_t s) {
  const long long tokens = static_cast<long long>(a.B) * a.N;
  long long grid = tokens;
  if (grid > 64 * 152) grid = 64 * 152;
  if (grid < 1) grid = 1;
  grouped_combine_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace da
