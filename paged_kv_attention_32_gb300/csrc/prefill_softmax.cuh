// Softmax pieces shared by the prefill kernels (one thread per query row, 64
// scores of one key tile per call).
#pragma once

#include <cstdint>

#include "device_common.cuh"
#include "tcgen05.cuh"

namespace pka {
namespace dev {

// Bounded mbarrier wait taken by the whole warp; true on every lane iff every
// lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int32_t* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// Row max of 64 scores (ra: keys 0-31, rb: keys 32-63) as four independent
// chains, so that the scheduler has short dependency chains to interleave.
__device__ __forceinline__ float row_max64(const uint32_t* ra, const uint32_t* rb) {
  float mq[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
#pragma unroll
  for (int i = 0; i < 32; ++i)
    mq[i & 3] = fmax3(mq[i & 3], __uint_as_float(ra[i]), __uint_as_float(rb[i]));
  return fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
}

// p = exp2(s * sl2 - m) for the 64 scores of one row (ra: keys key0 .. key0+31,
// rb: key0+32 .. key0+63), packed two per 32-bit TMEM column into the 32 columns
// at p_tm (16 per tcgen05.st; the caller waits for the stores); returns the
// (even-key, odd-key) partial sums of p.  MASKED: keys outside [lo, lo + span)
// give p = 0 (their scores were already set to -inf for the row max; p is zeroed
// again because -inf * 0 or -inf + inf would give NaN).
template <bool MASKED, bool F16>
__device__ __forceinline__ float2 exp_tile(const uint32_t* ra, const uint32_t* rb, float sl2,
                                           float neg_m, int key0, int lo, unsigned span,
                                           uint32_t p_tm) {
  const float2 sc = make_float2(sl2, sl2), nm = make_float2(neg_m, neg_m);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t* r = half ? rb : ra;
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 x = __ffma2_rn(
          make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc, nm);
      float2 p = make_float2(ex2(x.x), ex2(x.y));
      if constexpr (MASKED) {
        if ((unsigned)(key0 + 32 * half + 2 * i - lo) >= span) p.x = 0.f;
        if ((unsigned)(key0 + 32 * half + 2 * i + 1 - lo) >= span) p.y = 0.f;
      }
      if (i & 1) acc1 = __fadd2_rn(acc1, p);
      else acc0 = __fadd2_rn(acc0, p);
      pk[i] = pack2<F16>(p.x, p.y);
    }
    tmem_st16(p_tm + 16u * (uint32_t)half, pk);
  }
  return __fadd2_rn(acc0, acc1);
}

// Sets the scores of keys outside [lo, lo + span) to -inf (ra: key0 .. key0+31,
// rb: key0+32 .. key0+63).
__device__ __forceinline__ void mask_scores64(uint32_t* ra, uint32_t* rb, int key0, int lo,
                                              unsigned span) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if ((unsigned)(key0 + i - lo) >= span) ra[i] = __float_as_uint(neg_inf());
    if ((unsigned)(key0 + 32 + i - lo) >= span) rb[i] = __float_as_uint(neg_inf());
  }
}

}  // namespace dev
}  // namespace pka
