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

// Visible keys of one 64-key tile as bits, for a row that sees keys
// [lo, lo + span): bit i of w0 is key key0 + i, bit i of w1 key key0 + 32 + i.
// One bit test per score then replaces the add, compare and select that a
// range test takes per score.
__device__ __forceinline__ void visible_bits(int key0, int lo, unsigned span, uint32_t& w0,
                                             uint32_t& w1) {
  const int a = min(max(lo - key0, 0), 64);
  const int b = max(min(lo + (int)span - key0, 64), a);
  auto range32 = [](int x, int y) -> uint32_t {   // bits [x, y), 0 <= x <= y <= 32
    const uint32_t below_y = y >= 32 ? 0xffffffffu : ((1u << y) - 1u);
    const uint32_t below_x = x >= 32 ? 0xffffffffu : ((1u << x) - 1u);
    return below_y & ~below_x;
  };
  w0 = range32(min(a, 32), min(b, 32));
  w1 = range32(max(a - 32, 0), max(b - 32, 0));
}

// p = exp2(s * sl2 - m) for the 64 scores of one row (ra: keys key0 .. key0+31,
// rb: key0+32 .. key0+63), packed two per 32-bit TMEM column into the 32 columns
// at p_tm (16 per tcgen05.st; the caller waits for the stores); returns the
// (even-key, odd-key) partial sums of p.  MASKED: keys whose bit in (w0, w1) is
// clear give p = 0 -- needed only when the scale is 0 (the masked scores are
// -inf already, and -inf * 0 would give NaN).
template <bool MASKED, bool F16>
__device__ __forceinline__ float2 exp_tile(const uint32_t* ra, const uint32_t* rb, float sl2,
                                           float neg_m, uint32_t w0, uint32_t w1,
                                           uint32_t p_tm) {
  const float2 sc = make_float2(sl2, sl2), nm = make_float2(neg_m, neg_m);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t* r = half ? rb : ra;
    const uint32_t w = half ? w1 : w0;
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 x = __ffma2_rn(
          make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc, nm);
      float2 p = make_float2(ex2(x.x), ex2(x.y));
      if constexpr (MASKED) {
        if (!(w & (1u << (2 * i)))) p.x = 0.f;
        if (!(w & (1u << (2 * i + 1)))) p.y = 0.f;
      }
      if (i & 1) acc1 = __fadd2_rn(acc1, p);
      else acc0 = __fadd2_rn(acc0, p);
      pk[i] = pack2<F16>(p.x, p.y);
    }
    tmem_st16(p_tm + 16u * (uint32_t)half, pk);
  }
  return __fadd2_rn(acc0, acc1);
}

// Sets the scores of keys whose bit in (w0, w1) is clear to -inf (ra: keys
// key0 .. key0+31, rb: key0+32 .. key0+63; see visible_bits).
__device__ __forceinline__ void mask_scores64(uint32_t* ra, uint32_t* rb, uint32_t w0,
                                              uint32_t w1) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (!(w0 & (1u << i))) ra[i] = __float_as_uint(neg_inf());
    if (!(w1 & (1u << i))) rb[i] = __float_as_uint(neg_inf());
  }
}

}  // namespace dev
}  // namespace pka
