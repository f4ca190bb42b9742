// Device helpers for sm_103a: mbarriers with bounded waits, TMA tensor loads,
// ldmatrix / mma.sync fragments, packed fp32 math, bf16 unpacking.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pka.h"
#include "plan.h"

namespace pka {
namespace dev {

constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- time ----------------------------------------------------------------
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound on any single wait: a wait that has not completed after this
// long records STATUS_WAIT_TIMEOUT and gives up (no trap, no endless spin).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of the barrier to complete.  Gives up after
// limit_ns, OR-ing STATUS_WAIT_TIMEOUT into *status; returns false then.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, int32_t* status,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      if (status) atomicOr(status, STATUS_WAIT_TIMEOUT);
      return false;
    }
  }
}

// Every kernel's wait: mbar_wait_for with the kWaitLimitNs bound.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status) {
  return mbar_wait_for(bar, parity, status, kWaitLimitNs);
}

// ---- TMA -------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 5-D tiled load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3,
                                            int32_t c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
      : "memory");
}

// Loads one 16-token unit of an HND K or V pool (map from encode_kv_pool_map)
// into 4 KB at dst: two 2 KB halves (dims 0-63, then 64-127), each 16 rows of
// 128 bytes with 128-byte swizzle.  One copy instruction per unit: the
// issuing thread's cost is per instruction, not per byte.
__device__ __forceinline__ void tma_load_kv_unit(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int32_t slot, int32_t head,
                                                 int32_t page) {
  tma_load_5d(dst, map, bar, 0, slot, 0, head, page);
}

// The K and V units of one 16-token unit (as tma_load_kv_unit) for a converged
// warp: one elected lane arms `bar` for `bytes` and issues both copies from one
// asm block.  Issued from a divergent lane as three separate statements the
// same work costs the warp ~1.5x the cycles (~340 against ~225 per unit).
__device__ __forceinline__ void tma_load_kv_pair_elect(uint32_t dst_k, uint32_t dst_v,
                                                       const CUtensorMap* map_k,
                                                       const CUtensorMap* map_v, uint32_t bar,
                                                       uint32_t bytes, int32_t slot, int32_t head,
                                                       int32_t page) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%4], %5;\n\t"
      "@e cp.async.bulk.tensor.5d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%2, {%6, %7, %6, %8, %9}], [%4];\n\t"
      "@e cp.async.bulk.tensor.5d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%1], [%3, {%6, %7, %6, %8, %9}], [%4];\n\t}" ::"r"(dst_k),
      "r"(dst_v), "l"(reinterpret_cast<uint64_t>(map_k)), "l"(reinterpret_cast<uint64_t>(map_v)),
      "r"(bar), "r"(bytes), "r"(0), "r"(slot), "r"(head), "r"(page)
      : "memory");
}

// Contiguous bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// 3-D tiled load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// ---- 128-byte swizzle --------------------------------------------------------
// A TMA box with 128-byte rows and CU_TENSOR_MAP_SWIZZLE_128B stores 16-byte
// chunk c of row r at chunk position c ^ (r & 7), inside 1024-byte aligned
// groups of eight rows.  Byte offset of (row, chunk) inside such a box:
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// ---- bf16 ------------------------------------------------------------------
// Two bf16 packed in a 32-bit word -> two floats (exact: bf16 is the upper
// half of a float32).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  float2 r;
  r.x = __uint_as_float(w << 16);
  r.y = __uint_as_float(w & 0xffff0000u);
  return r;
}

__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---- the two 16-bit input formats (F16 = false: bf16, true: IEEE half) ------
template <bool F16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (F16) {
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
  } else {
    return bf16x2_to_float2(w);
  }
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    const __half2 h = __floats2half2_rn(lo, hi);
    uint32_t w;
    memcpy(&w, &h, 4);
    return w;
  } else {
    return float2_to_bf16x2(lo, hi);
  }
}

// ---- outputs: PKA_DTYPE_BF16, PKA_DTYPE_F16 or PKA_DTYPE_F32 ------------------
// v[0..N) * sc to N consecutive elements at element offset `off` of `out`
// (N = 4, 8 or 16; off a multiple of 4, so every store is 8- or 16-byte aligned).
template <int N>
__device__ __forceinline__ void store_out(void* out, int64_t off, const float* v, float sc,
                                          int dtype) {
  static_assert(N == 4 || N == 8 || N == 16, "4, 8 or 16 values");
  if (dtype == PKA_DTYPE_F32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(out) + off);
#pragma unroll
    for (int x = 0; x < N / 4; ++x)
      d[x] = make_float4(v[4 * x] * sc, v[4 * x + 1] * sc, v[4 * x + 2] * sc, v[4 * x + 3] * sc);
    return;
  }
  uint32_t w[N / 2];
#pragma unroll
  for (int x = 0; x < N / 2; ++x)
    w[x] = dtype == PKA_DTYPE_F16 ? pack2<true>(v[2 * x] * sc, v[2 * x + 1] * sc)
                                  : pack2<false>(v[2 * x] * sc, v[2 * x + 1] * sc);
  uint16_t* base = static_cast<uint16_t*>(out) + off;
  if constexpr (N == 4) {
    *reinterpret_cast<uint2*>(base) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int x = 0; x < N / 8; ++x)
      reinterpret_cast<uint4*>(base)[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
  }
}

// One value to element `off` of `out`.
__device__ __forceinline__ void store_out1(void* out, int64_t off, float v, int dtype) {
  if (dtype == PKA_DTYPE_F32) {
    static_cast<float*>(out)[off] = v;
  } else if (dtype == PKA_DTYPE_F16) {
    static_cast<__half*>(out)[off] = __float2half_rn(v);
  } else {
    static_cast<__nv_bfloat16*>(out)[off] = __float2bfloat16_rn(v);
  }
}

// ---- fast exp2 (hardware MUFU.EX2) -------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- packed fp32 -------------------------------------------------------------
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// ---- ldmatrix / mma.sync -----------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transposes an 8x8 matrix of 16-bit elements held one 32-bit word per lane
// (lane 4r + c holds row r, columns 2c and 2c + 1): afterwards lane 4r + c
// holds row r, columns 2c and 2c + 1 of the transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// As mma_bf16_16816 with IEEE half A and B.
__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <bool F16>
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (F16)
    mma_f16_16816(d, a, b0, b1);
  else
    mma_bf16_16816(d, a, b0, b1);
}

}  // namespace dev
}  // namespace pka
