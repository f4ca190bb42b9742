// Ragged causal prefill on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// batch_prefill (packed qo_indptr / kv_indptr): for every request and query
// head, O = softmax(sm_scale * Q K^T + causal mask) V * output_scale, with the
// causal diagonal bottom-right aligned (row i sees keys 0 .. Lk - Lq + i) and
// an optional left window (window_left = W >= 0: keys from Lk - Lq + i - W on),
// or, for fixed-shape batches, per-row inclusive bounds (variable_window).
//
// One CTA = one 128-row query tile of one request for two query heads that
// share a KV head (GQA), so every K/V tile loaded serves both heads.
//   warp 8      TMA producer: Q tiles once, then K and V tiles of 128 keys
//               (two stages each), 128-byte swizzled, completing on mbarriers;
//   warp 9      allocates 512 TMEM columns and issues every tcgen05.mma from
//               one thread: S_h = Q_h K^T (M=128, N=128, K=128) into TMEM,
//               O_h += P_h V with P_h read from TMEM and V (MN-major) from
//               shared memory; the two heads ping-pong so the tensor core
//               works on one head while the softmax of the other runs;
//   warps 0-3   softmax of head 0, warps 4-7 softmax of head 1: one thread
//               per query row (TMEM lane), two passes over S in TMEM (row
//               max of the raw scores, then p = exp2(s*scale*log2e - m) as one
//               FFMA + MUFU, row sum, bf16 P written back over the first 64
//               columns of S), lazy rescaling of O in TMEM only when the row
//               max grew by more than 2^8, final O / l and base-2 LSE.
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512); P_h
// occupies columns [0,64) of S_h (two bf16 per column).
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "host_common.h"
#include "prefill.h"
#include "tcgen05.cuh"

namespace pka {

using namespace dev;

namespace {

constexpr int kTile = 128;
constexpr uint32_t kBox = 16384;            // 128 rows x 128 bytes
constexpr uint32_t kOffQ = 0;               // 2 heads x 32 KB
constexpr uint32_t kOffK = 65536;           // 2 stages x 32 KB
constexpr uint32_t kOffV = 131072;          // 2 stages x 32 KB
constexpr uint32_t kOffBar = 196608;
constexpr size_t kSmemBytes = 1024 + kOffBar + 256;
constexpr int kThreads = 320;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when the max grows by > 2^8

constexpr uint32_t kColS = 0, kColO = 256;

enum {
  B_Q = 0, B_KFULL = 1, B_KEMPTY = 3, B_VFULL = 5, B_VEMPTY = 7, B_SFULL = 9, B_PFULL = 11,
  B_ODONE = 13, B_MMADONE = 15, B_COUNT = 16
};

// A, B K-major (QK) / A K-major, B = V MN-major (PV); operands bf16 or f16
template <bool F16> constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0, F16);
template <bool F16> constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1, F16);

// K-major operand of 128 rows x 128 columns stored as two 16 KB boxes of
// 64 columns: descriptor for k-step kk (16 columns).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return smem_desc_sw128(base + (uint32_t)(kk >> 2) * kBox + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
}
// V tile (keys x D) as the MN-major B operand: k-step kk covers keys 16kk..16kk+15.
__device__ __forceinline__ uint64_t vmn_desc(uint32_t base, int kk) {
  return smem_desc_sw128(base + (uint32_t)kk * 2048u, kBox, 1024u);
}

// A bounded wait whose outcome is the same for every lane of the warp (the
// warp-collective tcgen05.ld/st that follow must not diverge).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int32_t* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// F16: q/K/V (and P) are IEEE half, else bf16.
template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmq,
               const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + B_COUNT * 8);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PrefillTile tile = a.tiles[blockIdx.x];
  const int b = tile.request, h0 = tile.head, mt = tile.q_tile, n_kv = tile.n_kv;
  const int kv0 = tile.kv0;
  const int q0 = a.qo_indptr[b], Lq = a.qo_indptr[b + 1] - q0;
  const int k0 = a.kv_indptr[b], Lk = a.kv_indptr[b + 1] - k0;
  const int nh = a.heads_per_cta;
  const int hk = h0 / a.group;

  if (tid == 0) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), 128);
      mbar_init(bar(B_ODONE + s), 1);
    }
    mbar_init(bar(B_MMADONE), 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      const int qrow = q0 + mt * kTile;
      mbar_arrive_expect_tx(bar(B_Q), (uint32_t)nh * 2u * kBox);
      for (int hh = 0; hh < nh; ++hh)
        for (int half = 0; half < 2; ++half)
          tma_load_3d(sbase + kOffQ + (uint32_t)(hh * 2 + half) * kBox, &tmq, bar(B_Q), half * 64,
                      h0 + hh, qrow);
      int last_k = -1, last_v = -1;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int st = j & 1;
        if (j >= 2) ok = mbar_wait(bar(B_KEMPTY + st), (uint32_t)(((j >> 1) - 1) & 1), a.status);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(B_KFULL + st), 2u * kBox);
        for (int half = 0; half < 2; ++half)
          tma_load_3d(sbase + kOffK + (uint32_t)(st * 2 + half) * kBox, &tmk, bar(B_KFULL + st),
                      half * 64, hk, k0 + (kv0 + j) * kTile);
        last_k = j;
        if (j >= 2) ok = mbar_wait(bar(B_VEMPTY + st), (uint32_t)(((j >> 1) - 1) & 1), a.status);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(B_VFULL + st), 2u * kBox);
        for (int half = 0; half < 2; ++half)
          tma_load_3d(sbase + kOffV + (uint32_t)(st * 2 + half) * kBox, &tmv, bar(B_VFULL + st),
                      half * 64, hk, k0 + (kv0 + j) * kTile);
        last_v = j;
      }
      if (!ok) {   // give the copies already issued a bounded chance to land
        mbar_wait(bar(B_Q), 0, nullptr);
        if (last_k >= 0) mbar_wait(bar(B_KFULL + (last_k & 1)), (uint32_t)((last_k >> 1) & 1), nullptr);
        if (last_v >= 0) mbar_wait(bar(B_VFULL + (last_v & 1)), (uint32_t)((last_v >> 1) & 1), nullptr);
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (one thread) ----------------
    if (lane == 0) {
      auto issue_qk = [&](int hh, int st) {
        const uint32_t d = tmem + kColS + (uint32_t)hh * 128u;
        const uint32_t qb = sbase + kOffQ + (uint32_t)hh * 2u * kBox;
        const uint32_t kb = sbase + kOffK + (uint32_t)st * 2u * kBox;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(d, kmajor_desc(qb, kk), kmajor_desc(kb, kk), kIdescQK<F16>, kk > 0 ? 1u : 0u);
      };
      bool ok = mbar_wait(bar(B_Q), 0, a.status) && mbar_wait(bar(B_KFULL), 0, a.status);
      if (ok) {
        tc_fence_after();
        for (int hh = 0; hh < nh; ++hh) {
          issue_qk(hh, 0);
          umma_commit(bar(B_SFULL + hh));
        }
        umma_commit(bar(B_KEMPTY));
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int vst = j & 1;
        ok = mbar_wait(bar(B_VFULL + vst), (uint32_t)((j >> 1) & 1), a.status);
        for (int hh = 0; ok && hh < nh; ++hh) {
          ok = mbar_wait(bar(B_PFULL + hh), (uint32_t)(j & 1), a.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + kColO + (uint32_t)hh * 128u;
          const uint32_t p_tm = tmem + kColS + (uint32_t)hh * 128u;   // P: 64 columns, lanes 0-127
          const uint32_t vb = sbase + kOffV + (uint32_t)vst * 2u * kBox;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16_ts(d, p_tm + (uint32_t)kk * 8u, vmn_desc(vb, kk), kIdescPV<F16>,
                         (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(B_ODONE + hh));
          if (hh == nh - 1) umma_commit(bar(B_VEMPTY + vst));
          if (j + 1 < n_kv) {
            const int st = (j + 1) & 1;
            if (hh == 0) {
              ok = mbar_wait(bar(B_KFULL + st), (uint32_t)(((j + 1) >> 1) & 1), a.status);
              if (!ok) break;
              tc_fence_after();
            }
            issue_qk(hh, st);
            umma_commit(bar(B_SFULL + hh));
            if (hh == nh - 1) umma_commit(bar(B_KEMPTY + st));
          }
        }
      }
      umma_commit(bar(B_MMADONE));
      mbar_wait(bar(B_MMADONE), 0, a.status);   // nothing of ours still runs on the tensor core
    }
  } else if ((warp >> 2) < nh) {
    // ---------------- softmax: one thread per query row ----------------
    const int hh = warp >> 2, q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int t = mt * kTile + row;
    const bool row_valid = t < Lq;
    int hi = a.causal ? min(Lk, Lk - Lq + t + 1) : Lk;   // keys [lo, hi) visible
    int lo = a.window_left >= 0 ? min(hi, max(0, Lk - Lq + t - a.window_left)) : 0;
    if (a.window_lo != nullptr) {   // variable_window: the row's inclusive bounds
      lo = row_valid ? __ldg(a.window_lo + q0 + t) : 0;
      hi = row_valid ? __ldg(a.window_hi + q0 + t) + 1 : 0;
    }
    const unsigned span = (unsigned)(hi - lo);   // key visible <=> (unsigned)(key - lo) < span
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + kColS + (uint32_t)hh * 128u;
    const uint32_t o_tm = tmem + lane_off + kColO + (uint32_t)hh * 128u;
    const float sl2 = a.scale_log2;   // >= 0 (checked by the planner)
    float m_ref = neg_inf(), l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = warp_wait(bar(B_SFULL + hh), (uint32_t)(j & 1), a.status))) break;
      tc_fence_after();
      const int key0 = (kv0 + j) * kTile;
      const bool masked = key0 < lo || key0 + kTile > hi;
      // pass 1: row max of the raw scores (scale >= 0 keeps the order); two
      // 32-column loads in flight per wait, three-input max
      float mraw = neg_inf();
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
        uint32_t ra[32], rb[32];
        tmem_ld32(s_tm + (uint32_t)c * 32u, ra);
        tmem_ld32(s_tm + (uint32_t)(c + 1) * 32u, rb);
        tmem_wait_ld();
        reg_fence32(ra);
        reg_fence32(rb);
        if (masked) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if ((unsigned)(key0 + c * 32 + i - lo) >= span) ra[i] = __float_as_uint(neg_inf());
            if ((unsigned)(key0 + (c + 1) * 32 + i - lo) >= span) rb[i] = __float_as_uint(neg_inf());
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          mraw = fmax3(mraw, __uint_as_float(ra[i]), __uint_as_float(rb[i]));
      }
      // lazy rescale: move the reference max only when it grew by more than 2^8
      const float mx = mraw == neg_inf() ? neg_inf() : mraw * sl2;
      const bool grow = mx > m_ref + kRescaleThreshold;
      const float m_new = grow ? mx : m_ref;
      const float alpha = grow ? ex2(m_ref - m_new) : 1.f;
      if (j > 0) {
        if (!(ok = warp_wait(bar(B_ODONE + hh), (uint32_t)((j - 1) & 1), a.status))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld32_sync(o_tm + (uint32_t)c * 32u, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(o_tm + (uint32_t)c * 32u, r);
          }
          tmem_wait_st();
        }
      }
      m_ref = m_new;
      // pass 2: p = exp2(s * scale*log2e - m) (one FFMA + MUFU), row sum, and
      // bf16 P written over columns [16c, 16c+16) of S -- columns of chunks
      // this thread has already read.
      const float neg_m = -m_ref;
      float sum0 = 0.f, sum1 = 0.f;
      auto exp_chunk = [&](const uint32_t* r, int c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float p0 = ex2(fmaf(__uint_as_float(r[2 * i]), sl2, neg_m));
          float p1 = ex2(fmaf(__uint_as_float(r[2 * i + 1]), sl2, neg_m));
          if (masked) {
            if ((unsigned)(key0 + c * 32 + 2 * i - lo) >= span) p0 = 0.f;
            if ((unsigned)(key0 + c * 32 + 2 * i + 1 - lo) >= span) p1 = 0.f;
          }
          sum0 += p0;
          sum1 += p1;
          pk[i] = pack2<F16>(p0, p1);
        }
        tmem_st16(s_tm + (uint32_t)c * 16u, pk);
      };
      {
        // the next chunk's load is in flight while this one is exponentiated
        uint32_t ra[32], rb[32];
        tmem_ld32_sync(s_tm, ra);
        tmem_ld32(s_tm + 32u, rb);
        exp_chunk(ra, 0);
        tmem_wait_ld();
        reg_fence32(rb);
        tmem_ld32(s_tm + 64u, ra);
        exp_chunk(rb, 1);
        tmem_wait_ld();
        reg_fence32(ra);
        tmem_ld32(s_tm + 96u, rb);
        exp_chunk(ra, 2);
        tmem_wait_ld();
        reg_fence32(rb);
        exp_chunk(rb, 3);
      }
      const float sum = sum0 + sum1;
      tmem_wait_st();
      l = l * alpha + sum;
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + hh));
    }
    if (ok && warp_wait(bar(B_ODONE + hh), (uint32_t)((n_kv - 1) & 1), a.status)) {
      tc_fence_after();
      const int h = h0 + hh;
      const float inv = l > 0.f ? a.output_scale / l : 0.f;
      const int64_t dst = ((int64_t)(q0 + t) * a.num_qo_heads + h) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32_sync(o_tm + (uint32_t)c * 32u, r);
        if (row_valid) {
#pragma unroll
          for (int qd = 0; qd < 2; ++qd) {
            float f[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) f[x] = __uint_as_float(r[16 * qd + x]);
            store_out<16>(a.out, dst + c * 32 + qd * 16, f, inv, a.out_dtype);
          }
        }
      }
      if (row_valid && a.lse != nullptr)
        a.lse[(int64_t)(q0 + t) * a.num_qo_heads + h] = l > 0.f ? m_ref + log2f(l) : neg_inf();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_prefill(const pka_prefill_plan& plan, const PrefillArgs& args, const CUtensorMap& qmap,
                   const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t stream) {
  if (args.num_tiles == 0) return PKA_OK;
  auto kern = plan.desc.dtype == PKA_DTYPE_F16 ? prefill_kernel<true> : prefill_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill)");
  kern<<<args.num_tiles, kThreads, kSmemBytes, stream>>>(args, qmap, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "prefill_kernel launch");
  return PKA_OK;
}

}  // namespace pka
