// Prefill, one query head per CTA, on the 5th-generation tensor cores
// (tcgen05 + TMEM); head_dim D = 128 or 256.
//
// Masks and outputs: bottom-right causal diagonal, dense, left window,
// variable_window; O scaled by output_scale, base-2 LSE.  One CTA = one
// 128-row query tile of one request and one query head, keys in tiles of 64:
// Q (D/64 boxes of 16 KB) + two K and two V stages (D/64 boxes of 8 KB each)
// in shared memory.
//   warp 4      TMA producer: Q once, then K and V tiles (64-column boxes,
//               128-byte swizzle);
//   warp 5      allocates TMEM and issues every tcgen05.mma (one elected lane,
//               four chained k-steps per asm block):
//               S_b = Q K^T (M=128, N=64, D/16 k-steps) into one of two S
//               buffers -- two key tiles ahead of the softmax, so the tensor
//               core works while the softmax runs -- and O += P V (M=128,
//               N=D, 4 k-steps of 16 keys, P read from TMEM, V MN-major);
//   warps 0-3   softmax, one thread per query row (TMEM lane): row max of the
//               64 scores, lazy rescaling of O only when the max grew by more
//               than 2^8, p = exp2(s * scale*log2e - m), bf16/f16 P over the
//               first 32 columns of the S buffer, final O / l and LSE.
// TMEM columns: S0 [0,64) S1 [64,128) O [128,128+D) (256 or 512 allocated;
// with D = 128 two CTAs share an SM).
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "host_common.h"
#include "prefill.h"
#include "prefill_softmax.cuh"
#include "tcgen05.cuh"

namespace pka {

using namespace dev;

namespace {

constexpr int kTileQ = 128, kTileK = 64;
constexpr uint32_t kQBox = 16384;           // 128 rows x 128 bytes (64 columns)
constexpr uint32_t kKBox = 8192;            // 64 rows x 128 bytes
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kColO = 128;

// Shared memory and TMEM of head_dim D (NB = D / 64 column blocks): Q NB x 16 KB,
// then two K and two V stages of NB x 8 KB; S0 S1 (64 columns each) then O (D).
template <int D>
struct Geo {
  static constexpr int NB = D / 64;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = NB * kQBox;
  static constexpr uint32_t kOffV = kOffK + 2 * NB * kKBox;
  static constexpr uint32_t kOffBar = kOffV + 2 * NB * kKBox;
  static constexpr size_t kSmemBytes = 1024 + kOffBar + 256;
  static constexpr uint32_t kTmemCols = kColO + D <= 256 ? 256 : 512;
  static constexpr int kMinBlocks = D == 128 ? 2 : 1;   // 2 x 97 KB, 2 x 256 TMEM columns
};

// mbarriers, two of each per stage or S buffer (tile j uses j & 1).  A parity
// wait is only correct when the barrier has completed the phase before the
// awaited one, and every wait here keeps to that: K/V full/empty and S/P are
// waited in order by one consumer each; the O-done wait for P V of tile j - 1
// (lazy rescale) or n_kv - 1 (epilogue) comes after S of tile j, whose QK was
// issued after P V of tile j - 2, which therefore completed.
enum {
  B_Q = 0, B_KFULL = 1, B_KEMPTY = 3, B_VFULL = 5, B_VEMPTY = 7, B_SFULL = 9, B_PFULL = 11,
  B_ODONE = 13, B_MMADONE = 15, B_COUNT = 16
};

template <bool F16> constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, 0, 0, F16);
template <int D, bool F16> constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1, F16);

// Q (128 rows) or K (64 rows) as the K-major operand: column block kk / 4,
// 32-byte step kk % 4 inside the 128-byte rows, 8-row groups every 1024 bytes.
__device__ __forceinline__ uint64_t kmajor(uint32_t base, uint32_t block_bytes, int kk) {
  return smem_desc_sw128(base + (uint32_t)(kk >> 2) * block_bytes + (uint32_t)(kk & 3) * 32u, 16u,
                         1024u);
}
// V tile (64 keys x 256 dims) as the MN-major B operand of k-step kk (keys
// 16kk .. 16kk+15): 64-dim blocks every 8 KB, 8-key groups every 1024 bytes.
__device__ __forceinline__ uint64_t vmn(uint32_t base, int kk) {
  return smem_desc_sw128(base + (uint32_t)kk * 2048u, kKBox, 1024u);
}

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, Geo<D>::kMinBlocks)
prefill_1h_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using Gm = Geo<D>;
  constexpr int NB = Gm::NB;
  constexpr uint32_t kOffQ = Gm::kOffQ, kOffK = Gm::kOffK, kOffV = Gm::kOffV, kOffBar = Gm::kOffBar;
  constexpr uint32_t kTmemCols = Gm::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + B_COUNT * 8);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PrefillTile tile = a.tiles[blockIdx.x];
  const int h = tile.head, mt = tile.q_tile, n_kv = tile.n_kv;
  const int kv0 = tile.kv0;
  const int q0 = tile.q0, Lq = tile.lq;
  const int k0 = tile.k0, Lk = tile.lk;
  const int hk = h / a.group;

  // Q rows in the order of a row map (variable_window tiles of similar
  // windows) are gathered by the softmax threads, one row each; else one TMA copy
  const bool gather_q = a.row_map != nullptr;
  if (tid == 0) {
    mbar_init(bar(B_Q), gather_q ? 128 : 1);
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
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      if (!gather_q) {
        mbar_arrive_expect_tx(bar(B_Q), NB * kQBox);
        for (int blk = 0; blk < NB; ++blk)
          tma_load_3d(sbase + kOffQ + (uint32_t)blk * kQBox, &tmq, bar(B_Q), blk * 64, h,
                      q0 + mt * kTileQ);
      }
      auto load_kv = [&](int j, int which) -> bool {   // which: 0 = K, 1 = V
        const int st = j & 1;
        const int full = which ? B_VFULL : B_KFULL, empty = which ? B_VEMPTY : B_KEMPTY;
        if (j >= 2 && !mbar_wait(bar(empty + st), (uint32_t)(((j >> 1) - 1) & 1), a.status))
          return false;
        const uint32_t dst = sbase + (which ? kOffV : kOffK) + (uint32_t)st * NB * kKBox;
        mbar_arrive_expect_tx(bar(full + st), NB * kKBox);
        for (int blk = 0; blk < NB; ++blk)
          tma_load_3d(dst + (uint32_t)blk * kKBox, which ? &tmv : &tmk, bar(full + st), blk * 64,
                      hk, k0 + (kv0 + j) * kTileK);
        return true;
      };
      bool ok = true;
      int kd = 0, vd = 0;   // K and V tiles issued
      // order K0 K1 V0 K2 V1 K3 ...: S of tile j + 2 is issued after P V of tile j
      while (ok && (kd < n_kv || vd < n_kv)) {
        if (kd < n_kv && kd <= vd + 1) {
          ok = load_kv(kd, 0);
          kd += ok;
        } else {
          ok = load_kv(vd, 1);
          vd += ok;
        }
      }
      if (!ok) {   // give the copies already issued a bounded chance to land
        if (!gather_q) mbar_wait(bar(B_Q), 0, nullptr);
        if (kd > 0) mbar_wait(bar(B_KFULL + ((kd - 1) & 1)), (uint32_t)(((kd - 1) >> 1) & 1), nullptr);
        if (vd > 0) mbar_wait(bar(B_VFULL + ((vd - 1) & 1)), (uint32_t)(((vd - 1) >> 1) & 1), nullptr);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer: the warp waits, one elected lane issues ----------------
    auto issue_qk = [&](int j) -> bool {   // S of tile j into buffer j & 1
      const int st = j & 1;
      if (!warp_wait(bar(B_KFULL + st), (uint32_t)((j >> 1) & 1), a.status)) return false;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)st * 64u;
      const uint32_t kb = sbase + kOffK + (uint32_t)st * NB * kKBox;
#pragma unroll
      for (int blk = 0; blk < NB; ++blk)   // 4 k-steps of 16 per 64-column block
        umma_ss_k4(d, kmajor(sbase + kOffQ, kQBox, 4 * blk), kmajor(kb, kKBox, 4 * blk),
                   kIdescQK<F16>, blk > 0 ? 1u : 0u);
      umma_commit_elect(bar(B_SFULL + st));
      umma_commit_elect(bar(B_KEMPTY + st));
      return true;
    };
    bool ok = warp_wait(bar(B_Q), 0, a.status);
    for (int j = 0; ok && j < n_kv && j < 2; ++j) ok = issue_qk(j);
    for (int j = 0; ok && j < n_kv; ++j) {
      const int st = j & 1;
      ok = warp_wait(bar(B_VFULL + st), (uint32_t)((j >> 1) & 1), a.status) &&
           warp_wait(bar(B_PFULL + st), (uint32_t)((j >> 1) & 1), a.status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t p_tm = tmem + (uint32_t)st * 64u;   // P: 32 columns, lanes 0-127
      const uint32_t vb = sbase + kOffV + (uint32_t)st * NB * kKBox;
      // 4 k-steps of 16 keys: P columns +8, V rows +16 (2048 bytes)
      umma_ts_k4<2048 / 16>(tmem + kColO, p_tm, vmn(vb, 0), kIdescPV<D, F16>, j > 0 ? 1u : 0u);
      umma_commit_elect(bar(B_ODONE + st));
      umma_commit_elect(bar(B_VEMPTY + st));
      // S buffer st is free again once this P V has read P (issue order)
      if (j + 2 < n_kv) ok = issue_qk(j + 2);
    }
    umma_commit_elect(bar(B_MMADONE));
    warp_wait(bar(B_MMADONE), 0, a.status);   // nothing of ours still runs on the tensor core
  } else {
    // ---------------- softmax: one thread per query row ----------------
    const int row = tid;                       // warps 0-3
    const int pos = mt * kTileQ + row;         // the row's position in the request's tiles
    const bool row_valid = pos < Lq;
    const int t = gather_q && row_valid ? __ldg(a.row_map + q0 + pos) : pos;   // query row
    if (gather_q) {
      // this thread's Q row into the tile's shared-memory layout (128-byte
      // swizzle, D / 64 column blocks), zeros past the request's rows
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint16_t*>(a.q) + (int64_t)(q0 + t) * a.q_stride_tok +
          (int64_t)h * a.q_stride_head);
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = row_valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + kOffQ + (uint32_t)(c >> 3) * kQBox +
                                  swz128((uint32_t)row, (uint32_t)(c & 7))) = v;
      }
      fence_proxy_async_smem();   // generic writes -> the tensor core's operand reads
      mbar_arrive(bar(B_Q));
    }
    int hi = a.causal ? min(Lk, Lk - Lq + t + 1) : Lk;   // keys [lo, hi) visible
    int lo = a.window_left >= 0 ? min(hi, max(0, Lk - Lq + t - a.window_left)) : 0;
    if (a.window_lo != nullptr) {   // variable_window: the row's inclusive bounds
      lo = row_valid ? __ldg(a.window_lo + q0 + t) : 0;
      hi = row_valid ? __ldg(a.window_hi + q0 + t) + 1 : 0;
    }
    const unsigned span = (unsigned)(hi - lo);   // key visible <=> (unsigned)(key - lo) < span
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t o_tm = tmem + lane_off + kColO;
    const float sl2 = a.scale_log2;   // >= 0 (checked by the planner)
    float m_ref = neg_inf(), l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      if (!(ok = warp_wait(bar(B_SFULL + st), (uint32_t)((j >> 1) & 1), a.status))) break;
      tc_fence_after();
      const uint32_t s_tm = tmem + lane_off + (uint32_t)st * 64u;
      const int key0 = (kv0 + j) * kTileK;
      // warp-uniform: a tile that needs the mask in any row takes the masked path
      const bool masked = __any_sync(0xffffffffu, key0 < lo || key0 + kTileK > hi);
      uint32_t ra[32], rb[32];
      tmem_ld32(s_tm, ra);
      tmem_ld32(s_tm + 32u, rb);
      tmem_wait_ld();
      reg_fence32(ra);
      reg_fence32(rb);
      uint32_t w0 = 0xffffffffu, w1 = 0xffffffffu;
      if (masked) {
        visible_bits(key0, lo, span, w0, w1);
        mask_scores64(ra, rb, w0, w1);
      }
      const float mraw = row_max64(ra, rb);
      // lazy rescale: move the reference max only when it grew by more than 2^8
      const float mx = mraw == neg_inf() ? neg_inf() : mraw * sl2;
      const bool grow = mx > m_ref + kRescaleThreshold;
      const float m_new = grow ? mx : m_ref;
      // A row that had no visible key yet holds O = 0 and l = 0 (its P was 0):
      // it takes its first reference without a rescale, so that rows whose
      // windows start at different key tiles do not stall the warp on the
      // previous tile's P V one after another.
      const bool rescale = grow && m_ref != neg_inf();
      const float alpha = rescale ? ex2(m_ref - m_new) : 1.f;
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // O holds tiles before j: wait for P V of tile j - 1 before rescaling
        if (!(ok = warp_wait(bar(B_ODONE + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1),
                             a.status)))
          break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(o_tm + (uint32_t)c * 32u, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(o_tm + (uint32_t)c * 32u, r);
        }
        tmem_wait_st();
      }
      m_ref = m_new;
      // A row with no visible key so far keeps m_ref = -inf: its scores here
      // are all -inf, and exp2(-inf * sl2 + 0) = 0 (-inf - -inf would be NaN).
      // Masked scores give 0 through their -inf unless the scale is 0.
      const float neg_m = m_ref == neg_inf() ? 0.f : -m_ref;
      const bool zero_again = masked && !(sl2 > 0.f);
      const float2 sum = zero_again
                             ? exp_tile<true, F16>(ra, rb, sl2, neg_m, w0, w1, s_tm)
                             : exp_tile<false, F16>(ra, rb, sl2, neg_m, w0, w1, s_tm);
      tmem_wait_st();
      l = l * alpha + (sum.x + sum.y);
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + st));
    }
    if (ok && n_kv > 0 &&
        warp_wait(bar(B_ODONE + ((n_kv - 1) & 1)), (uint32_t)(((n_kv - 1) >> 1) & 1), a.status)) {
      tc_fence_after();
      const float inv = l > 0.f ? a.output_scale / l : 0.f;
      // head_dim 256 (one CTA per SM) measured faster with direct stores
      if (D != 128 || a.out_dtype == PKA_DTYPE_F32) {
        const int64_t dst = ((int64_t)(q0 + t) * a.num_qo_heads + h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
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
      } else {
        // 16-bit O: each warp stages its 32 rows in the Q buffer (every QK has
        // completed) with 16-byte chunks XOR-swizzled by row, then writes whole
        // rows back, two per store instruction (coalesced 256-byte rows instead
        // of 32 rows touched by every store).
        constexpr int kRowBytes = D * 2, kChunks = kRowBytes / 16;
        constexpr int kLanesPerRow = kChunks < 32 ? kChunks : 32;
        uint8_t* wbuf = smem + kOffQ + (uint32_t)warp * 32u * kRowBytes;
        const bool f16o = a.out_dtype == PKA_DTYPE_F16;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(o_tm + (uint32_t)c * 32u, r);
#pragma unroll
          for (int k = 0; k < 4; ++k) {   // 8 values = one 16-byte chunk
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float lo = __uint_as_float(r[8 * k + 2 * x]) * inv;
              const float hi = __uint_as_float(r[8 * k + 2 * x + 1]) * inv;
              w[x] = f16o ? pack2<true>(lo, hi) : pack2<false>(lo, hi);
            }
            const int q = c * 4 + k;
            *reinterpret_cast<uint4*>(wbuf + lane * kRowBytes + ((q ^ (lane & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        __syncwarp();
        const int q = lane % kLanesPerRow;
#pragma unroll 4
        for (int r0 = 0; r0 < 32; r0 += 32 / kLanesPerRow) {
          const int rr = r0 + lane / kLanesPerRow;
          const int pr = mt * kTileQ + warp * 32 + rr;
          const uint4 val =
              *reinterpret_cast<const uint4*>(wbuf + rr * kRowBytes + ((q ^ (rr & 7)) << 4));
          const int tr = __shfl_sync(0xffffffffu, t, rr);   // row rr's query row (lane rr's t)
          if (pr < Lq) {
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) +
                                      ((int64_t)(q0 + tr) * a.num_qo_heads + h) * kRowBytes +
                                      q * 16) = val;
          }
        }
      }
      if (row_valid && a.lse != nullptr)
        a.lse[(int64_t)(q0 + t) * a.num_qo_heads + h] = l > 0.f ? m_ref + log2f(l) : neg_inf();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
int launch_1h(const pka_prefill_plan& plan, const PrefillArgs& args, const CUtensorMap& qmap,
              const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t stream) {
  if (args.num_tiles == 0) return PKA_OK;
  auto kern = plan.desc.dtype == PKA_DTYPE_F16 ? prefill_1h_kernel<D, true>
                                               : prefill_1h_kernel<D, false>;
  const int smem = (int)Geo<D>::kSmemBytes;
  static std::atomic<uint64_t> smem_set[2];   // per input type: devices whose limit was raised
  cudaError_t e = set_smem_once(kern, smem, smem_set[plan.desc.dtype == PKA_DTYPE_F16]);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_1h)");
  kern<<<args.num_tiles, kThreads, smem, stream>>>(args, qmap, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "prefill_1h_kernel launch");
  return PKA_OK;
}

}  // namespace

int launch_prefill_1h(const pka_prefill_plan& plan, const PrefillArgs& args,
                      const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      cudaStream_t stream) {
  if (plan.D == 256) return launch_1h<256>(plan, args, qmap, kmap, vmap, stream);
  return launch_1h<128>(plan, args, qmap, kmap, vmap, stream);
}

}  // namespace pka
