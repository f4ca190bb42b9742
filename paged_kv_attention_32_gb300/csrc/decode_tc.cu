// Paged decode attention on the 5th-generation tensor cores (tcgen05 + TMEM)
// for query groups wider than one 16-row tile ((Hq/Hkv) * max_q_len in
// 17..128 rows per KV head, e.g. speculative packed-Q verification with
// cudnn_batch_decode_with_kv_cache's q_len_per_req rows).
//
// Same work items, masks, softmax and outputs as the other decode kernels.
// One CTA per (request, KV head, chunk) holds all of the group's rows (row
// r = i * group + g, padded to M = 128), so each K/V unit is streamed once.
// Keys move in 16-token units (TMA, 128-byte swizzle) and are consumed in
// groups of four units (64 keys):
//   warp 4     TMA producer; K and V go to separate NSTAGE-deep rings laid
//              out so that four consecutive stages form one 64-row operand;
//   warp 5     one thread issues tcgen05.mma: S_g = Q K_g^T (M=128, N=64,
//              K=128) into one of two 64-column TMEM buffers, one group ahead
//              of the softmax, and O += P_g V_g (M=128, N=128, one K=16 step
//              per unit, P read from TMEM, V MN-major);
//   warps 0-3  stage Q once; then one thread per row (TMEM lane): per group,
//              read 64 S columns, mask, online softmax in base 2 with lazy
//              rescaling of O (only when the row max grew by more than 2^8),
//              write bf16 P over the group's first 32 S columns.
// TMEM: S buffers [0, 128), O [128, 256); 256 columns, two CTAs per SM.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "host_common.h"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pka {

using namespace dev;

namespace {

constexpr int kUnit = 16;                // tokens per TMA unit
constexpr int kGroup = 4;                // units per softmax step (64 keys)
constexpr uint32_t kBoxBytes = 2048;     // 16 rows x 128 bytes
constexpr uint32_t kQBytes = 32768;      // 128 rows x 256 bytes
constexpr int kThreads = 192;
constexpr uint32_t kColO = 128;
constexpr uint32_t kTmemCols = 256;
constexpr float kRescaleThreshold = 8.0f;

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);

__device__ __forceinline__ void row_key_range(int kv_len, int q_len, int i, int causal, int window,
                                              int& lo, int& hi) {
  const int d = kv_len - q_len + i;
  hi = causal ? d + 1 : kv_len;
  lo = window >= 0 ? max(0, d - window) : 0;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int32_t* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// Barriers: KVFULL [NSTAGE], KVEMPTY [NSTAGE], SFULL [2], PFULL [2], PVDONE [2],
// MMADONE.  Group buffers alternate; the softmax runs at most one group ahead
// of the PV stream, so a per-buffer barrier waited by phase parity is exact.
template <int NSTAGE>
struct TcBars {
  static constexpr int KVFULL = 0, KVEMPTY = NSTAGE, SFULL = 2 * NSTAGE, PFULL = SFULL + 2,
                       PVDONE = PFULL + 2, MMADONE = PVDONE + 2, COUNT = MMADONE + 1;
};

template <int NSTAGE>
__global__ void __launch_bounds__(kThreads, 2)
decode_tc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
  static_assert(NSTAGE % kGroup == 0, "a group must occupy consecutive stages");
  using BI = TcBars<NSTAGE>;
  constexpr unsigned FULL = 0xffffffffu;
  constexpr uint32_t kHalf = NSTAGE * kBoxBytes;   // one 64-column half of a ring
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_u32 = sbase;
  const uint32_t kring = sbase + kQBytes;            // [half][stage][16 rows x 128 B]
  const uint32_t vring = kring + 2 * kHalf;
  const uint32_t bar0 = vring + 2 * kHalf;
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(smem + kQBytes + 4 * kHalf + BI::COUNT * 8);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const WorkItem it = a.items[blockIdx.x];
  const int b = it.request;
  const int hk = it.head_chunk & 0xffff;
  const int chunk = it.head_chunk >> 16;
  const ReqInfo rq = a.reqs[b];
  const int L = rq.q_len, G = a.group;
  int kv_len = rq.kv_len;
  if (a.seq_lens_live != nullptr) kv_len = max(min(__ldg(a.seq_lens_live + b), rq.kv_len), L);
  const int rows_b = G * L;
  const int upp = a.page_size / kUnit;

  int lo_first, hi_first, lo_last, hi_last;
  row_key_range(kv_len, L, 0, a.causal, a.window_left, lo_first, hi_first);
  row_key_range(kv_len, L, L - 1, a.causal, a.window_left, lo_last, hi_last);
  const int unit0 = max(it.page_lo * upp, lo_first / kUnit);
  const int unit1 = min(it.page_hi * upp, (hi_last + kUnit - 1) / kUnit);
  const int n_units = max(0, unit1 - unit0);
  const int n_groups = (n_units + kGroup - 1) / kGroup;
  const int all_lo = lo_last, all_hi = hi_first;

  if (tid == 0) {
    for (int i = 0; i < BI::COUNT; ++i)
      mbar_init(bar(i), (i == BI::PFULL || i == BI::PFULL + 1) ? 128u : 1u);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {
    // ---- stage Q rows (row = tid) into the 128-byte swizzled K-major layout ----
    const int r = tid;
    uint4 w[16];
    if (r < rows_b) {
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(a.q) +
          (int64_t)(rq.q_start + r / G) * a.q_stride_tok + (int64_t)(hk * G + r % G) * a.q_stride_head);
#pragma unroll
      for (int c = 0; c < 16; ++c) w[c] = __ldg(src + c);
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) w[c] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int c = 0; c < 16; ++c)
      *reinterpret_cast<uint4*>(smem + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = w[c];
    fence_proxy_async_smem();   // Q is read by the tensor core (async proxy)
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
    }
    const int32_t* trow = a.block_tables + (int64_t)b * a.bt_row_stride;
    auto table_batch = [&](int batch) -> int {
      const int k = batch * 32 + lane;
      if (k < n_units) return __ldg(trow + (unit0 + k) / upp);
      return 0;
    };
    int tcur = table_batch(0), tnext = table_batch(1), tbatch = 0;
    int issued = 0;
    bool ok = true;
    for (int k = 0; k < n_units; ++k) {
      if ((k >> 5) > tbatch) {
        tcur = tnext;
        tnext = table_batch(tbatch + 2);
        ++tbatch;
      }
      const int pid = __shfl_sync(FULL, tcur, k & 31);
      if (lane == 0) {
        const int st = k % NSTAGE;
        if (k >= NSTAGE)
          ok = mbar_wait(bar(BI::KVEMPTY + st), (uint32_t)(((k / NSTAGE) - 1) & 1), a.status);
        if (ok) {
          const int u = unit0 + k;
          const int slot = (u % upp) * kUnit;
          const uint32_t fb = bar(BI::KVFULL + st);
          const uint32_t off = (uint32_t)st * kBoxBytes;
          mbar_arrive_expect_tx(fb, 4 * kBoxBytes);
          tma_load_4d(kring + off, &tmk, fb, 0, slot, hk, pid);
          tma_load_4d(kring + kHalf + off, &tmk, fb, 64, slot, hk, pid);
          tma_load_4d(vring + off, &tmv, fb, 0, slot, hk, pid);
          tma_load_4d(vring + kHalf + off, &tmv, fb, 64, slot, hk, pid);
          ++issued;
        }
      }
      if (!__shfl_sync(FULL, (int)ok, 0)) break;
    }
    if (lane == 0 && !ok && issued > 0) {   // bounded drain of loads already issued
      const int k = issued - 1;
      mbar_wait(bar(BI::KVFULL + k % NSTAGE), (uint32_t)((k / NSTAGE) & 1), nullptr);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // S of group g: wait for its units, then 8 k-steps of N = 64 keys
      auto issue_s = [&](int g) -> bool {
        const int u0 = g * kGroup, nu = min(kGroup, n_units - u0);
        for (int k = 0; k < nu; ++k) {
          const int u = u0 + k;
          if (!mbar_wait(bar(BI::KVFULL + u % NSTAGE), (uint32_t)((u / NSTAGE) & 1), a.status))
            return false;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(g & 1) * 64u;
        const uint32_t kb = kring + (uint32_t)(u0 % NSTAGE) * kBoxBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t adesc =
              smem_desc_sw128(q_u32 + (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
          const uint64_t bdesc =
              smem_desc_sw128(kb + (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
          umma_bf16(d, adesc, bdesc, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(BI::SFULL + (g & 1)));
        return true;
      };
      bool ok = true;
      for (int g = 0; ok && g < n_groups && g < 2; ++g) ok = issue_s(g);
      for (int g = 0; ok && g < n_groups; ++g) {
        ok = mbar_wait(bar(BI::PFULL + (g & 1)), (uint32_t)((g >> 1) & 1), a.status);
        if (!ok) break;
        tc_fence_after();
        const int u0 = g * kGroup, nu = min(kGroup, n_units - u0);
        const uint32_t p_tm = tmem + (uint32_t)(g & 1) * 64u;
        for (int k = 0; k < nu; ++k) {   // one K=16 step per unit present
          const uint32_t vb = vring + (uint32_t)((u0 + k) % NSTAGE) * kBoxBytes;
          umma_bf16_ts(tmem + kColO, p_tm + (uint32_t)k * 8u, smem_desc_sw128(vb, kHalf, 1024u),
                       kIdescPV, (g > 0 || k > 0) ? 1u : 0u);
        }
        for (int k = 0; k < nu; ++k) umma_commit(bar(BI::KVEMPTY + (u0 + k) % NSTAGE));
        umma_commit(bar(BI::PVDONE + (g & 1)));
        if (g + 2 < n_groups) ok = issue_s(g + 2);
      }
      umma_commit(bar(BI::MMADONE));
      mbar_wait(bar(BI::MMADONE), 0, a.status);   // nothing of ours still runs on the tensor core
    }
  } else {
    // ---------------- softmax: one thread per row (TMEM lane) ----------------
    const int r = tid;                                   // 0..127
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    int lo = 0, hi = 0x7fffffff;
    if (r < rows_b) row_key_range(kv_len, L, r / G, a.causal, a.window_left, lo, hi);
    const float sl2 = a.scale_log2;
    float m_ref = neg_inf(), l = 0.f;
    bool ok = true;
    for (int g = 0; g < n_groups; ++g) {
      if (!(ok = warp_wait(bar(BI::SFULL + (g & 1)), (uint32_t)((g >> 1) & 1), a.status))) break;
      tc_fence_after();
      const uint32_t s_tm = tmem + lane_off + (uint32_t)(g & 1) * 64u;
      uint32_t sa[32], sb[32];
      tmem_ld32(s_tm, sa);
      tmem_ld32(s_tm + 32u, sb);
      tmem_wait_ld();
      reg_fence32(sa);
      reg_fence32(sb);
      const int tok0 = (unit0 + g * kGroup) * kUnit;
      const int tok_end = unit1 * kUnit;                 // keys past the item are not loaded
      const bool full = tok0 >= all_lo && tok0 + kGroup * kUnit <= all_hi &&
                        tok0 + kGroup * kUnit <= tok_end;
      float v[64];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        v[c] = __uint_as_float(sa[c]) * sl2;
        v[32 + c] = __uint_as_float(sb[c]) * sl2;
      }
      if (!full) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int tok = tok0 + c;
          if (tok < lo || tok >= hi || tok >= tok_end) v[c] = neg_inf();
        }
      }
      float mx = fmax3(v[0], v[1], v[2]);
#pragma unroll
      for (int c = 3; c < 63; c += 2) mx = fmax3(mx, v[c], v[c + 1]);
      mx = fmaxf(mx, v[63]);
      const bool grow = mx > m_ref + kRescaleThreshold;
      const float m_new = grow ? mx : m_ref;
      const float alpha = grow ? ex2(m_ref - m_new) : 1.f;
      if (g > 0 && __any_sync(FULL, grow)) {
        // O holds the groups before g: wait for PV(g-1) before rescaling
        if (!(ok = warp_wait(bar(BI::PVDONE + ((g - 1) & 1)), (uint32_t)(((g - 1) >> 1) & 1),
                             a.status)))
          break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32_sync(tmem + lane_off + kColO + (uint32_t)c * 32u, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_off + kColO + (uint32_t)c * 32u, o);
        }
        tmem_wait_st();
      }
      m_ref = m_new;
      // a row that has seen no key yet keeps m = -inf; its p are exactly 0
      const float m_use = m_ref == neg_inf() ? 0.f : m_ref;
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2(v[2 * c] - m_use), p1 = ex2(v[2 * c + 1] - m_use);
        sum0 += p0;
        sum1 += p1;
        pk[c] = float2_to_bf16x2(p0, p1);
      }
      tmem_st32(s_tm, pk);   // P (bf16 pairs) over S columns already read
      tmem_wait_st();
      l = l * alpha + (sum0 + sum1);
      tc_fence_before();
      mbar_arrive(bar(BI::PFULL + (g & 1)));
    }
    // ---- epilogue: O / l (+ sink), or an fp32 partial ----
    const bool have_o = ok && n_groups > 0 && warp_wait(bar(BI::MMADONE), 0u, a.status);
    if (have_o) tc_fence_after();
    const int i = r / G, h = hk * G + r % G;
    const int t = rq.q_start + i;
    float sc = 0.f;
    if (r < rows_b) {   // base-2 LSE of the row (final) or of the chunk (partial)
      const float lse2 = l > 0.f ? m_ref + log2f(l) : neg_inf();
      if (rq.part_base < 0) {
        float denom = l;
        if (a.sinks != nullptr && m_ref != neg_inf()) denom += ex2(__ldg(a.sinks + h) * kLog2e - m_ref);
        sc = denom > 0.f ? a.bmm2_scale / denom : 0.f;
        if (a.lse != nullptr) a.lse[(int64_t)t * a.num_qo_heads + h] = lse2;
      } else {
        sc = l > 0.f ? 1.f / l : 0.f;
        a.ws_lse[rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h] = lse2;
      }
    }
    if (!have_o) sc = 0.f;   // no key reached the item (or a wait gave up): zeros
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32_sync(tmem + lane_off + kColO + (uint32_t)c * 32u, o);
      } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) o[x] = 0u;
      }
      if (r < rows_b) {
        if (rq.part_base < 0) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                                ((int64_t)t * a.num_qo_heads + h) * 128 + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            dst[q4] = make_uint4(
                float2_to_bf16x2(__uint_as_float(o[8 * q4]) * sc, __uint_as_float(o[8 * q4 + 1]) * sc),
                float2_to_bf16x2(__uint_as_float(o[8 * q4 + 2]) * sc, __uint_as_float(o[8 * q4 + 3]) * sc),
                float2_to_bf16x2(__uint_as_float(o[8 * q4 + 4]) * sc, __uint_as_float(o[8 * q4 + 5]) * sc),
                float2_to_bf16x2(__uint_as_float(o[8 * q4 + 6]) * sc, __uint_as_float(o[8 * q4 + 7]) * sc));
        } else {
          const int64_t prow = rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h;
          float4* dst = reinterpret_cast<float4*>(a.ws_o + prow * 128 + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * sc, __uint_as_float(o[4 * q4 + 1]) * sc,
                                  __uint_as_float(o[4 * q4 + 2]) * sc, __uint_as_float(o[4 * q4 + 3]) * sc);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NSTAGE>
int launch_tc(const DecodeArgs& args, const CUtensorMap& kmap, const CUtensorMap& vmap,
              cudaStream_t stream) {
  const size_t smem = 1024 + kQBytes + (size_t)4 * NSTAGE * kBoxBytes + 256;
  auto kern = decode_tc_kernel<NSTAGE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_tc)");
  kern<<<args.num_items, kThreads, smem, stream>>>(args, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_tc_kernel launch");
  return PKA_OK;
}

}  // namespace

int launch_decode_tc(const DecodeArgs& args, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     cudaStream_t stream) {
  return launch_tc<8>(args, kmap, vmap, stream);
}

}  // namespace pka
