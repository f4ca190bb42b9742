// Paged decode attention on the 5th-generation tensor cores (tcgen05 + TMEM)
// for query groups wider than one 16-row tile ((Hq/Hkv) * max_q_len in
// 17..128 rows per KV head, e.g. speculative packed-Q verification with
// cudnn_batch_decode_with_kv_cache's q_len_per_req rows).
//
// Same work items, masks, softmax and outputs as the other decode kernels.
// One CTA per (request, KV head, chunk) holds all of the group's rows (row
// r = i * group + g, padded to M = 128) so each K/V unit is streamed once:
//   warps 0-3  stage Q (bf16, 128-byte swizzle) once; then one thread per
//              row (TMEM lane): for every 16-token unit, read S (16 fp32
//              columns) from TMEM, mask, online softmax in base 2 with lazy
//              rescaling of O (only when the row max grew by more than 2^8),
//              write bf16 P over the unit's S columns;
//   warp 4     TMA producer: 16-token K/V units (four 2 KB boxes) through an
//              NSTAGE-deep ring, page ids from block_tables;
//   warp 5     one thread issues tcgen05.mma: S_u = Q K_u^T (M=128, N=16,
//              K=128) into one of NS TMEM buffers, running NS units ahead of
//              the softmax, and O += P_u V_u (M=128, N=128, K=16, P read from
//              TMEM, V MN-major from shared memory).
// TMEM: S buffers [0, 16*NS), O [128, 256); 256 columns, so two CTAs share an SM.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "host_common.h"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pka {

using namespace dev;

namespace {

constexpr int kUnit = 16;
constexpr uint32_t kStageBytes = 8192;   // K (2 boxes) + V (2 boxes)
constexpr uint32_t kBoxBytes = 2048;     // 16 rows x 128 bytes
constexpr uint32_t kQBytes = 32768;      // 128 rows x 256 bytes
constexpr int kThreads = 192;
constexpr int NS = 4;                    // S buffers in TMEM
constexpr uint32_t kColO = 128;
constexpr uint32_t kTmemCols = 256;
constexpr float kRescaleThreshold = 8.0f;

// barrier indices
enum { B_KVFULL = 0 };   // [NSTAGE], then KVEMPTY [NSTAGE], SFULL [NS], PFULL [NS], PVDONE, MMADONE

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 16, 0, 0);
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

// Registers -> TMEM: 32 lanes x 8 columns of 32 bits per warp.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// TMEM -> registers: 32 lanes x 16 columns, waited for.
__device__ __forceinline__ void tmem_ld16_sync(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  tmem_wait_ld();
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
               "+r"(r[6]), "+r"(r[7]));
  asm volatile("" : "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
               "+r"(r[14]), "+r"(r[15]));
}

template <int NSTAGE>
__global__ void __launch_bounds__(kThreads, 2)
decode_tc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int B_KVEMPTY = B_KVFULL + NSTAGE, B_SFULL = B_KVEMPTY + NSTAGE;
  constexpr int B_PFULL = B_SFULL + NS, B_PVDONE = B_PFULL + NS, B_MMADONE = B_PVDONE + 1;
  constexpr int B_COUNT = B_MMADONE + 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_u32 = sbase, stage0 = sbase + kQBytes;
  const uint32_t bar0 = stage0 + NSTAGE * kStageBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kQBytes + NSTAGE * kStageBytes + B_COUNT * 8);
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
  const int all_lo = lo_last, all_hi = hi_first;

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(bar(i), (i >= B_PFULL && i < B_PFULL + NS) ? 128u : 1u);
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
          reinterpret_cast<const __nv_bfloat16*>(a.q) + (int64_t)(rq.q_start + r / G) * a.q_stride_tok +
          (int64_t)(hk * G + r % G) * a.q_stride_head);
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
          ok = mbar_wait(bar(B_KVEMPTY + st), (uint32_t)(((k / NSTAGE) - 1) & 1), a.status);
        if (ok) {
          const int u = unit0 + k;
          const int slot = (u % upp) * kUnit;
          const uint32_t dst = stage0 + st * kStageBytes;
          mbar_arrive_expect_tx(bar(B_KVFULL + st), kStageBytes);
          tma_load_4d(dst, &tmk, bar(B_KVFULL + st), 0, slot, hk, pid);
          tma_load_4d(dst + kBoxBytes, &tmk, bar(B_KVFULL + st), 64, slot, hk, pid);
          tma_load_4d(dst + 2 * kBoxBytes, &tmv, bar(B_KVFULL + st), 0, slot, hk, pid);
          tma_load_4d(dst + 3 * kBoxBytes, &tmv, bar(B_KVFULL + st), 64, slot, hk, pid);
          ++issued;
        }
      }
      if (!__shfl_sync(FULL, (int)ok, 0)) break;
    }
    if (lane == 0 && !ok && issued > 0) {   // bounded drain of loads already issued
      const int k = issued - 1;
      mbar_wait(bar(B_KVFULL + k % NSTAGE), (uint32_t)((k / NSTAGE) & 1), nullptr);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      auto issue_s = [&](int u) {
        const uint32_t d = tmem + (uint32_t)(u % NS) * 16u;
        const uint32_t kb = stage0 + (uint32_t)(u % NSTAGE) * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t adesc =
              smem_desc_sw128(q_u32 + (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
          const uint64_t bdesc =
              smem_desc_sw128(kb + (uint32_t)(kk >> 2) * kBoxBytes + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
          umma_bf16(d, adesc, bdesc, kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      bool ok = true;
      const int pre = n_units < NS ? n_units : NS;
      for (int u = 0; ok && u < pre; ++u) {
        ok = mbar_wait(bar(B_KVFULL + u % NSTAGE), (uint32_t)((u / NSTAGE) & 1), a.status);
        if (!ok) break;
        tc_fence_after();
        issue_s(u);
        umma_commit(bar(B_SFULL + u % NS));
      }
      for (int j = 0; ok && j < n_units; ++j) {
        ok = mbar_wait(bar(B_PFULL + j % NS), (uint32_t)((j / NS) & 1), a.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vb = stage0 + (uint32_t)(j % NSTAGE) * kStageBytes + 2 * kBoxBytes;
        umma_bf16_ts(tmem + kColO, tmem + (uint32_t)(j % NS) * 16u, smem_desc_sw128(vb, kBoxBytes, 1024u),
                     kIdescPV, j > 0 ? 1u : 0u);
        umma_commit(bar(B_KVEMPTY + j % NSTAGE));
        umma_commit(bar(B_PVDONE));
        const int u = j + NS;
        if (u < n_units) {
          ok = mbar_wait(bar(B_KVFULL + u % NSTAGE), (uint32_t)((u / NSTAGE) & 1), a.status);
          if (!ok) break;
          tc_fence_after();
          issue_s(u);
          umma_commit(bar(B_SFULL + u % NS));
        }
      }
      umma_commit(bar(B_MMADONE));
      mbar_wait(bar(B_MMADONE), 0, a.status);   // nothing of ours still runs on the tensor core
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
    for (int j = 0; j < n_units; ++j) {
      if (!(ok = warp_wait(bar(B_SFULL + j % NS), (uint32_t)((j / NS) & 1), a.status))) break;
      tc_fence_after();
      const uint32_t s_tm = tmem + lane_off + (uint32_t)(j % NS) * 16u;
      uint32_t s[16];
      tmem_ld16_sync(s_tm, s);
      const int tok0 = (unit0 + j) * kUnit;
      float v[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = __uint_as_float(s[c]) * sl2;
      if (!(tok0 >= all_lo && tok0 + kUnit <= all_hi)) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (tok0 + c < lo || tok0 + c >= hi) v[c] = neg_inf();
      }
      float mx = fmax3(v[0], v[1], v[2]);
#pragma unroll
      for (int c = 3; c < 15; c += 2) mx = fmax3(mx, v[c], v[c + 1]);
      mx = fmaxf(mx, v[15]);
      const bool grow = mx > m_ref + kRescaleThreshold;
      const float m_new = grow ? mx : m_ref;
      const float alpha = grow ? ex2(m_ref - m_new) : 1.f;
      if (j > 0 && __any_sync(FULL, grow)) {
        // O holds P_0..P_{j-1} V: wait for the last of them before rescaling
        if (!(ok = warp_wait(bar(B_PVDONE), (uint32_t)((j - 1) & 1), a.status))) break;
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
      float sum = 0.f;
      uint32_t pk[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float p0 = ex2(v[2 * c] - m_use), p1 = ex2(v[2 * c + 1] - m_use);
        sum += p0 + p1;
        pk[c] = float2_to_bf16x2(p0, p1);
      }
      tmem_st8(s_tm, pk);
      tmem_wait_st();
      l = l * alpha + sum;
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + j % NS));
    }
    // ---- epilogue: O / l (+ sink), or an fp32 partial ----
    const bool have_o = ok && n_units > 0 &&
                        warp_wait(bar(B_PVDONE), (uint32_t)((n_units - 1) & 1), a.status);
    if (have_o) tc_fence_after();
    if (r < rows_b) {   // base-2 LSE of the row (final) or of the chunk (partial)
      const int i = r / G, h = hk * G + r % G;
      const float lse2 = l > 0.f ? m_ref + log2f(l) : neg_inf();
      if (rq.part_base < 0) {
        if (a.lse != nullptr) a.lse[(int64_t)(rq.q_start + i) * a.num_qo_heads + h] = lse2;
      } else {
        a.ws_lse[rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h] = lse2;
      }
    }
    if (have_o) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32_sync(tmem + lane_off + kColO + (uint32_t)c * 32u, o);
        if (r < rows_b) {
          const int i = r / G, h = hk * G + r % G;
          const int t = rq.q_start + i;
          if (rq.part_base < 0) {
            float denom = l;
            if (a.sinks != nullptr && m_ref != neg_inf())
              denom += ex2(__ldg(a.sinks + h) * kLog2e - m_ref);
            const float sc = denom > 0.f ? a.bmm2_scale / denom : 0.f;
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
            const float sc = l > 0.f ? 1.f / l : 0.f;
            const int64_t prow = rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h;
            float4* dst = reinterpret_cast<float4*>(a.ws_o + prow * 128 + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * sc, __uint_as_float(o[4 * q4 + 1]) * sc,
                                    __uint_as_float(o[4 * q4 + 2]) * sc, __uint_as_float(o[4 * q4 + 3]) * sc);
          }
        }
      }
    } else if (r < rows_b) {
      // no key reached this item (or a wait gave up): zeros
      const int i = r / G, h = hk * G + r % G;
      const int t = rq.q_start + i;
      if (rq.part_base < 0) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                              ((int64_t)t * a.num_qo_heads + h) * 128);
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) dst[q4] = make_uint4(0u, 0u, 0u, 0u);
      } else {
        const int64_t prow = rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h;
        float4* dst = reinterpret_cast<float4*>(a.ws_o + prow * 128);
#pragma unroll
        for (int q4 = 0; q4 < 32; ++q4) dst[q4] = make_float4(0.f, 0.f, 0.f, 0.f);
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
  const size_t smem = 1024 + kQBytes + (size_t)NSTAGE * kStageBytes + 256;
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
