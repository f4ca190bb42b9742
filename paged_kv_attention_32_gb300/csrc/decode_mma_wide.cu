// Paged decode attention on tensor cores for groups wider than one 16-row
// tile ((Hq/Hkv) * max_q_len in 17..64 rows, e.g. speculative packed-Q
// verification with up to 6 rows per request and 8 query heads per KV head).
//
// One CTA per work item holds all MT tiles of the item's query rows, so each
// K/V unit is streamed once.  The four warps work on the same 16-token unit:
//   phase A  warp t < MT: S = Q_t K^T (mma.sync m16n8k16), mask, online
//            softmax (base 2) for tile t's rows; it publishes its bf16 P
//            A-fragments (one 16-byte word per lane) and the rows' rescale
//            factors in shared memory;
//   barrier  (one per unit, a CTA-wide vote that also carries wait
//            failures; P and the factors are double-buffered by unit parity,
//            and every warp reaches it only after its phase B of the previous
//            unit, whose stage is then refilled);
//   phase B  warp w: O[:, 32w:32w+32] += P_t V for every tile t (V through
//            ldmatrix.trans), after rescaling its accumulator rows.
// A unit's stage is refilled (TMA, 4 boxes of 2 KB, 128-byte swizzle) by
// thread 0 right after the barrier that follows the last read of it.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "host_common.h"
#include "kernels.h"

namespace pka {

using namespace dev;

namespace {

constexpr int kWarps = 4;
constexpr int kUnit = 16;
constexpr int kStageBytes = 8192;
constexpr int kBoxBytes = 2048;

__device__ __forceinline__ void row_key_range(int kv_len, int q_len, int i, int causal, int window,
                                              int& lo, int& hi) {
  const int d = kv_len - q_len + i;
  hi = causal ? d + 1 : kv_len;
  lo = window >= 0 ? max(0, d - window) : 0;
}

__device__ __forceinline__ uint32_t unit_chunk_offset(int j, int cg) {
  return (uint32_t)(cg >> 3) * kBoxBytes + swz128((uint32_t)j, (uint32_t)(cg & 7));
}

template <int MT, int NSTAGE>
__global__ void __launch_bounds__(kWarps * 32, 3)
decode_mma_wide_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv) {
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint4* pfrag = reinterpret_cast<uint4*>(smem + NSTAGE * kStageBytes);        // [2][MT][32]
  float* alpha_s = reinterpret_cast<float*>(pfrag + 2 * MT * 32);               // [2][MT][16]
  float* ml_s = alpha_s + 2 * MT * 16;                                          // [MT][16][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ml_s + MT * 32);

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
  const int mt_b = (rows_b + 15) >> 4;      // tiles this request uses (<= MT)
  const int upp = a.page_size / kUnit;

  int lo_first, hi_first, lo_last, hi_last;
  row_key_range(kv_len, L, 0, a.causal, a.window_left, lo_first, hi_first);
  row_key_range(kv_len, L, L - 1, a.causal, a.window_left, lo_last, hi_last);
  const int unit0 = max(it.page_lo * upp, lo_first / kUnit);
  const int unit1 = min(it.page_hi * upp, (hi_last + kUnit - 1) / kUnit);
  const int n_units = max(0, unit1 - unit0);
  const int all_lo = lo_last, all_hi = hi_first;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(smem_u32(bars + s), 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  __syncthreads();

  const int32_t* trow = a.block_tables + (int64_t)b * a.bt_row_stride;
  auto issue = [&](int k) {   // thread 0 only
    const int u = unit0 + k;
    const int pid = __ldg(trow + u / upp);
    const int slot = (u % upp) * kUnit;
    const int st = k % NSTAGE;
    const uint32_t dst = smem_u32(stages + st * kStageBytes), bar = smem_u32(bars + st);
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_4d(dst, &tmk, bar, 0, slot, hk, pid);
    tma_load_4d(dst + kBoxBytes, &tmk, bar, 64, slot, hk, pid);
    tma_load_4d(dst + 2 * kBoxBytes, &tmv, bar, 0, slot, hk, pid);
    tma_load_4d(dst + 3 * kBoxBytes, &tmv, bar, 64, slot, hk, pid);
  };
  if (tid == 0) {
    const int pre = n_units < NSTAGE ? n_units : NSTAGE;
    for (int k = 0; k < pre; ++k) issue(k);
  }

  const int g4 = lane >> 2, t4 = lane & 3;
  const int lm_mat = lane >> 3, lm_row = lane & 7;
  const bool tile_warp = warp < mt_b;        // warp t owns tile t in phase A
  // ---- phase A state (tile warps) ----
  const int rA = warp * 16 + g4, rB = rA + 8;
  int loA = 0, hiA = 0x7fffffff, loB = 0, hiB = 0x7fffffff;
  if (rA < rows_b) row_key_range(kv_len, L, rA / G, a.causal, a.window_left, loA, hiA);
  if (rB < rows_b) row_key_range(kv_len, L, rB / G, a.causal, a.window_left, loB, hiB);
  uint32_t qa[8][4];
  {
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* srcA = nullptr;
    const __nv_bfloat16* srcB = nullptr;
    if (tile_warp && rA < rows_b)
      srcA = qb + (int64_t)(rq.q_start + rA / G) * a.q_stride_tok +
             (int64_t)(hk * G + rA % G) * a.q_stride_head;
    if (tile_warp && rB < rows_b)
      srcB = qb + (int64_t)(rq.q_start + rB / G) * a.q_stride_tok +
             (int64_t)(hk * G + rB % G) * a.q_stride_head;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c0 = ks * 16 + t4 * 2;
      qa[ks][0] = srcA ? __ldg(reinterpret_cast<const uint32_t*>(srcA + c0)) : 0u;
      qa[ks][1] = srcB ? __ldg(reinterpret_cast<const uint32_t*>(srcB + c0)) : 0u;
      qa[ks][2] = srcA ? __ldg(reinterpret_cast<const uint32_t*>(srcA + c0 + 8)) : 0u;
      qa[ks][3] = srcB ? __ldg(reinterpret_cast<const uint32_t*>(srcB + c0 + 8)) : 0u;
    }
  }
  float mA = neg_inf(), mB = neg_inf(), lA = 0.f, lB = 0.f;
  const float sl2 = a.scale_log2;
  // ---- phase B state: O[tile][4 n-tiles of this warp's 32 columns] ----
  float acc[MT][4][4];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int n = 0; n < 4; ++n) acc[t][n][0] = acc[t][n][1] = acc[t][n][2] = acc[t][n][3] = 0.f;

  bool ok = true;
  for (int k = 0; k < n_units; ++k) {
    const int st = k % NSTAGE, par = k & 1;
    ok = __all_sync(FULL, mbar_wait(smem_u32(bars + st), (uint32_t)((k / NSTAGE) & 1), a.status));
    const uint32_t k_u32 = smem_u32(stages + st * kStageBytes);
    const uint32_t v_u32 = k_u32 + 2 * kBoxBytes;
    if (ok && tile_warp) {
      // ---------------- phase A: scores and softmax of tile `warp` ----------------
      float s[2][4], s2[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
      }
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(k_u32 + unit_chunk_offset(nt * 8 + lm_row, kp * 4 + lm_mat), b0, b1, b2, b3);
          mma_bf16_16816(s[nt], qa[2 * kp], b0, b1);
          mma_bf16_16816(s2[nt], qa[2 * kp + 1], b2, b3);
        }
      }
      const int tok0 = (unit0 + k) * kUnit;
      const bool full_unit = tok0 >= all_lo && tok0 + kUnit <= all_hi;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v = (s[nt][c] + s2[nt][c]) * sl2;
          if (!full_unit) {
            const int tok = tok0 + nt * 8 + t4 * 2 + (c & 1);
            const int lo = c >= 2 ? loB : loA, hi = c >= 2 ? hiB : hiA;
            if (tok < lo || tok >= hi) v = neg_inf();
          }
          s[nt][c] = v;
        }
      float pmA = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float pmB = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      pmA = fmaxf(pmA, __shfl_xor_sync(FULL, pmA, 1));
      pmB = fmaxf(pmB, __shfl_xor_sync(FULL, pmB, 1));
      pmA = fmaxf(pmA, __shfl_xor_sync(FULL, pmA, 2));
      pmB = fmaxf(pmB, __shfl_xor_sync(FULL, pmB, 2));
      const float mAn = fmaxf(mA, pmA), mBn = fmaxf(mB, pmB);
      const float uA = mAn == neg_inf() ? 0.f : mAn, uB = mBn == neg_inf() ? 0.f : mBn;
      const float alA = ex2(mA - uA), alB = ex2(mB - uB);
      mA = mAn;
      mB = mBn;
      float sumA = 0.f, sumB = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = ex2(s[nt][0] - uA);
        s[nt][1] = ex2(s[nt][1] - uA);
        s[nt][2] = ex2(s[nt][2] - uB);
        s[nt][3] = ex2(s[nt][3] - uB);
        sumA += s[nt][0] + s[nt][1];
        sumB += s[nt][2] + s[nt][3];
      }
      lA = lA * alA + sumA;
      lB = lB * alB + sumB;
      pfrag[(par * MT + warp) * 32 + lane] =
          make_uint4(float2_to_bf16x2(s[0][0], s[0][1]), float2_to_bf16x2(s[0][2], s[0][3]),
                     float2_to_bf16x2(s[1][0], s[1][1]), float2_to_bf16x2(s[1][2], s[1][3]));
      if (t4 == 0) {
        alpha_s[(par * MT + warp) * 16 + g4] = alA;
        alpha_s[(par * MT + warp) * 16 + g4 + 8] = alB;
      }
    }
    // CTA barrier and vote: every warp reaches it after its phase B of unit k-1,
    // so the stage of unit k-1 is free; a failed wait anywhere stops all warps.
    const int failed = __syncthreads_or(ok ? 0 : 1);
    if (failed) break;
    if (tid == 0 && k >= 1 && k - 1 + NSTAGE < n_units) issue(k - 1 + NSTAGE);
    // ---------------- phase B: O[:, 32w:32w+32] += P_t V ----------------
    uint32_t vb[4][2];
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      const int key = (lm_mat & 1) * 8 + lm_row;
      const int cg = warp * 4 + np * 2 + (lm_mat >> 1);
      ldmatrix_x4_trans(v_u32 + unit_chunk_offset(key, cg), vb[2 * np][0], vb[2 * np][1],
                        vb[2 * np + 1][0], vb[2 * np + 1][1]);
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      if (t < mt_b) {
        const float aA = alpha_s[(par * MT + t) * 16 + g4];
        const float aB = alpha_s[(par * MT + t) * 16 + g4 + 8];
        if (__any_sync(FULL, aA != 1.f || aB != 1.f)) {
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            acc[t][n][0] *= aA;
            acc[t][n][1] *= aA;
            acc[t][n][2] *= aB;
            acc[t][n][3] *= aB;
          }
        }
        const uint4 pw = pfrag[(par * MT + t) * 32 + lane];
        const uint32_t pa[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
        for (int n = 0; n < 4; ++n) mma_bf16_16816(acc[t][n], pa, vb[n][0], vb[n][1]);
      }
    }
  }

  // ---- finalize: tile warps publish (m, l) per row ----
  if (tile_warp) {
    lA += __shfl_xor_sync(FULL, lA, 1);
    lA += __shfl_xor_sync(FULL, lA, 2);
    lB += __shfl_xor_sync(FULL, lB, 1);
    lB += __shfl_xor_sync(FULL, lB, 2);
    if (t4 == 0) {
      ml_s[(warp * 16 + g4) * 2] = mA;
      ml_s[(warp * 16 + g4) * 2 + 1] = lA;
      ml_s[(warp * 16 + g4 + 8) * 2] = mB;
      ml_s[(warp * 16 + g4 + 8) * 2 + 1] = lB;
    }
  }
  __syncthreads();
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
#pragma unroll
  for (int t = 0; t < MT; ++t) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int rr = t * 16 + g4 + half * 8;   // row of the group
      if (rr >= rows_b) continue;
      const float m = ml_s[rr * 2], l = ml_s[rr * 2 + 1];
      const int i = rr / G, h = hk * G + rr % G;
      const int tt = rq.q_start + i;
      const int col0 = warp * 32 + t4 * 2;
      if (rq.part_base < 0) {
        float denom = l;
        if (a.sinks != nullptr && m != neg_inf()) denom += ex2(__ldg(a.sinks + h) * kLog2e - m);
        const float sc = denom > 0.f ? a.bmm2_scale / denom : 0.f;
        __nv_bfloat16* dst = out + ((int64_t)tt * a.num_qo_heads + h) * 128 + col0;
#pragma unroll
        for (int n = 0; n < 4; ++n)
          *reinterpret_cast<uint32_t*>(dst + n * 8) =
              float2_to_bf16x2(acc[t][n][2 * half] * sc, acc[t][n][2 * half + 1] * sc);
        if (a.lse != nullptr && warp == 0 && t4 == 0)
          a.lse[(int64_t)tt * a.num_qo_heads + h] = l > 0.f ? m + log2f(l) : neg_inf();
      } else {
        const int64_t prow = rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h;
        const float sc = l > 0.f ? 1.f / l : 0.f;
        float* dst = a.ws_o + prow * 128 + col0;
#pragma unroll
        for (int n = 0; n < 4; ++n)
          *reinterpret_cast<float2*>(dst + n * 8) =
              make_float2(acc[t][n][2 * half] * sc, acc[t][n][2 * half + 1] * sc);
        if (warp == 0 && t4 == 0) a.ws_lse[prow] = l > 0.f ? m + log2f(l) : neg_inf();
      }
    }
  }
}

template <int MT, int NSTAGE>
int launch_wide(const DecodeArgs& args, const CUtensorMap& kmap, const CUtensorMap& vmap,
                cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)NSTAGE * kStageBytes + 2 * MT * 32 * 16 + 2 * MT * 16 * 4 +
                      MT * 32 * 4 + NSTAGE * 8;
  auto kern = decode_mma_wide_kernel<MT, NSTAGE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_mma_wide)");
  kern<<<args.num_items, kWarps * 32, smem, stream>>>(args, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_mma_wide_kernel launch");
  return PKA_OK;
}

}  // namespace

int launch_decode_mma_wide(const DecodeArgs& args, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t stream) {
  const int mt = (args.rows_per_cta + 15) / 16;
  switch (mt) {
    case 2: return launch_wide<2, 8>(args, kmap, vmap, stream);
    case 3: return launch_wide<3, 8>(args, kmap, vmap, stream);
    default: return launch_wide<4, 8>(args, kmap, vmap, stream);
  }
}

}  // namespace pka
