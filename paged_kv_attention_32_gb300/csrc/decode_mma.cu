// Paged decode attention, tensor-core variant for wide query groups
// ((Hq/Hkv) * max_q_len >= 16 rows per KV head, e.g. speculative packed-Q
// verification with cudnn_batch_decode_with_kv_cache's q_len_per_req rows).
//
// Same work item, masks, softmax and outputs as the CUDA-core kernel; the
// contractions run on mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//  * MT consumer warps each own one 16-row tile of the group's query rows
//    (row r = i * group + g: token i, head g of the group); Q stays in
//    A-fragment registers for the whole item;
//  * one producer warp streams the item's 16-token K/V units with TMA into an
//    NSTAGE-deep shared ring (full / empty mbarriers; 128-byte swizzle keeps
//    ldmatrix conflict-free);
//  * per unit: S = Q K^T (2 n-tiles x 8 k-steps), mask, online softmax in
//    base 2 on the fragments, P re-packed to bf16 A fragments in registers,
//    O += P V (16 n-tiles, V read with ldmatrix.trans).
// Decode is bound by HBM, not by the tensor pipe: the mma path exists to take
// the per-key arithmetic of 16..64 rows off the FP32 pipe.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "host_common.h"
#include "kernels.h"

namespace pka {

using namespace dev;

namespace {

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
__global__ void __launch_bounds__((MT + 1) * 32)
decode_mma_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + NSTAGE * kStageBytes);
  uint64_t* empty_bar = full_bar + NSTAGE;

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
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(smem_u32(full_bar + s), 1);
      mbar_init(smem_u32(empty_bar + s), MT);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == MT) {
    // ---------------- producer warp ----------------
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
    for (int k = 0; k < n_units; ++k) {
      if ((k >> 5) > tbatch) {
        tcur = tnext;
        tnext = table_batch(tbatch + 2);
        ++tbatch;
      }
      const int pid = __shfl_sync(FULL, tcur, k & 31);
      bool ok = true;
      if (lane == 0) {
        const int st = k % NSTAGE;
        if (k >= NSTAGE)
          ok = mbar_wait(smem_u32(empty_bar + st), (uint32_t)(((k / NSTAGE) - 1) & 1), a.status);
        if (ok) {
          const int u = unit0 + k;
          const int slot = (u % upp) * kUnit;
          const uint32_t dst = smem_u32(stages + st * kStageBytes);
          const uint32_t bar = smem_u32(full_bar + st);
          mbar_arrive_expect_tx(bar, kStageBytes);
          tma_load_4d(dst, &tmk, bar, 0, slot, hk, pid);
          tma_load_4d(dst + kBoxBytes, &tmk, bar, 64, slot, hk, pid);
          tma_load_4d(dst + 2 * kBoxBytes, &tmv, bar, 0, slot, hk, pid);
          tma_load_4d(dst + 3 * kBoxBytes, &tmv, bar, 64, slot, hk, pid);
        }
      }
      if (!__shfl_sync(FULL, (int)ok, 0)) break;
    }
    return;
  }

  // ---------------- consumer warps: one 16-row tile each ----------------
  const int g4 = lane >> 2, t4 = lane & 3;
  const int rA = warp * 16 + g4, rB = rA + 8;
  const bool tile_active = warp * 16 < rows_b;

  int loA = 0, hiA = 0x7fffffff, loB = 0, hiB = 0x7fffffff;
  if (rA < rows_b) row_key_range(kv_len, L, rA / G, a.causal, a.window_left, loA, hiA);
  if (rB < rows_b) row_key_range(kv_len, L, rB / G, a.causal, a.window_left, loB, hiB);

  // Q A-fragments for the 8 k-steps of D = 128
  uint32_t qa[8][4];
  {
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* srcA = nullptr;
    const __nv_bfloat16* srcB = nullptr;
    if (rA < rows_b)
      srcA = qb + (int64_t)(rq.q_start + rA / G) * a.q_stride_tok +
             (int64_t)(hk * G + rA % G) * a.q_stride_head;
    if (rB < rows_b)
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

  float acc[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  float mA = neg_inf(), mB = neg_inf(), lA = 0.f, lB = 0.f;
  const float sl2 = a.scale_log2;

  // ldmatrix row addresses: lane i supplies row (i & 7) of matrix (i >> 3)
  const int lm_mat = lane >> 3, lm_row = lane & 7;

  for (int k = 0; k < n_units; ++k) {
    const int st = k % NSTAGE;
    if (!mbar_wait(smem_u32(full_bar + st), (uint32_t)((k / NSTAGE) & 1), a.status)) break;
    const uint8_t* ks_base = stages + st * kStageBytes;
    const uint32_t k_u32 = smem_u32(ks_base);
    const uint32_t v_u32 = k_u32 + 2 * kBoxBytes;
    if (tile_active) {
      // ---- S = Q K^T : two n-tiles of 8 keys ----
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {   // pairs of k-steps: chunks 4kp .. 4kp+3
          uint32_t b0, b1, b2, b3;
          const int key = nt * 8 + lm_row;
          const int cg = kp * 4 + lm_mat;
          ldmatrix_x4(k_u32 + unit_chunk_offset(key, cg), b0, b1, b2, b3);
          mma_bf16_16816(s[nt], qa[2 * kp], b0, b1);
          mma_bf16_16816(s[nt], qa[2 * kp + 1], b2, b3);
        }
      }
      // ---- mask + online softmax (base 2) ----
      const int tok0 = (unit0 + k) * kUnit;
      const bool full_unit = tok0 >= all_lo && tok0 + kUnit <= all_hi;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v = s[nt][c] * sl2;
          if (!full_unit) {
            const int tok = tok0 + nt * 8 + t4 * 2 + (c & 1);
            const bool rowB = c >= 2;
            const int lo = rowB ? loB : loA, hi = rowB ? hiB : hiA;
            if (tok < lo || tok >= hi) v = neg_inf();
          }
          s[nt][c] = v;
        }
      float pmA = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float pmB = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      pmA = fmaxf(pmA, __shfl_xor_sync(FULL, pmA, 1));
      pmA = fmaxf(pmA, __shfl_xor_sync(FULL, pmA, 2));
      pmB = fmaxf(pmB, __shfl_xor_sync(FULL, pmB, 1));
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
      if (__any_sync(FULL, alA != 1.f || alB != 1.f)) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          acc[n][0] *= alA;
          acc[n][1] *= alA;
          acc[n][2] *= alB;
          acc[n][3] *= alB;
        }
      }
      uint32_t pa[4];
      pa[0] = float2_to_bf16x2(s[0][0], s[0][1]);
      pa[1] = float2_to_bf16x2(s[0][2], s[0][3]);
      pa[2] = float2_to_bf16x2(s[1][0], s[1][1]);
      pa[3] = float2_to_bf16x2(s[1][2], s[1][3]);
      // ---- O += P V : 16 n-tiles of 8 dims ----
#pragma unroll
      for (int np = 0; np < 8; ++np) {   // pairs of d-chunks 2np, 2np+1
        uint32_t b0, b1, b2, b3;
        const int key = (lm_mat & 1) * 8 + lm_row;
        const int cg = np * 2 + (lm_mat >> 1);
        ldmatrix_x4_trans(v_u32 + unit_chunk_offset(key, cg), b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * np], pa, b0, b1);
        mma_bf16_16816(acc[2 * np + 1], pa, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty_bar + st));
  }

  if (!tile_active) return;
  lA += __shfl_xor_sync(FULL, lA, 1);
  lA += __shfl_xor_sync(FULL, lA, 2);
  lB += __shfl_xor_sync(FULL, lB, 1);
  lB += __shfl_xor_sync(FULL, lB, 2);

  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rB : rA;
    if (r >= rows_b) continue;
    const float m = half ? mB : mA;
    const float l = half ? lB : lA;
    const int i = r / G, h = hk * G + r % G;
    const int t = rq.q_start + i;
    if (rq.part_base < 0) {
      float denom = l;
      if (a.sinks != nullptr && m != neg_inf()) denom += ex2(__ldg(a.sinks + h) * kLog2e - m);
      const float sc = denom > 0.f ? a.bmm2_scale / denom : 0.f;
      __nv_bfloat16* dst = out + ((int64_t)t * a.num_qo_heads + h) * 128 + t4 * 2;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        *reinterpret_cast<uint32_t*>(dst + n * 8) =
            float2_to_bf16x2(acc[n][2 * half] * sc, acc[n][2 * half + 1] * sc);
      if (a.lse != nullptr && t4 == 0)
        a.lse[(int64_t)t * a.num_qo_heads + h] = l > 0.f ? m + log2f(l) : neg_inf();
    } else {
      const int64_t prow = rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h;
      const float sc = l > 0.f ? 1.f / l : 0.f;
      float* dst = a.ws_o + prow * 128 + t4 * 2;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        *reinterpret_cast<float2*>(dst + n * 8) =
            make_float2(acc[n][2 * half] * sc, acc[n][2 * half + 1] * sc);
      if (t4 == 0) a.ws_lse[prow] = l > 0.f ? m + log2f(l) : neg_inf();
    }
  }
}

template <int MT, int NSTAGE>
int launch_mma(const DecodeArgs& args, const CUtensorMap& kmap, const CUtensorMap& vmap,
               cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)NSTAGE * kStageBytes + 2 * NSTAGE * 8;
  auto kern = decode_mma_kernel<MT, NSTAGE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_mma)");
  kern<<<args.num_items, (MT + 1) * 32, smem, stream>>>(args, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_mma_kernel launch");
  return PKA_OK;
}

}  // namespace

int launch_decode_mma(const pka_plan& plan, const DecodeArgs& args, const CUtensorMap& kmap,
                      const CUtensorMap& vmap, cudaStream_t stream) {
  const int mt = (plan.rows_per_cta + 15) / 16;
  switch (mt) {
    case 1: return launch_mma<1, 8>(args, kmap, vmap, stream);
    case 2: return launch_mma<2, 8>(args, kmap, vmap, stream);
    case 3: return launch_mma<3, 8>(args, kmap, vmap, stream);
    default: return launch_mma<4, 8>(args, kmap, vmap, stream);
  }
}

}  // namespace pka
