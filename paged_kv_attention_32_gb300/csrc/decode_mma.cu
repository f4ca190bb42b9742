// Paged decode attention, tensor-core variant for wide query groups
// ((Hq/Hkv) * max_q_len >= 16 rows per KV head by default, e.g. speculative
// packed-Q verification with cudnn_batch_decode_with_kv_cache's
// q_len_per_req rows).
//
// Same work items, masks, softmax and outputs as the CUDA-core kernel; the
// two contractions run on mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//  * a CTA handles one 16-row tile of the item's query rows (row r = i*group
//    + g: token i, head g of the group); blockIdx.x = item * MT + tile, so
//    the MT tiles of one item run side by side and all but the first read its
//    K/V pages from L2;
//  * its four warps each stream their own 16-token units (w, w+4, ...) with
//    TMA into a private NSTAGE-deep ring (128-byte swizzle keeps ldmatrix
//    conflict-free), exactly as in the CUDA-core kernel;
//  * per unit: S = Q K^T (2 n-tiles x 8 k-steps, Q in A-fragment registers),
//    mask, online softmax in base 2 on the fragments, P re-packed to bf16
//    A fragments in registers, O += P V (16 n-tiles, V via ldmatrix.trans);
//  * the four warps' (m, l, O) are merged through shared memory and the CTA
//    writes final O/LSE (sink added) or an fp32 partial for the merge kernel.
// Decode is bound by HBM, not by the tensor pipe: mma takes the per-key
// arithmetic of wide groups off the FP32 pipe.
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
constexpr int kCombStride = 136;   // floats per row of the merge buffer (padded)

__device__ __forceinline__ void row_key_range(int kv_len, int q_len, int i, int causal, int window,
                                              int& lo, int& hi) {
  const int d = kv_len - q_len + i;
  hi = causal ? d + 1 : kv_len;
  lo = window >= 0 ? max(0, d - window) : 0;
}

__device__ __forceinline__ uint32_t unit_chunk_offset(int j, int cg) {
  return (uint32_t)(cg >> 3) * kBoxBytes + swz128((uint32_t)j, (uint32_t)(cg & 7));
}

template <int NSTAGE>
__global__ void __launch_bounds__(kWarps * 32, 3)
decode_mma_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * NSTAGE * kStageBytes);

  const int mt_count = (a.rows_per_cta + 15) >> 4;
  const int item_idx = blockIdx.x / mt_count, mt = blockIdx.x % mt_count;
  const WorkItem it = a.items[item_idx];
  const int b = it.request;
  const ReqInfo rq = a.reqs[b];
  const int L = rq.q_len, G = a.group;
  const int rows_b = G * L;
  if (mt * 16 >= rows_b) return;   // the whole CTA: this request has fewer rows

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hk = it.head_chunk & 0xffff;
  const int chunk = it.head_chunk >> 16;
  int kv_len = rq.kv_len;
  if (a.seq_lens_live != nullptr) kv_len = max(min(__ldg(a.seq_lens_live + b), rq.kv_len), L);
  const int upp = a.page_size / kUnit;

  int lo_first, hi_first, lo_last, hi_last;
  row_key_range(kv_len, L, 0, a.causal, a.window_left, lo_first, hi_first);
  row_key_range(kv_len, L, L - 1, a.causal, a.window_left, lo_last, hi_last);
  const int unit0 = max(it.page_lo * upp, lo_first / kUnit);
  const int unit1 = min(it.page_hi * upp, (hi_last + kUnit - 1) / kUnit);
  const int n_units = max(0, unit1 - unit0);
  const int all_lo = lo_last, all_hi = hi_first;

  if (tid == 0) {
    for (int i = 0; i < kWarps * NSTAGE; ++i) mbar_init(smem_u32(bars + i), 1);
    fence_barrier_init();
  }
  if (tid == 32) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  __syncthreads();

  // ---- this lane's two rows of the 16-row tile ----
  const int g4 = lane >> 2, t4 = lane & 3;
  const int rA = mt * 16 + g4, rB = rA + 8;
  int loA = 0, hiA = 0x7fffffff, loB = 0, hiB = 0x7fffffff;
  if (rA < rows_b) row_key_range(kv_len, L, rA / G, a.causal, a.window_left, loA, hiA);
  if (rB < rows_b) row_key_range(kv_len, L, rB / G, a.causal, a.window_left, loB, hiB);

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
  const int lm_mat = lane >> 3, lm_row = lane & 7;

  // ---- per-warp TMA pipeline over units warp, warp+4, ... ----
  const int my_units = n_units > warp ? (n_units - warp + kWarps - 1) / kWarps : 0;
  uint8_t* my_stages = stages + warp * NSTAGE * kStageBytes;
  const uint32_t stage_u32 = smem_u32(my_stages);
  const uint32_t bar_u32 = smem_u32(bars + warp * NSTAGE);
  const int32_t* trow = a.block_tables + (int64_t)b * a.bt_row_stride;
  auto table_batch = [&](int batch) -> int {
    const int k = batch * 32 + lane;
    if (k < my_units) return __ldg(trow + (unit0 + warp + k * kWarps) / upp);
    return 0;
  };
  int tcur = table_batch(0), tnext = table_batch(1), tbatch = 0;
  auto issue = [&](int k) {
    if ((k >> 5) > tbatch) {
      tcur = tnext;
      tnext = table_batch(tbatch + 2);
      ++tbatch;
    }
    const int pid = __shfl_sync(FULL, tcur, k & 31);
    if (lane == 0) {
      const int u = unit0 + warp + k * kWarps;
      const int slot = (u % upp) * kUnit;
      const int st = k % NSTAGE;
      const uint32_t dst = stage_u32 + st * kStageBytes, bar = bar_u32 + st * 8;
      mbar_arrive_expect_tx(bar, kStageBytes);
      tma_load_4d(dst, &tmk, bar, 0, slot, hk, pid);
      tma_load_4d(dst + kBoxBytes, &tmk, bar, 64, slot, hk, pid);
      tma_load_4d(dst + 2 * kBoxBytes, &tmv, bar, 0, slot, hk, pid);
      tma_load_4d(dst + 3 * kBoxBytes, &tmv, bar, 64, slot, hk, pid);
    }
  };
  const int pre = my_units < NSTAGE ? my_units : NSTAGE;
  for (int k = 0; k < pre; ++k) issue(k);

  for (int k = 0; k < my_units; ++k) {
    const int st = k % NSTAGE;
    if (!__all_sync(FULL, mbar_wait(bar_u32 + st * 8, (uint32_t)((k / NSTAGE) & 1), a.status)))
      break;
    const uint32_t k_u32 = stage_u32 + st * kStageBytes;
    const uint32_t v_u32 = k_u32 + 2 * kBoxBytes;
    // ---- S = Q K^T : two n-tiles of 8 keys; even and odd k-steps accumulate
    // separately, so four chains of four dependent mma run side by side ----
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
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[nt][c] += s2[nt][c];
    // ---- mask + online softmax (base 2) ----
    const int tok0 = (unit0 + warp + k * kWarps) * kUnit;
    const bool full_unit = tok0 >= all_lo && tok0 + kUnit <= all_hi;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v = s[nt][c] * sl2;
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
    for (int np = 0; np < 8; ++np) {
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(v_u32 + unit_chunk_offset((lm_mat & 1) * 8 + lm_row, np * 2 + (lm_mat >> 1)),
                        b0, b1, b2, b3);
      mma_bf16_16816(acc[2 * np], pa, b0, b1);
      mma_bf16_16816(acc[2 * np + 1], pa, b2, b3);
    }
    __syncwarp();
    if (k + NSTAGE < my_units) issue(k + NSTAGE);
  }

  lA += __shfl_xor_sync(FULL, lA, 1);
  lA += __shfl_xor_sync(FULL, lA, 2);
  lB += __shfl_xor_sync(FULL, lB, 1);
  lB += __shfl_xor_sync(FULL, lB, 2);

  // ---- merge the four warps through shared memory ----
  __syncthreads();   // every warp is done with its stages
  float* comb_o = reinterpret_cast<float*>(stages);              // [warps][16][kCombStride]
  float* comb_m = comb_o + kWarps * 16 * kCombStride;            // [warps][16]
  float* comb_l = comb_m + kWarps * 16;                          // [warps][16]
  {
    float* oA = comb_o + (warp * 16 + g4) * kCombStride + t4 * 2;
    float* oB = oA + 8 * kCombStride;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      *reinterpret_cast<float2*>(oA + n * 8) = make_float2(acc[n][0], acc[n][1]);
      *reinterpret_cast<float2*>(oB + n * 8) = make_float2(acc[n][2], acc[n][3]);
    }
    if (t4 == 0) {
      comb_m[warp * 16 + g4] = mA;
      comb_l[warp * 16 + g4] = lA;
      comb_m[warp * 16 + g4 + 8] = mB;
      comb_l[warp * 16 + g4 + 8] = lB;
    }
  }
  __syncthreads();

  // thread -> (row of the tile, 16 consecutive dims)
  const int row = tid >> 3, d0 = (tid & 7) * 16;
  const int r = mt * 16 + row;
  if (r >= rows_b) return;
  float m = neg_inf();
#pragma unroll
  for (int w = 0; w < kWarps; ++w) m = fmaxf(m, comb_m[w * 16 + row]);
  float o[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) o[x] = 0.f;
  float lsum = 0.f;
  if (m != neg_inf()) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = comb_m[w * 16 + row];
      if (mw == neg_inf()) continue;
      const float f = ex2(mw - m);
      lsum += comb_l[w * 16 + row] * f;
      const float* src = comb_o + (w * 16 + row) * kCombStride + d0;
#pragma unroll
      for (int x = 0; x < 16; x += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + x);
        o[x] += v.x * f;
        o[x + 1] += v.y * f;
        o[x + 2] += v.z * f;
        o[x + 3] += v.w * f;
      }
    }
  }
  const int i = r / G, h = hk * G + r % G;
  const int t = rq.q_start + i;
  if (rq.part_base < 0) {
    float denom = lsum;
    if (a.sinks != nullptr && m != neg_inf()) denom += ex2(__ldg(a.sinks + h) * kLog2e - m);
    const float sc = denom > 0.f ? a.bmm2_scale / denom : 0.f;
    uint4 w0, w1;
    w0.x = float2_to_bf16x2(o[0] * sc, o[1] * sc);
    w0.y = float2_to_bf16x2(o[2] * sc, o[3] * sc);
    w0.z = float2_to_bf16x2(o[4] * sc, o[5] * sc);
    w0.w = float2_to_bf16x2(o[6] * sc, o[7] * sc);
    w1.x = float2_to_bf16x2(o[8] * sc, o[9] * sc);
    w1.y = float2_to_bf16x2(o[10] * sc, o[11] * sc);
    w1.z = float2_to_bf16x2(o[12] * sc, o[13] * sc);
    w1.w = float2_to_bf16x2(o[14] * sc, o[15] * sc);
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                          ((int64_t)t * a.num_qo_heads + h) * 128 + d0);
    dst[0] = w0;
    dst[1] = w1;
    if (a.lse != nullptr && d0 == 0)
      a.lse[(int64_t)t * a.num_qo_heads + h] = lsum > 0.f ? m + log2f(lsum) : neg_inf();
  } else {
    const int64_t prow = rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h;
    const float sc = lsum > 0.f ? 1.f / lsum : 0.f;
    float4* dst = reinterpret_cast<float4*>(a.ws_o + prow * 128 + d0);
#pragma unroll
    for (int x = 0; x < 4; ++x)
      dst[x] = make_float4(o[4 * x] * sc, o[4 * x + 1] * sc, o[4 * x + 2] * sc, o[4 * x + 3] * sc);
    if (d0 == 0) a.ws_lse[prow] = lsum > 0.f ? m + log2f(lsum) : neg_inf();
  }
}

template <int NSTAGE>
int launch_mma(const DecodeArgs& args, const CUtensorMap& kmap, const CUtensorMap& vmap,
               cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)kWarps * NSTAGE * kStageBytes + kWarps * NSTAGE * 8;
  static_assert(kWarps * 16 * (kCombStride + 2) * 4 <= kWarps * NSTAGE * kStageBytes,
                "merge buffer does not fit in the stage area");
  auto kern = decode_mma_kernel<NSTAGE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_mma)");
  const int mt = (args.rows_per_cta + 15) / 16;
  const int64_t grid = (int64_t)args.num_items * mt;
  if (grid > 0x7fffffff) return fail(PKA_ERR_INVALID_ARG, "decode grid too large");
  kern<<<(unsigned)grid, kWarps * 32, smem, stream>>>(args, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_mma_kernel launch");
  return PKA_OK;
}

}  // namespace

int launch_decode_mma(const pka_plan& plan, const DecodeArgs& args, const CUtensorMap& kmap,
                      const CUtensorMap& vmap, cudaStream_t stream) {
  (void)plan;
  return launch_mma<2>(args, kmap, vmap, stream);
}

}  // namespace pka
