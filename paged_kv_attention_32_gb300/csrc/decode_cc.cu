// Paged decode attention, CUDA-core variant (FFMA2 + warp shuffles), for
// groups of up to 8 query rows per KV head when the plan's mma_min_rows is set
// above them (the tensor-core variant, decode_mma.cu, is the default).
//
// Computes, for every query row of one (request, KV head, key chunk) work
// item, softmax(scale * q K^T) V over the keys the row may see
// (cudnn_batch_decode_with_kv_cache: q_len_per_req causal rows, window_left,
// sinks, the base-2 "LSE convention"; batch_decode_with_paged_kv_cache:
// block_tables page addressing).
//
// Design (GB300):
//  * one CTA per work item, four warps; the whole GQA group of query rows
//    (group * q_len <= 8) sits in every warp's registers, pre-scaled by
//    scale * log2(e) so that the softmax runs on exp2;
//  * the item's keys are cut into 16-token units; warp w owns units
//    w, w+4, ...  Each warp streams its units through its own ring of
//    NSTAGE shared-memory stages with TMA tensor loads (one 4 KB copy each
//    for K and V, stored as two 64-column halves, 128-byte swizzle)
//    completing on an mbarrier; the page id of each unit comes from block_tables,
//    prefetched 32 units ahead into registers;
//  * q.k: 2R lanes share one key, each holding 64/R of its 128 dims; the R
//    partial dot products are reduced with a halving butterfly (R shuffles
//    per lane) whose row order is pre-permuted per lane, so no selects are
//    needed;  p = exp2(s - m) with a running max per row (online softmax);
//  * p.v: the same lanes accumulate p * v for all R rows over their dims;
//    probabilities go through a 16 x R shared buffer;
//  * the four warps' (m, l, acc) are merged through shared memory; the CTA
//    then writes the final O (bf16, f16 or fp32) and LSE (sink added here), or an fp32
//    partial (O/l, m + log2 l) when the request was split; the chunk CTA of
//    a (request, KV head) that finishes last merges the partials.
#include <cuda_bf16.h>

#include "decode_merge.cuh"
#include "device_common.cuh"
#include "host_common.h"
#include "kernels.h"

namespace pka {

using namespace dev;

namespace {

constexpr int kWarps = 4;
constexpr int kUnit = 16;            // tokens per TMA unit
constexpr int kStageBytes = 8192;    // K (4 KB) + V (4 KB) of one unit
constexpr int kBoxBytes = 2048;      // 16 rows x 128 bytes

__device__ __forceinline__ void row_key_range(int kv_len, int q_len, int i, int causal, int window,
                                              int& lo, int& hi) {
  const int d = kv_len - q_len + i;   // the row's diagonal key
  hi = causal ? d + 1 : kv_len;
  lo = window >= 0 ? max(0, d - window) : 0;
}

// Byte offset of 16-byte chunk `cg` (0..15, i.e. dims 8cg..8cg+7) of unit row `j`
// inside a K or V unit: two 2 KB boxes (dims 0-63, 64-127), 128-byte swizzle.
__device__ __forceinline__ uint32_t unit_chunk_offset(int j, int cg) {
  return (uint32_t)(cg >> 3) * kBoxBytes + swz128((uint32_t)j, (uint32_t)(cg & 7));
}

// F16: q/K/V are IEEE half (else bf16).
template <int R, int NSTAGE, bool F16>
__global__ void __launch_bounds__(128, 2)
decode_cc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
  constexpr int LK = 2 * R;       // lanes per key
  constexpr int KS = 32 / LK;     // keys per warp step
  constexpr int DL = 64 / R;      // dims per lane
  constexpr int NCH = DL / 8;     // 16-byte chunks per lane
  constexpr int NSTEP = kUnit / KS;
  constexpr unsigned FULL = 0xffffffffu;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* pbuf = reinterpret_cast<float*>(smem + kWarps * NSTAGE * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(pbuf + kWarps * kUnit * R);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kslot = lane / LK, e = lane % LK;

  const WorkItem it = a.items[blockIdx.x];
  const int b = it.request;
  const int hk = it.head_chunk & 0xffff;
  const int chunk = it.head_chunk >> 16;
  const ReqInfo rq = a.reqs[b];
  const int L = rq.q_len, G = a.group;
  int kv_len = rq.kv_len;
  if (a.seq_lens_live != nullptr) kv_len = max(min(__ldg(a.seq_lens_live + b), rq.kv_len), L);
  const int rows_b = G * L;
  const int upp = a.page_size / kUnit;   // units per page

  // keys visible to any row: [lo of row 0, hi of row L-1)
  int lo_first, hi_first, lo_last, hi_last;
  row_key_range(kv_len, L, 0, a.causal, a.window_left, lo_first, hi_first);
  row_key_range(kv_len, L, L - 1, a.causal, a.window_left, lo_last, hi_last);
  const int unit0 = max(it.page_lo * upp, lo_first / kUnit);
  const int unit1 = min(it.page_hi * upp, (hi_last + kUnit - 1) / kUnit);
  const int n_units = max(0, unit1 - unit0);
  // a unit needs no mask when every valid row sees all of its keys
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

  // the row whose score this lane ends up holding after the butterfly
  const int my_row = (e >> 1) & (R - 1);
  int my_lo = 0, my_hi = 0x7fffffff;   // padding rows are left unmasked (their output is dropped)
  if (my_row < rows_b) row_key_range(kv_len, L, my_row / G, a.causal, a.window_left, my_lo, my_hi);

  // ---- q in registers, slot s holding row s ^ my_row, scaled by scale*log2(e) ----
  float2 q2[R][DL / 2];
  {
    const uint16_t* qb = static_cast<const uint16_t*>(a.q);   // 16-bit elements
#pragma unroll
    for (int s = 0; s < R; ++s) {
      const int r = s ^ my_row;
      if (r < rows_b) {
        const int t = rq.q_start + r / G, h = hk * G + r % G;
        const uint16_t* src = qb + (int64_t)t * a.q_stride_tok + (int64_t)h * a.q_stride_head;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int cg = e + c * LK;
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(src + cg * 8));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            float2 f = unpack2<F16>(ws[x]);
            q2[s][c * 4 + x] = make_float2(f.x * a.scale_log2, f.y * a.scale_log2);
          }
        }
      } else {
#pragma unroll
        for (int x = 0; x < DL / 2; ++x) q2[s][x] = make_float2(0.f, 0.f);
      }
    }
  }

  float2 acc[R][DL / 2];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int x = 0; x < DL / 2; ++x) acc[r][x] = make_float2(0.f, 0.f);
  float m_run = neg_inf(), l_run = 0.f;

  // ---- per-warp TMA pipeline ----
  const int my_units = n_units > warp ? (n_units - warp + kWarps - 1) / kWarps : 0;
  uint8_t* my_stages = stages + warp * NSTAGE * kStageBytes;
  const uint32_t stage_u32 = smem_u32(my_stages);
  const uint32_t bar_u32 = smem_u32(bars + warp * NSTAGE);
  const int32_t* trow = a.block_tables + (int64_t)b * a.bt_row_stride;
  auto table_batch = [&](int batch) -> int {
    const int k = batch * 32 + lane;
    if (k < my_units) {
      const int u = unit0 + warp + k * kWarps;
      return __ldg(trow + u / upp);
    }
    return 0;
  };
  int tcur = table_batch(0), tnext = table_batch(1), tbatch = 0;
  auto issue = [&](int k) {
    if ((k >> 5) > tbatch) {   // entering the prefetched batch: rotate, prefetch the next
      tcur = tnext;
      tnext = table_batch(tbatch + 2);
      ++tbatch;
    }
    const int pid = __shfl_sync(FULL, tcur, k & 31);
    const int u = unit0 + warp + k * kWarps;
    const int slot = (u % upp) * kUnit;
    const int st = k % NSTAGE;
    const uint32_t dst = stage_u32 + st * kStageBytes, bar = bar_u32 + st * 8;
    if constexpr (!F16) {
      tma_load_kv_pair_elect(dst, dst + 2 * kBoxBytes, &tmk, &tmv, bar, kStageBytes, slot, hk,
                             pid);
    } else if (lane == 0) {
      // measured: the fp16 instantiation runs ~1 % faster with the copies issued
      // as separate statements from lane 0 (the bf16 one ~0.7 % slower)
      mbar_arrive_expect_tx(bar, kStageBytes);
      tma_load_kv_unit(dst, &tmk, bar, slot, hk, pid);
      tma_load_kv_unit(dst + 2 * kBoxBytes, &tmv, bar, slot, hk, pid);
    }
  };
  const int pre = my_units < NSTAGE ? my_units : NSTAGE;
  for (int k = 0; k < pre; ++k) issue(k);

  float* pw = pbuf + warp * kUnit * R;
  int k = 0;
  for (; k < my_units; ++k) {
    const int st = k % NSTAGE;
    // same outcome in every lane: the shuffles below need the whole warp
    if (!__all_sync(FULL, mbar_wait(bar_u32 + st * 8, (uint32_t)((k / NSTAGE) & 1), a.status)))
      break;
    const uint8_t* ks = my_stages + st * kStageBytes;
    const uint8_t* vs = ks + 2 * kBoxBytes;
    const int tok0 = (unit0 + warp + k * kWarps) * kUnit;
    const bool full_unit = tok0 >= all_lo && tok0 + kUnit <= all_hi;

    // scores of this lane's row for keys s*KS + kslot
    float sv[NSTEP];
#pragma unroll
    for (int s = 0; s < NSTEP; ++s) {
      const int j = s * KS + kslot;
      float2 k2[DL / 2];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(ks + unit_chunk_offset(j, e + c * LK));
        k2[c * 4 + 0] = unpack2<F16>(w.x);
        k2[c * 4 + 1] = unpack2<F16>(w.y);
        k2[c * 4 + 2] = unpack2<F16>(w.z);
        k2[c * 4 + 3] = unpack2<F16>(w.w);
      }
      float part[R];
#pragma unroll
      for (int sl = 0; sl < R; ++sl) {
        float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int x = 0; x < DL / 2; ++x) d2 = ffma2(q2[sl][x], k2[x], d2);
        part[sl] = d2.x + d2.y;
      }
      // halving butterfly over the 2R lanes of this key
#pragma unroll
      for (int cnt = R; cnt > 1; cnt >>= 1) {
#pragma unroll
        for (int jj = 0; jj < cnt / 2; ++jj)
          part[jj] += __shfl_xor_sync(FULL, part[jj + cnt / 2], cnt);
      }
      float sc = part[0] + __shfl_xor_sync(FULL, part[0], 1);
      if (!full_unit) {
        const int tok = tok0 + j;
        if (tok < my_lo || tok >= my_hi) sc = neg_inf();
      }
      sv[s] = sc;
    }

    // online softmax update (base 2)
    float pm = sv[0];
#pragma unroll
    for (int s = 1; s < NSTEP; ++s) pm = fmaxf(pm, sv[s]);
#pragma unroll
    for (int delta = LK; delta < 32; delta <<= 1) pm = fmaxf(pm, __shfl_xor_sync(FULL, pm, delta));
    const float m_new = fmaxf(m_run, pm);
    const float m_use = (m_new == neg_inf()) ? 0.f : m_new;
    const float alpha = ex2(m_run - m_use);
    float psum = 0.f;
#pragma unroll
    for (int s = 0; s < NSTEP; ++s) {
      sv[s] = ex2(sv[s] - m_use);
      psum += sv[s];
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
    if (__any_sync(FULL, alpha != 1.f)) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float ar = __shfl_sync(FULL, alpha, 2 * r);
#pragma unroll
        for (int x = 0; x < DL / 2; ++x) acc[r][x] = fmul2(acc[r][x], make_float2(ar, ar));
      }
    }
    if ((e & 1) == 0) {
#pragma unroll
      for (int s = 0; s < NSTEP; ++s) pw[(s * KS + kslot) * R + my_row] = sv[s];
    }
    __syncwarp();

    // acc[r] += p[r, j] * v_j over this lane's dims
#pragma unroll
    for (int s = 0; s < NSTEP; ++s) {
      const int j = s * KS + kslot;
      float pr[R];
#pragma unroll
      for (int r4 = 0; r4 < R; r4 += 4) {
        const float4 p4 = *reinterpret_cast<const float4*>(pw + j * R + r4);
        pr[r4 + 0] = p4.x;
        pr[r4 + 1] = p4.y;
        pr[r4 + 2] = p4.z;
        pr[r4 + 3] = p4.w;
      }
      float2 v2[DL / 2];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(vs + unit_chunk_offset(j, e + c * LK));
        v2[c * 4 + 0] = unpack2<F16>(w.x);
        v2[c * 4 + 1] = unpack2<F16>(w.y);
        v2[c * 4 + 2] = unpack2<F16>(w.z);
        v2[c * 4 + 3] = unpack2<F16>(w.w);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float2 pp = make_float2(pr[r], pr[r]);
#pragma unroll
        for (int x = 0; x < DL / 2; ++x) acc[r][x] = ffma2(pp, v2[x], acc[r][x]);
      }
    }
    __syncwarp();
    if (k + NSTAGE < my_units) issue(k + NSTAGE);
  }
  // a wait gave up: let the copies still in flight land (bounded) before the
  // stages are reused or the CTA exits
  for (int j = k; j < my_units && j < k + NSTAGE; ++j)
    (void)mbar_wait(bar_u32 + (j % NSTAGE) * 8, (uint32_t)((j / NSTAGE) & 1), a.status);

  // ---- reduce over the key slots of the warp ----
#pragma unroll
  for (int delta = LK; delta < 32; delta <<= 1) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int x = 0; x < DL / 2; ++x) {
        acc[r][x].x += __shfl_xor_sync(FULL, acc[r][x].x, delta);
        acc[r][x].y += __shfl_xor_sync(FULL, acc[r][x].y, delta);
      }
    l_run += __shfl_xor_sync(FULL, l_run, delta);
  }

  // ---- merge the four warps through shared memory ----
  __syncthreads();   // every warp is done with its stages
  float* comb_o = reinterpret_cast<float*>(stages);          // [warps][R][128]
  float* comb_m = comb_o + kWarps * R * 128;                 // [warps][R]
  float* comb_l = comb_m + kWarps * R;                       // [warps][R]
  if (kslot == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int cg = e + c * LK;
        float4* dst = reinterpret_cast<float4*>(comb_o + (warp * R + r) * 128 + cg * 8);
        dst[0] = make_float4(acc[r][c * 4 + 0].x, acc[r][c * 4 + 0].y, acc[r][c * 4 + 1].x,
                             acc[r][c * 4 + 1].y);
        dst[1] = make_float4(acc[r][c * 4 + 2].x, acc[r][c * 4 + 2].y, acc[r][c * 4 + 3].x,
                             acc[r][c * 4 + 3].y);
      }
    if ((e & 1) == 0) {
      comb_m[warp * R + my_row] = m_run;
      comb_l[warp * R + my_row] = l_run;
    }
  }
  __syncthreads();

  const int d = tid;   // 128 threads <-> 128 dims
  for (int r = 0; r < rows_b && r < R; ++r) {
    float m = neg_inf();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) m = fmaxf(m, comb_m[w * R + r]);
    float lsum = 0.f, o = 0.f;
    if (m != neg_inf()) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = comb_m[w * R + r];
        if (mw == neg_inf()) continue;
        const float f = ex2(mw - m);
        lsum += comb_l[w * R + r] * f;
        o += comb_o[(w * R + r) * 128 + d] * f;
      }
    }
    const int i = r / G, h = hk * G + r % G;
    const int t = rq.q_start + i;
    if (rq.part_base < 0) {
      float denom = lsum;
      if (a.sinks != nullptr && m != neg_inf()) denom += ex2(__ldg(a.sinks + h) * kLog2e - m);
      const float ov = denom > 0.f ? a.bmm2_scale * o / denom : 0.f;
      store_out1(a.out, ((int64_t)t * a.num_qo_heads + h) * 128 + d, ov, a.out_dtype);
      if (a.lse != nullptr && d == 0)
        a.lse[(int64_t)t * a.num_qo_heads + h] = lsum > 0.f ? m + log2f(lsum) : neg_inf();
    } else {
      const int64_t prow = rq.part_base + ((int64_t)chunk * L + i) * a.num_qo_heads + h;
      a.ws_o[prow * 128 + d] = lsum > 0.f ? o / lsum : 0.f;
      if (d == 0) a.ws_lse[prow] = lsum > 0.f ? m + log2f(lsum) : neg_inf();
    }
  }
  if (rq.part_base >= 0)   // a split request: the group's last chunk merges its rows
    split_merge_if_last(a, rq, hk, 0, 0, min(rows_b, R));
}

template <int R, int NSTAGE, bool F16>
int launch_cc(const DecodeArgs& args, const CUtensorMap& kmap, const CUtensorMap& vmap,
              cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)kWarps * NSTAGE * kStageBytes +
                      (size_t)kWarps * kUnit * R * sizeof(float) + kWarps * NSTAGE * 8;
  static_assert(kWarps * R * 130 * 4 <= kWarps * NSTAGE * kStageBytes, "combine area too small");
  auto kern = decode_cc_kernel<R, NSTAGE, F16>;
  static std::atomic<uint64_t> smem_set{0};   // devices whose limit this launcher raised
  cudaError_t e = set_smem_once(kern, (int)smem, smem_set);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode_cc)");
  kern<<<args.num_items, 128, smem, stream>>>(args, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_cc_kernel launch");
  return PKA_OK;
}

}  // namespace

int launch_decode_mma(const pka_plan& plan, const DecodeArgs& args, const CUtensorMap& kmap,
                      const CUtensorMap& vmap, cudaStream_t stream);

int launch_decode(const pka_plan& plan, const DecodeArgs& args, const CUtensorMap& kmap,
                  const CUtensorMap& vmap, cudaStream_t stream) {
  int rc;
  if (plan.kernel == PKA_KERNEL_MMA) {
    rc = launch_decode_mma(plan, args, kmap, vmap, stream);
  } else if (plan.rows_per_cta <= 4) {
    rc = args.in_f16 ? launch_cc<4, 3, true>(args, kmap, vmap, stream)
                     : launch_cc<4, 3, false>(args, kmap, vmap, stream);
  } else {
    rc = args.in_f16 ? launch_cc<8, 3, true>(args, kmap, vmap, stream)
                     : launch_cc<8, 3, false>(args, kmap, vmap, stream);
  }
  if (rc != PKA_OK) return rc;
  return PKA_OK;
}

}  // namespace pka
