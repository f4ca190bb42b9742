// The LSE merge of split decode requests, done inside the decode kernels: the
// chunk CTAs of one (request, KV head, tile) group each write their fp32
// partial rows (O / l and the base-2 LSE m + log2 l) and count themselves on
// a counter of the group; the CTA that counts last merges the group's rows.
// (The partial states of one row are combined as the LSE convention of
// cudnn_batch_decode_with_kv_cache describes: weights 2^(lse_i - m) with m
// the largest LSE, the sink added once to the denominator.)  This saves a
// second kernel launch that would have to wait for the whole decode grid.
#pragma once

#include "device_common.cuh"

namespace pka {
namespace dev {

// The merge of rows r0 .. r0 + nrows - 1 by one CTA of 128 threads: TPR
// threads per row, each owning 128 / TPR dims, with the loads of KR chunks in
// flight per round (16 float4 per thread whatever TPR is), in one pass with a
// running maximum.  A chunk without keys has LSE -inf: weight 0.
template <int TPR>
__device__ __forceinline__ void merge_rows(const DecodeArgs& a, const ReqInfo& rq, int hk, int r0,
                                           int nrows) {
  constexpr int DPT = 128 / TPR, KR = 64 / DPT, NV = DPT / 4;
  const int rr = threadIdx.x / TPR, d0 = (threadIdx.x % TPR) * DPT;
  if (rr >= nrows) return;
  const int G = a.group, r = r0 + rr;
  const int i = r / G, h = hk * G + r % G;
  const int nc = rq.n_chunks;
  const int64_t stride_c = (int64_t)rq.q_len * a.num_qo_heads;
  const int64_t p0 = rq.part_base + (int64_t)i * a.num_qo_heads + h;
  float m = neg_inf(), wsum = 0.f;
  float o[DPT];
#pragma unroll
  for (int x = 0; x < DPT; ++x) o[x] = 0.f;
  for (int c0 = 0; c0 < nc; c0 += KR) {
    float lc[KR];
    float4 v[KR][NV];
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const int64_t p = p0 + (c0 + k) * stride_c;
      const bool in = c0 + k < nc;
      lc[k] = in ? __ldcg(a.ws_lse + p) : neg_inf();
      const float4* src = reinterpret_cast<const float4*>(a.ws_o + p * 128 + d0);
#pragma unroll
      for (int x = 0; x < NV; ++x)
        v[k][x] = in ? __ldcg(src + x) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m_new = m;
#pragma unroll
    for (int k = 0; k < KR; ++k) m_new = fmaxf(m_new, lc[k]);
    if (m_new == neg_inf()) continue;   // no keys so far
    const float sc = ex2(m - m_new);    // 0 while m is still -inf
    m = m_new;
    wsum *= sc;
#pragma unroll
    for (int x = 0; x < DPT; ++x) o[x] *= sc;
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const float w = lc[k] == neg_inf() ? 0.f : ex2(lc[k] - m);
      wsum += w;
#pragma unroll
      for (int x = 0; x < NV; ++x) {
        o[4 * x] += w * v[k][x].x;
        o[4 * x + 1] += w * v[k][x].y;
        o[4 * x + 2] += w * v[k][x].z;
        o[4 * x + 3] += w * v[k][x].w;
      }
    }
  }
  float denom = wsum;
  if (a.sinks != nullptr && m != neg_inf()) denom += ex2(__ldg(a.sinks + h) * kLog2e - m);
  const float sc = denom > 0.f ? a.bmm2_scale / denom : 0.f;
  const int64_t t = rq.q_start + i;
  store_out<DPT>(a.out, (t * a.num_qo_heads + h) * 128 + d0, o, sc, a.out_dtype);
  if (a.lse != nullptr && d0 == 0)
    a.lse[t * a.num_qo_heads + h] = wsum > 0.f ? m + log2f(wsum) : neg_inf();
}

// Called by every thread of a CTA (128 threads) of a split request after the
// CTA wrote its partial rows r0 .. r0 + nrows - 1 (nrows <= 16) of the work
// item (row r = i * group + g: token i, head hk * group + g).  Returns at once
// unless this CTA is the group's last; that CTA resets the group's counter to
// zero (every chunk has counted) and writes the final O (out_dtype,
// bmm2_scale) and LSE of the rows.
__device__ __forceinline__ void split_merge_if_last(const DecodeArgs& a, const ReqInfo& rq, int hk,
                                                    int tile, int r0, int nrows) {
  __shared__ int s_last;
  // The CTA's partial writes happen before thread 0's count (barrier), and the
  // count is an acquire-release atomic at GPU scope: it publishes them (fences
  // are cumulative), and the last count acquires every earlier CTA's writes,
  // which the barrier below hands on to the CTA's other threads.
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t* cnt = a.merge_cnt + rq.cnt_base + hk * a.tiles_per_item + tile;
    int32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(cnt) : "memory");
    const bool last = old == rq.n_chunks - 1;
    if (last) *cnt = 0;   // every chunk has counted: ready for the next run
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  // a group of at most 8 rows with a long chunk list: 16 threads per row and
  // 8 chunks per round (fewer rounds of memory latency); else 8 threads per
  // row and 4 chunks per round
  if (rq.n_chunks > 8 && nrows <= 8) merge_rows<16>(a, rq, hk, r0, nrows);
  else merge_rows<8>(a, rq, hk, r0, nrows);
}

}  // namespace dev
}  // namespace pka
