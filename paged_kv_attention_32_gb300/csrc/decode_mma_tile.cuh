// One warp's share of the tensor-core decode: a 16-row query tile (or, with
// MmaTileWarpT, up to 8 rows on the instruction's narrow side) against a
// stream of 16-token K/V units staged in shared memory by TMA.
//
// Rows of a tile are r = i*group + g (token i of the request, head g of the
// KV head's group), as cudnn_batch_decode_with_kv_cache's q_len_per_req rows
// with their GQA heads.  Per unit:
//   S = Q K^T          (mma.sync m16n8k16: 2 n-tiles of 8 keys x 8 k-steps,
//                       Q kept as A fragments in registers)
//   mask               (causal diagonal kv_len - q_len + i, window_left)
//   online softmax     (base 2, the scale folded into one multiply; the
//                       reference max moves only when a row max passes it
//                       by more than 2^8, found by one warp vote per unit)
//   O += P V           (P re-packed to A fragments of the input type, V via
//                       ldmatrix.trans)
// A unit is four 2 KB blocks with 128-byte swizzle: K columns 0-63, K 64-127,
// V 0-63, V 64-127, each 16 tokens x 128 bytes.  q/K/V are bf16 or IEEE half.
#pragma once

#include "device_common.cuh"

namespace pka {
namespace dev {

constexpr int kMmaUnitTok = 16;
constexpr int kMmaBoxBytes = 2048;
constexpr int kMmaUnitBytes = 4 * kMmaBoxBytes;
constexpr int kMmaCombStride = 136;   // floats per row of a merge buffer (padded)

// Keys [lo, hi) that query row i of a request sees.
__device__ __forceinline__ void mma_row_key_range(int kv_len, int q_len, int i, int causal,
                                                  int window, int& lo, int& hi) {
  const int d = kv_len - q_len + i;
  hi = causal ? d + 1 : kv_len;
  lo = window >= 0 ? max(0, d - window) : 0;
}

// Byte offset of 16-byte chunk cg (0..15 over the 128 dims) of token j in a
// K or V half of a unit.
__device__ __forceinline__ uint32_t mma_unit_chunk_offset(int j, int cg) {
  return (uint32_t)(cg >> 3) * kMmaBoxBytes + swz128((uint32_t)j, (uint32_t)(cg & 7));
}

// F16: q/K/V are IEEE half (else bf16); P is packed in the same type.
template <bool F16>
struct MmaTileWarp {
  uint32_t qa[8][4];    // Q A fragments, k-step ks
  float acc[16][4];     // O accumulators, 16 n-tiles of 8 dims
  float mA, mB, lA, lB; // running max / sum of rows g4 and g4 + 8
  int loA, hiA, loB, hiB;

  // Loads the tile's query rows (rows past rows_b are zero and see no key).
  __device__ __forceinline__ void init(const DecodeArgs& a, const ReqInfo& rq, int kv_len, int hk,
                                       int tile, int lane) {
    const int G = a.group, L = rq.q_len, rows_b = G * L;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int rA = tile * 16 + g4, rB = rA + 8;
    loA = 0; hiA = 0x7fffffff; loB = 0; hiB = 0x7fffffff;
    if (rA < rows_b) mma_row_key_range(kv_len, L, rA / G, a.causal, a.window_left, loA, hiA);
    if (rB < rows_b) mma_row_key_range(kv_len, L, rB / G, a.causal, a.window_left, loB, hiB);
    const uint16_t* qb = static_cast<const uint16_t*>(a.q);   // 16-bit elements
    const uint16_t* srcA = nullptr;
    const uint16_t* srcB = nullptr;
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
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    mA = mB = neg_inf();
    lA = lB = 0.f;
  }

  // One 16-token unit: K at k_u32, V at k_u32 + 2 boxes; its first token is
  // tok0; full_unit = every row of the tile sees all 16 keys.
  __device__ __forceinline__ void step(uint32_t k_u32, int tok0, bool full_unit, float sl2,
                                       int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    const uint32_t v_u32 = k_u32 + 2 * kMmaBoxBytes;
    const int t4 = lane & 3, lm_mat = lane >> 3, lm_row = lane & 7;
    // S = Q K^T; even and odd k-steps accumulate separately, so four chains
    // of four dependent mma run side by side.
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
        ldmatrix_x4(k_u32 + mma_unit_chunk_offset(nt * 8 + lm_row, kp * 4 + lm_mat), b0, b1, b2,
                    b3);
        mma_16816<F16>(s[nt], qa[2 * kp], b0, b1);
        mma_16816<F16>(s2[nt], qa[2 * kp + 1], b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[nt][c] += s2[nt][c];
    // mask + online softmax (base 2)
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
    // lazy reference: the quad max is taken only when some lane's own max
    // passes its row's reference by more than 2^8 (one vote otherwise)
    float pmA = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float pmB = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    float alA = 1.f, alB = 1.f;
    if (__any_sync(FULL, pmA > mA + 8.f || pmB > mB + 8.f)) {
      pmA = fmaxf(pmA, __shfl_xor_sync(FULL, pmA, 1));
      pmB = fmaxf(pmB, __shfl_xor_sync(FULL, pmB, 1));
      pmA = fmaxf(pmA, __shfl_xor_sync(FULL, pmA, 2));
      pmB = fmaxf(pmB, __shfl_xor_sync(FULL, pmB, 2));
      const bool gA = pmA > mA + 8.f, gB = pmB > mB + 8.f;
      const float mAn = gA ? pmA : mA, mBn = gB ? pmB : mB;
      if (gA) alA = ex2(mA - mAn);
      if (gB) alB = ex2(mB - mBn);
      mA = mAn;
      mB = mBn;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        acc[n][0] *= alA;
        acc[n][1] *= alA;
        acc[n][2] *= alB;
        acc[n][3] *= alB;
      }
    }
    const float uA = mA == neg_inf() ? 0.f : mA, uB = mB == neg_inf() ? 0.f : mB;
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
    uint32_t pa[4];
    pa[0] = pack2<F16>(s[0][0], s[0][1]);
    pa[1] = pack2<F16>(s[0][2], s[0][3]);
    pa[2] = pack2<F16>(s[1][0], s[1][1]);
    pa[3] = pack2<F16>(s[1][2], s[1][3]);
    // O += P V : 16 n-tiles of 8 dims
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(v_u32 + mma_unit_chunk_offset((lm_mat & 1) * 8 + lm_row,
                                                      np * 2 + (lm_mat >> 1)),
                        b0, b1, b2, b3);
      mma_16816<F16>(acc[2 * np], pa, b0, b1);
      mma_16816<F16>(acc[2 * np + 1], pa, b2, b3);
    }
  }

  // Sums l over the quad of lanes that share a row.
  __device__ __forceinline__ void reduce_l() {
    constexpr unsigned FULL = 0xffffffffu;
    lA += __shfl_xor_sync(FULL, lA, 1);
    lA += __shfl_xor_sync(FULL, lA, 2);
    lB += __shfl_xor_sync(FULL, lB, 1);
    lB += __shfl_xor_sync(FULL, lB, 2);
  }

  // Writes (O, m, l) of the 16 rows to merge slot `slot` of the buffers
  // comb_o [slots][16][kMmaCombStride], comb_m / comb_l [slots][16].
  __device__ __forceinline__ void store_comb(float* comb_o, float* comb_m, float* comb_l, int slot,
                                             int lane) const {
    const int g4 = lane >> 2, t4 = lane & 3;
    float* oA = comb_o + (slot * 16 + g4) * kMmaCombStride + t4 * 2;
    float* oB = oA + 8 * kMmaCombStride;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      *reinterpret_cast<float2*>(oA + n * 8) = make_float2(acc[n][0], acc[n][1]);
      *reinterpret_cast<float2*>(oB + n * 8) = make_float2(acc[n][2], acc[n][3]);
    }
    if (t4 == 0) {
      comb_m[slot * 16 + g4] = mA;
      comb_l[slot * 16 + g4] = lA;
      comb_m[slot * 16 + g4 + 8] = mB;
      comb_l[slot * 16 + g4 + 8] = lB;
    }
  }
};

// The same warp step for a tile of at most 8 query rows, with the two
// contractions transposed so that the keys fill the 16-row side of
// m16n8k16 and the query rows its 8-column side:
//   S^T = K Q^T     (K as the A operand from the unit, Q^T as B fragments in
//                    registers: 8 mma per unit instead of 16)
//   O^T += V^T P^T  (V^T via ldmatrix.trans as A, P^T as B: 8 mma, one per 16
//                    dims, instead of 16)
// Lane (g4, t4) holds the scores of keys g4 and g4 + 8 for rows 2 t4 and
// 2 t4 + 1; P^T goes from that C layout to the B layout with one movmatrix
// transpose per 8 keys.  Row maxima and sums run across the 8 lanes of a t4.
template <bool F16>
struct MmaTileWarpT {
  uint32_t qb[8][2];    // Q^T B fragments, k-step ks
  float acc[8][4];      // O^T: dims m*16 + g4 (+ 8) x rows 2 t4, 2 t4 + 1
  float mA, mB, lA, lB; // running max / sum of rows 2 t4 (A) and 2 t4 + 1 (B)
  int loA, hiA, loB, hiB;

  __device__ __forceinline__ void init(const DecodeArgs& a, const ReqInfo& rq, int kv_len, int hk,
                                       int tile, int lane) {
    const int G = a.group, L = rq.q_len, rows_b = G * L;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int r0 = tile * 16;   // the tile's first row (its live rows are at most 8)
    const int rA = r0 + 2 * t4, rB = rA + 1;
    loA = 0; hiA = 0x7fffffff; loB = 0; hiB = 0x7fffffff;
    if (rA < rows_b) mma_row_key_range(kv_len, L, rA / G, a.causal, a.window_left, loA, hiA);
    if (rB < rows_b) mma_row_key_range(kv_len, L, rB / G, a.causal, a.window_left, loB, hiB);
    // B fragment of k-step ks: Q[row g4][dims ks*16 + 2 t4 (+1)] and [.. + 8 (+9)]
    const uint16_t* qp = static_cast<const uint16_t*>(a.q);
    const uint16_t* src = nullptr;
    if (r0 + g4 < rows_b)
      src = qp + (int64_t)(rq.q_start + (r0 + g4) / G) * a.q_stride_tok +
            (int64_t)(hk * G + (r0 + g4) % G) * a.q_stride_head;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c0 = ks * 16 + t4 * 2;
      qb[ks][0] = src ? __ldg(reinterpret_cast<const uint32_t*>(src + c0)) : 0u;
      qb[ks][1] = src ? __ldg(reinterpret_cast<const uint32_t*>(src + c0 + 8)) : 0u;
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
    mA = mB = neg_inf();
    lA = lB = 0.f;
  }

  __device__ __forceinline__ void step(uint32_t k_u32, int tok0, bool full_unit, float sl2,
                                       int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    const uint32_t v_u32 = k_u32 + 2 * kMmaBoxBytes;
    const int g4 = lane >> 2, lm_mat = lane >> 3, lm_row = lane & 7;
    // S^T = K Q^T: even and odd k-steps in two chains
    float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t ka[4];
      // matrices: keys 0-7 / 8-15 (lm_mat & 1) x dims ks*16 + 0-7 / 8-15 (lm_mat >> 1)
      ldmatrix_x4(k_u32 + mma_unit_chunk_offset((lm_mat & 1) * 8 + lm_row, 2 * ks + (lm_mat >> 1)),
                  ka[0], ka[1], ka[2], ka[3]);
      mma_16816<F16>((ks & 1) ? s2 : s, ka, qb[ks][0], qb[ks][1]);
    }
    // c: keys g4 (c < 2) or g4 + 8, rows A (even c) or B
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v = (s[c] + s2[c]) * sl2;
      if (!full_unit) {
        const int tok = tok0 + g4 + (c >= 2 ? 8 : 0);
        const int lo = (c & 1) ? loB : loA, hi = (c & 1) ? hiB : hiA;
        if (tok < lo || tok >= hi) v = neg_inf();
      }
      s[c] = v;
    }
    float pmA = fmaxf(s[0], s[2]), pmB = fmaxf(s[1], s[3]);
    float alA = 1.f, alB = 1.f;
    if (__any_sync(FULL, pmA > mA + 8.f || pmB > mB + 8.f)) {
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        pmA = fmaxf(pmA, __shfl_xor_sync(FULL, pmA, x));
        pmB = fmaxf(pmB, __shfl_xor_sync(FULL, pmB, x));
      }
      const bool gA = pmA > mA + 8.f, gB = pmB > mB + 8.f;
      const float mAn = gA ? pmA : mA, mBn = gB ? pmB : mB;
      if (gA) alA = ex2(mA - mAn);
      if (gB) alB = ex2(mB - mBn);
      mA = mAn;
      mB = mBn;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        acc[m][0] *= alA;
        acc[m][1] *= alB;
        acc[m][2] *= alA;
        acc[m][3] *= alB;
      }
    }
    const float uA = mA == neg_inf() ? 0.f : mA, uB = mB == neg_inf() ? 0.f : mB;
    const float p0 = ex2(s[0] - uA), p1 = ex2(s[1] - uB), p2 = ex2(s[2] - uA), p3 = ex2(s[3] - uB);
    lA = lA * alA + (p0 + p2);
    lB = lB * alB + (p1 + p3);
    // P^T in C layout (keys x rows) -> B layout (rows g4 x keys 2 t4 ..)
    const uint32_t b0 = movmatrix_trans(pack2<F16>(p0, p1));
    const uint32_t b1 = movmatrix_trans(pack2<F16>(p2, p3));
    // O^T += V^T P^T: one m-tile of 16 dims per mma
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      uint32_t va[4];
      // matrices: dims m*16 + 0-7 / 8-15 (lm_mat & 1) x keys 0-7 / 8-15 (lm_mat >> 1)
      ldmatrix_x4_trans(v_u32 + mma_unit_chunk_offset((lm_mat >> 1) * 8 + lm_row, 2 * m + (lm_mat & 1)),
                        va[0], va[1], va[2], va[3]);
      mma_16816<F16>(acc[m], va, b0, b1);
    }
  }

  // Sums l over the 8 lanes that share a row.
  __device__ __forceinline__ void reduce_l() {
    constexpr unsigned FULL = 0xffffffffu;
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      lA += __shfl_xor_sync(FULL, lA, x);
      lB += __shfl_xor_sync(FULL, lB, x);
    }
  }

  // Writes (O, m, l) of the tile's rows 0-7 to merge slot `slot` (layout of
  // store_comb).
  __device__ __forceinline__ void store_comb(float* comb_o, float* comb_m, float* comb_l, int slot,
                                             int lane) const {
    const int g4 = lane >> 2, t4 = lane & 3;
    float* oA = comb_o + (slot * 16 + 2 * t4) * kMmaCombStride + g4;
    float* oB = oA + kMmaCombStride;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      oA[m * 16] = acc[m][0];
      oB[m * 16] = acc[m][1];
      oA[m * 16 + 8] = acc[m][2];
      oB[m * 16 + 8] = acc[m][3];
    }
    if (g4 == 0) {
      comb_m[slot * 16 + 2 * t4] = mA;
      comb_l[slot * 16 + 2 * t4] = lA;
      comb_m[slot * 16 + 2 * t4 + 1] = mB;
      comb_l[slot * 16 + 2 * t4 + 1] = lB;
    }
  }
};

// Combines merge slots [slot0, slot0 + nslots) for row `row` of tile `tile`
// (dims d0 .. d0+15) and writes the final O (out_dtype) and base-2 LSE (sink added
// to the denominator, bmm2_scale applied) or, for a split request, the fp32
// partial (O/l, m + log2 l) of chunk `chunk`.
__device__ __forceinline__ void mma_combine_store(const DecodeArgs& a, const ReqInfo& rq,
                                                  const float* comb_o, const float* comb_m,
                                                  const float* comb_l, int slot0, int nslots,
                                                  int tile, int row, int d0, int hk, int chunk) {
  const int G = a.group, L = rq.q_len;
  const int r = tile * 16 + row;
  if (r >= G * L) return;
  float m = neg_inf();
  for (int w = 0; w < nslots; ++w) m = fmaxf(m, comb_m[(slot0 + w) * 16 + row]);
  float o[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) o[x] = 0.f;
  float lsum = 0.f;
  if (m != neg_inf()) {
    for (int w = 0; w < nslots; ++w) {
      const float mw = comb_m[(slot0 + w) * 16 + row];
      if (mw == neg_inf()) continue;
      const float f = ex2(mw - m);
      lsum += comb_l[(slot0 + w) * 16 + row] * f;
      const float* src = comb_o + ((slot0 + w) * 16 + row) * kMmaCombStride + d0;
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
    store_out<16>(a.out, ((int64_t)t * a.num_qo_heads + h) * 128 + d0, o, sc, a.out_dtype);
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

}  // namespace dev
}  // namespace pka
