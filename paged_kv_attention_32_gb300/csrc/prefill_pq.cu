// Prefill for head_dim 128 on the 5th-generation tensor cores: persistent
// CTAs (one per SM), Q held in tensor memory.
//
// Each 64-key step of the one-head-per-CTA design reads, through the shared
// memory port, Q (the A operand of S = Q K^T, 32 KB), K and V (the B operands,
// 16 KB each) and the TMA writes of the next K and V (32 KB).  Measured on the
// GB300 that port is saturated (31.8 of 32 bank accesses per cycle), so this
// kernel takes Q out of it: Q sits in TMEM, and S = Q K^T is a TS MMA (A from
// TMEM), which leaves K, V and their copies, 64 KB per step instead of 96.
// With TMEM to spare for a deeper S queue the tensor core can compute S up to
// three key tiles ahead of the softmax, and the queue also covers a tile
// change: the softmax warps write the output of one tile while the tensor
// core already computes the first scores of the next.
//
// One CTA per SM walks the plan's tiles (128 query rows of one request and
// one query head each, heaviest first) in a snake order over the CTAs.  Roles:
//   warps 0-7  softmax: warp w owns the query rows of TMEM lane quarter w % 4
//              and half w / 4 of each 64-key tile (32 keys) and of O (64
//              columns); the two warps of a quarter trade their partial row
//              maxima through shared memory (one named barrier per quarter),
//              so both take the same lazy-rescale decision (rescale O only
//              when the max grew by more than 2^8).  p = exp2, P (16-bit)
//              over the first 32 columns of the S slot, the final O / l and
//              LSE; between tiles they copy the next tile's Q from shared
//              memory into TMEM and write the finished tile's O;
//   warp 8     TMA: Q tiles (two staging buffers) and K tiles;
//   warp 9     TMA: V tiles;
//   warp 10    allocates TMEM and issues every tcgen05.mma (one elected
//              lane, four chained k-steps per asm block).
// TMEM (512 columns): S slots [0, 256) (4 x 64), O [256, 384), Q buffers
// [384, 448) and [448, 512) (two tiles' Q, bf16 pairs per column).
#include <cstdlib>
#include <string>

#include <cuda_bf16.h>

#include "device_common.cuh"
#include "host_common.h"
#include "prefill.h"
#include "prefill_softmax.cuh"
#include "tcgen05.cuh"

namespace pka {

using namespace dev;

namespace {

constexpr int kTileQ = 128, kTileK = 64, kD = 128;
constexpr uint32_t kQBox = 16384;              // 128 rows x 128 bytes (64 columns)
constexpr uint32_t kKBox = 8192;               // 64 rows x 128 bytes
constexpr uint32_t kQStage = 2 * kQBox;        // one tile's Q (two column blocks)
constexpr uint32_t kKVStage = 2 * kKBox;       // one K or V tile
constexpr int kSoftmaxWarps = 8, kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kWarpK = 8, kWarpV = 9, kWarpMma = 10;
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kXBytes = (2 * 2 + 2) * 128 * 4;     // row max [parity][half][row], sum [half][row]

// Shared memory: two Q staging buffers (each also the output staging of the
// tile before the one whose Q it held), NK K stages, NV V stages, barriers,
// the row-max / row-sum exchange.  TMEM: NS S slots of 64 columns, O, two Q
// buffers.
template <int NS, int NK, int NV>
struct PqLayout {
  static constexpr uint32_t kColO = NS * 64, kColQ = kColO + kD;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + 2 * kQStage;
  static constexpr uint32_t kOffV = kOffK + NK * kKVStage;
  static constexpr uint32_t kOffBar = kOffV + NV * kKVStage;
  static constexpr uint32_t kOffX = kOffBar + 512;
  static constexpr size_t kSmemBytes = 1024 + kOffX + kXBytes;
  static_assert(kColQ + 2 * 64 <= 512, "TMEM columns");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

template <bool F16> constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, 0, 0, F16);
template <bool F16> constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kD, 0, 1, F16);

// K tile (64 keys x 128 dims) as the K-major B operand of k-step kk.
__device__ __forceinline__ uint64_t kmajor_b(uint32_t base, int kk) {
  return smem_desc_sw128(base + (uint32_t)(kk >> 2) * kKBox + (uint32_t)(kk & 3) * 32u, 16u,
                         1024u);
}
// V tile (64 keys x 128 dims) as the MN-major B operand, k-step kk = keys 16kk..
__device__ __forceinline__ uint64_t vmn(uint32_t base, int kk) {
  return smem_desc_sw128(base + (uint32_t)kk * 2048u, kKBox, 1024u);
}

// Named barrier of the two softmax warps of one TMEM lane quarter (ids 1-4):
// both warps arrive, and each gets the AND of `v` over the 64 threads.  Every
// bounded wait of these warps is followed by one, so that a wait that gave up
// makes both warps of the pair leave together (a lone warp would otherwise
// wait at the next barrier with no partner).
__device__ __forceinline__ bool pair_all(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, 64, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

// Row max of 32 scores as four independent chains.
__device__ __forceinline__ float row_max32(const uint32_t* r) {
  float mq[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
#pragma unroll
  for (int i = 0; i < 32; i += 2)
    mq[(i >> 1) & 3] = fmax3(mq[(i >> 1) & 3], __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
  return fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
}

// Scores of keys outside [lo, lo + span) (r: keys key0 .. key0 + 31) to -inf.
__device__ __forceinline__ void mask_scores32(uint32_t* r, int key0, int lo, unsigned span) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if ((unsigned)(key0 + i - lo) >= span) r[i] = __float_as_uint(neg_inf());
}

// p = exp2(s * sl2 - m) for 32 scores (keys key0 .. key0 + 31), packed two
// per 32-bit TMEM column into the 16 columns at p_tm; returns the sum of p.
// MASKED: keys outside [lo, lo + span) give p = 0 (see exp_tile).
template <bool MASKED, bool F16>
__device__ __forceinline__ float exp_half(const uint32_t* r, float sl2, float neg_m, int key0,
                                          int lo, unsigned span, uint32_t p_tm) {
  const float2 sc = make_float2(sl2, sl2), nm = make_float2(neg_m, neg_m);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 x =
        __ffma2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc, nm);
    float2 p = make_float2(ex2(x.x), ex2(x.y));
    if constexpr (MASKED) {
      if ((unsigned)(key0 + 2 * i - lo) >= span) p.x = 0.f;
      if ((unsigned)(key0 + 2 * i + 1 - lo) >= span) p.y = 0.f;
    }
    if (i & 1) acc1 = __fadd2_rn(acc1, p);
    else acc0 = __fadd2_rn(acc0, p);
    pk[i] = pack2<F16>(p.x, p.y);
  }
  tmem_st16(p_tm, pk);
  const float2 t = __fadd2_rn(acc0, acc1);
  return t.x + t.y;
}

// The plan's tile processed by CTA `cta` (of `ctas`) in its round r, or -1:
// rounds alternate direction so that every CTA gets a similar share of the
// heaviest-first list.
__device__ __forceinline__ int tile_of(int r, int cta, int ctas, int num_tiles) {
  const int idx = r * ctas + ((r & 1) ? ctas - 1 - cta : cta);
  return idx < num_tiles ? idx : -1;
}

// Walks the CTA's tiles and the 64-key steps inside them, in the order every
// role uses (t: local tile count, j: step in the tile, g: step count).  The
// next tile's description is loaded one tile ahead, so that no role waits on
// a global load at a tile change.  The planner gives every tile at least one
// key tile.
struct StepCursor {
  int t = 0, j = 0, g = 0, tile = -1, next = -1;
  PrefillTile cur, nxt;
  __device__ __forceinline__ void start(const PrefillArgs& a) {
    tile = tile_of(0, blockIdx.x, gridDim.x, a.num_tiles);
    next = tile_of(1, blockIdx.x, gridDim.x, a.num_tiles);
    if (tile >= 0) cur = a.tiles[tile];
    if (next >= 0) nxt = a.tiles[next];
  }
  __device__ __forceinline__ bool done() const { return tile < 0; }
  __device__ __forceinline__ void advance(const PrefillArgs& a) {
    ++g;
    if (++j == cur.n_kv) {
      ++t;
      j = 0;
      tile = next;
      cur = nxt;
      next = tile_of(t + 1, blockIdx.x, gridDim.x, a.num_tiles);
      if (next >= 0) nxt = a.tiles[next];
    }
  }
};

template <int NS, int NK, int NV, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
prefill_pq_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using Lay = PqLayout<NS, NK, NV>;
  constexpr uint32_t kColO = Lay::kColO, kColQ = Lay::kColQ;
  constexpr uint32_t kOffQ = Lay::kOffQ, kOffK = Lay::kOffK, kOffV = Lay::kOffV;
  constexpr uint32_t kOffBar = Lay::kOffBar, kOffX = Lay::kOffX;
  // mbarriers.  A parity wait is only correct when the barrier has completed
  // the phase before the awaited one; the argument for each is given where it
  // is waited on.
  constexpr int B_QFULL = 0;               // [2] Q staging buffer b holds tile 2k + b (TMA)
  constexpr int B_QEMPTY = 2;              // [2] staging buffer b may take the next Q (256)
  constexpr int B_QTM = 4;                 // [2] Q of tile 2k + b is in TMEM buffer b (256)
  constexpr int B_KFULL = 6;               // [NK]
  constexpr int B_KEMPTY = B_KFULL + NK;   // [NK] QK of the step that used the stage completed
  constexpr int B_VFULL = B_KEMPTY + NK;   // [NV]
  constexpr int B_VEMPTY = B_VFULL + NV;   // [NV] P V of the step completed
  constexpr int B_SFULL = B_VEMPTY + NV;   // [NS] S of the step is in its slot
  constexpr int B_PFULL = B_SFULL + NS;    // [NS] P of the step is in its slot (256)
  constexpr int B_ODONE = B_PFULL + NS;    // [NS] P V of the step completed
  constexpr int B_OFREE = B_ODONE + NS;    // softmax read O of a finished tile (256)
  constexpr int B_MMADONE = B_OFREE + 1;
  constexpr int B_COUNT = B_MMADONE + 1;
  static_assert(B_COUNT * 8 + 16 <= 512, "barrier area");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + B_COUNT * 8);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_QFULL + b), 1);
      mbar_init(bar(B_QEMPTY + b), kSoftmaxThreads);
      mbar_init(bar(B_QTM + b), kSoftmaxThreads);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), kSoftmaxThreads);
      mbar_init(bar(B_ODONE + s), 1);
    }
    mbar_init(bar(B_OFREE), kSoftmaxThreads);
    mbar_init(bar(B_MMADONE), 1);
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpK) {
    // ---------------- TMA: Q tiles and K tiles ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      // Q of local tile t into staging buffer t & 1.  For t >= 2 the buffer is
      // free once the softmax copied Q of tile t - 2 into TMEM (release number
      // (t >> 1) - 1 of that buffer's QEMPTY; the one after it needs this load).
      auto load_q = [&](int t, const PrefillTile& tl) -> bool {
        const int qb = t & 1;
        if (t >= 2 && !mbar_wait(bar(B_QEMPTY + qb), (uint32_t)(((t >> 1) - 1) & 1), a.status))
          return false;
        const uint32_t dst = sbase + kOffQ + (uint32_t)qb * kQStage;
        mbar_arrive_expect_tx(bar(B_QFULL + qb), kQStage);
        for (int blk = 0; blk < 2; ++blk)
          tma_load_3d(dst + (uint32_t)blk * kQBox, &tmq, bar(B_QFULL + qb), blk * 64, tl.head,
                      tl.q0 + tl.q_tile * kTileQ);
        return true;
      };
      StepCursor c;
      c.start(a);
      bool ok = true;
      int q_loaded = 0;   // Q tiles issued (local tile numbers 0 .. q_loaded - 1)
      int last_k = -1;
      if (!c.done()) {
        ok = load_q(0, c.cur);
        q_loaded = ok;
      }
      while (ok && !c.done()) {
        const int g = c.g, st = g % NK, t = c.t;
        const bool first = c.j == 0;
        if (g >= NK && !mbar_wait(bar(B_KEMPTY + st), (uint32_t)(((g / NK) - 1) & 1), a.status)) {
          ok = false;
          break;
        }
        const PrefillTile& tl = c.cur;
        const uint32_t dst = sbase + kOffK + (uint32_t)st * kKVStage;
        mbar_arrive_expect_tx(bar(B_KFULL + st), kKVStage);
        for (int blk = 0; blk < 2; ++blk)
          tma_load_3d(dst + (uint32_t)blk * kKBox, &tmk, bar(B_KFULL + st), blk * 64,
                      tl.head / a.group, tl.k0 + (tl.kv0 + c.j) * kTileK);
        last_k = g;
        // once the first K tile of tile t is out, Q of tile t + 1
        if (first && c.next >= 0) {
          const PrefillTile nt = c.nxt;
          c.advance(a);
          ok = load_q(t + 1, nt);
          q_loaded += ok;
        } else {
          c.advance(a);
        }
      }
      if (!ok) {   // give the copies already issued a bounded chance to land
        if (q_loaded > 0)
          mbar_wait(bar(B_QFULL + ((q_loaded - 1) & 1)), (uint32_t)(((q_loaded - 1) >> 1) & 1),
                    nullptr);
        if (last_k >= 0)
          mbar_wait(bar(B_KFULL + last_k % NK), (uint32_t)((last_k / NK) & 1), nullptr);
      }
    }
  } else if (warp == kWarpV) {
    // ---------------- TMA: V tiles ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmv);
      StepCursor c;
      c.start(a);
      bool ok = true;
      int last_v = -1;
      while (!c.done()) {
        const int g = c.g, st = g % NV;
        if (g >= NV && !mbar_wait(bar(B_VEMPTY + st), (uint32_t)(((g / NV) - 1) & 1), a.status)) {
          ok = false;
          break;
        }
        const PrefillTile& tl = c.cur;
        const uint32_t dst = sbase + kOffV + (uint32_t)st * kKVStage;
        mbar_arrive_expect_tx(bar(B_VFULL + st), kKVStage);
        for (int blk = 0; blk < 2; ++blk)
          tma_load_3d(dst + (uint32_t)blk * kKBox, &tmv, bar(B_VFULL + st), blk * 64,
                      tl.head / a.group, tl.k0 + (tl.kv0 + c.j) * kTileK);
        last_v = g;
        c.advance(a);
      }
      if (!ok && last_v >= 0)
        mbar_wait(bar(B_VFULL + last_v % NV), (uint32_t)((last_v / NV) & 1), nullptr);
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer ----------------
    // QK of step gq may be issued once P V of step gq - NS was (its S slot then
    // holds nothing the tensor core still reads: tcgen05 MMAs of one thread run
    // in issue order), its K stage is full and its tile's Q is in TMEM.  While
    // some P V is still to issue, QK waits only by polling: the softmax may be
    // waiting for that P V (lazy rescale, end of a tile) before it can produce
    // the Q the next tile's QK needs.
    StepCursor qk, pv;
    qk.start(a);
    pv.start(a);
    bool ok = true;
    while (ok && !pv.done()) {
      while (ok && !qk.done() && qk.g <= pv.g + (NS - 1)) {
        const int g = qk.g, t = qk.t;
        const bool must = qk.g == pv.g;   // nothing else to issue: block
        const uint32_t qtm_bar = bar(B_QTM + (t & 1)), qtm_par = (uint32_t)((t >> 1) & 1);
        const uint32_t k_bar = bar(B_KFULL + g % NK), k_par = (uint32_t)((g / NK) & 1);
        if (must) {
          ok = (qk.j != 0 || warp_wait(qtm_bar, qtm_par, a.status)) &&
               warp_wait(k_bar, k_par, a.status);
          if (!ok) break;
        } else {
          const bool ready =
              __all_sync(0xffffffffu, (qk.j != 0 || mbar_test_wait(qtm_bar, qtm_par)) &&
                                          mbar_test_wait(k_bar, k_par));
          if (!ready) break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(g % NS) * 64u;
        const uint32_t q_tm = tmem + kColQ + (uint32_t)(t & 1) * 64u;
        const uint32_t kb = sbase + kOffK + (uint32_t)(g % NK) * kKVStage;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)   // 4 k-steps of 16 dims per 64-column block
          umma_ts_k4<2>(d, q_tm + 32u * (uint32_t)blk, kmajor_b(kb, 4 * blk), kIdescQK<F16>,
                        blk > 0 ? 1u : 0u);
        umma_commit_elect(bar(B_SFULL + g % NS));
        umma_commit_elect(bar(B_KEMPTY + g % NK));
        qk.advance(a);
      }
      if (!ok) break;
      // P V of step pv.g
      const int g = pv.g, s = g % NS;
      ok = warp_wait(bar(B_VFULL + g % NV), (uint32_t)((g / NV) & 1), a.status) &&
           warp_wait(bar(B_PFULL + s), (uint32_t)((g / NS) & 1), a.status);
      // the first P V of tile t overwrites O: the softmax must have read tile
      // t - 1's O (OFREE completion t - 1; completion t needs this P V)
      if (ok && pv.j == 0 && pv.t > 0)
        ok = warp_wait(bar(B_OFREE), (uint32_t)((pv.t - 1) & 1), a.status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t p_tm = tmem + (uint32_t)s * 64u;   // P: 32 columns, lanes 0-127
      const uint32_t vb = sbase + kOffV + (uint32_t)(g % NV) * kKVStage;
      umma_ts_k4<2048 / 16>(tmem + kColO, p_tm, vmn(vb, 0), kIdescPV<F16>, pv.j > 0 ? 1u : 0u);
      umma_commit_elect(bar(B_ODONE + s));
      umma_commit_elect(bar(B_VEMPTY + g % NV));
      pv.advance(a);
    }
    umma_commit_elect(bar(B_MMADONE));
    warp_wait(bar(B_MMADONE), 0, a.status);   // nothing of ours still runs on the tensor core
  } else {
    // ---------------- softmax: 8 warps, two per TMEM lane quarter ----------------
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;            // query row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t o_tm = tmem + lane_off + kColO + 64u * (uint32_t)half;   // this warp's O half
    const float sl2 = a.scale_log2;                 // >= 0 (checked by the planner)
    float* xmax = reinterpret_cast<float*>(smem + kOffX);     // [2][2][128]
    float* xsum = xmax + 2 * 2 * 128;                         // [2][128]
    bool ok = true;
    // Q of local tile t: staging buffer t & 1 (128-byte swizzle) -> TMEM Q
    // buffer t & 1, bf16 pairs per column (the A operand of QK); this warp
    // copies its rows' column block `half` (dims 64 half .. 64 half + 63).
    auto copy_q = [&](int t) -> bool {
      const int qb = t & 1;
      if (!warp_wait(bar(B_QFULL + qb), (uint32_t)((t >> 1) & 1), a.status))
        return pair_all(1 + quarter, false);
      const uint8_t* src = smem + kOffQ + (uint32_t)qb * kQStage + (uint32_t)half * kQBox;
      uint32_t r[32];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + swz128((uint32_t)row, (uint32_t)cc));
        r[4 * cc] = v.x;
        r[4 * cc + 1] = v.y;
        r[4 * cc + 2] = v.z;
        r[4 * cc + 3] = v.w;
      }
      tmem_st32(tmem + lane_off + kColQ + (uint32_t)qb * 64u + 32u * (uint32_t)half, r);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_QTM + qb));     // QK of tile t may read it
      // the staging buffer may take tile t + 2 now for tile 0; for a later
      // tile it first stages the output of tile t - 1 (released after that)
      if (t == 0) mbar_arrive(bar(B_QEMPTY + qb));
      return pair_all(1 + quarter, true);
    };
    StepCursor c;
    c.start(a);
    if (!c.done()) ok = copy_q(0);
    while (ok && !c.done()) {
      const PrefillTile tl = c.cur;
      const int h = tl.head, mt = tl.q_tile, n_kv = tl.n_kv, kv0 = tl.kv0;
      const int q0 = tl.q0, Lq = tl.lq, Lk = tl.lk;
      const int t_idx = mt * kTileQ + row;
      const bool row_valid = t_idx < Lq;
      int hi = a.causal ? min(Lk, Lk - Lq + t_idx + 1) : Lk;   // keys [lo, hi) visible
      int lo = a.window_left >= 0 ? min(hi, max(0, Lk - Lq + t_idx - a.window_left)) : 0;
      if (a.window_lo != nullptr) {   // variable_window: the row's inclusive bounds
        lo = row_valid ? __ldg(a.window_lo + q0 + t_idx) : 0;
        hi = row_valid ? __ldg(a.window_hi + q0 + t_idx) + 1 : 0;
      }
      const unsigned span = (unsigned)(hi - lo);
      float m_ref = neg_inf(), l = 0.f;
      int g_last = c.g;
      const int t_fin = c.t;
      for (int j = 0; j < n_kv; ++j) {
        const int g = c.g, s = g % NS;
        // SFULL of slot s completes once per step that uses it, in order
        const bool s_ok = warp_wait(bar(B_SFULL + s), (uint32_t)((g / NS) & 1), a.status);
        tc_fence_after();
        const uint32_t s_tm = tmem + lane_off + (uint32_t)s * 64u;
        const int key0 = (kv0 + j) * kTileK + 32 * half;   // this warp's 32 keys
        const bool masked = __any_sync(0xffffffffu, key0 < lo || key0 + 32 > hi);
        uint32_t ra[32];
        float pm = neg_inf();
        float* xm = xmax + (g & 1) * 256;
        if (s_ok) {
          tmem_ld32(s_tm + 32u * (uint32_t)half, ra);
          tmem_wait_ld();
          reg_fence32(ra);
          if (masked) mask_scores32(ra, key0, lo, span);
          pm = row_max32(ra);
          // trade the partial maxima with the other half's warp.  The slot of
          // step g is rewritten at step g + 2, after both warps passed step
          // g + 1's barrier.
          xm[half * 128 + row] = pm;
        }
        if (!(ok = pair_all(1 + quarter, s_ok))) break;
        const float mraw = fmaxf(pm, xm[(1 - half) * 128 + row]);
        // both warps of the pair now hold S in registers: P may overwrite it
        const float mx = mraw == neg_inf() ? neg_inf() : mraw * sl2;
        const bool grow = mx > m_ref + kRescaleThreshold;
        const float m_new = grow ? mx : m_ref;
        const float alpha = grow ? ex2(m_ref - m_new) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // O holds steps before g: wait for P V of step g - 1.  ODONE of its
          // slot completed the phase before (P V of g - 1 - NS): S of step g is
          // full, and QK of g was issued after P V of g - NS.
          const int gp = g - 1;
          ok = warp_wait(bar(B_ODONE + gp % NS), (uint32_t)((gp / NS) & 1), a.status);
          if (!(ok = pair_all(1 + quarter, ok))) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t r[32];
            tmem_ld32_sync(o_tm + (uint32_t)cc * 32u, r);
#pragma unroll
            for (int i2 = 0; i2 < 32; ++i2) r[i2] = __float_as_uint(__uint_as_float(r[i2]) * alpha);
            tmem_st32(o_tm + (uint32_t)cc * 32u, r);
          }
          tmem_wait_st();
        }
        m_ref = m_new;
        const float neg_m = -m_ref;
        const bool zero_again =
            masked && __any_sync(0xffffffffu, !(sl2 > 0.f) || m_ref == neg_inf());
        const uint32_t p_tm = s_tm + 16u * (uint32_t)half;   // P of keys 32 half .. : 16 columns
        const float sum = zero_again ? exp_half<true, F16>(ra, sl2, neg_m, key0, lo, span, p_tm)
                                     : exp_half<false, F16>(ra, sl2, neg_m, key0, lo, span, p_tm);
        tmem_wait_st();
        l = l * alpha + sum;
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + s));
        g_last = g;
        c.advance(a);
      }
      if (!ok) break;
      // the next tile's Q into TMEM first: its QKs run while this tile's O is written
      if (!c.done() && !(ok = copy_q(c.t))) break;
      // the row sum of both halves (the slot is rewritten only after the next
      // tile's barriers).  O is complete once P V of the tile's last step is
      // (the phase before, P V of g_last - NS, completed: S of g_last is full).
      xsum[half * 128 + row] = l;
      ok = warp_wait(bar(B_ODONE + g_last % NS), (uint32_t)((g_last / NS) & 1), a.status);
      if (!(ok = pair_all(1 + quarter, ok))) break;
      const float l_row = l + xsum[(1 - half) * 128 + row];
      tc_fence_after();
      const float inv = l_row > 0.f ? a.output_scale / l_row : 0.f;
      const int stg = (t_fin + 1) & 1;   // staging buffer of Q(t + 1), copied out above
      uint32_t o[2][32];
      tmem_ld32(o_tm, o[0]);
      tmem_ld32(o_tm + 32u, o[1]);
      tmem_wait_ld();
      reg_fence32(o[0]);
      reg_fence32(o[1]);
      tc_fence_before();
      mbar_arrive(bar(B_OFREE));   // the next tile's first P V may overwrite O
      const int64_t row_elem = ((int64_t)(q0 + t_idx) * a.num_qo_heads + h) * kD + 64 * half;
      if (a.out_dtype == PKA_DTYPE_F32) {
        if (row_valid) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int qd = 0; qd < 2; ++qd) {
              float f[16];
#pragma unroll
              for (int x = 0; x < 16; ++x) f[x] = __uint_as_float(o[cc][16 * qd + x]);
              store_out<16>(a.out, row_elem + cc * 32 + qd * 16, f, inv, a.out_dtype);
            }
        }
      } else {
        // 16-bit O: the warp stages its 32 half-rows (128 bytes each, 16-byte
        // chunks XOR-swizzled by row), then writes them back four rows per
        // store instruction (whole 128-byte segments instead of 32 rows per store)
        // this warp's 4 KB of the staging buffer hold the Q rows it copied itself
        uint8_t* wbuf = smem + kOffQ + (uint32_t)stg * kQStage + (uint32_t)warp * 32u * 128u;
        const bool f16o = a.out_dtype == PKA_DTYPE_F16;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float lo_v = __uint_as_float(o[cc][8 * k + 2 * x]) * inv;
              const float hi_v = __uint_as_float(o[cc][8 * k + 2 * x + 1]) * inv;
              w[x] = f16o ? pack2<true>(lo_v, hi_v) : pack2<false>(lo_v, hi_v);
            }
            const int qc = cc * 4 + k;
            *reinterpret_cast<uint4*>(wbuf + lane * 128 + ((qc ^ (lane & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        __syncwarp();
        const int qc = lane & 7;
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += 4) {
          const int rr = r0 + (lane >> 3);
          const int tr = mt * kTileQ + quarter * 32 + rr;
          const uint4 val =
              *reinterpret_cast<const uint4*>(wbuf + rr * 128 + ((qc ^ (rr & 7)) << 4));
          if (tr < Lq)
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) +
                                      (((int64_t)(q0 + tr) * a.num_qo_heads + h) * kD +
                                       64 * half) * 2 + qc * 16) = val;
        }
        __syncwarp();   // the staging rows are read before the next tile writes them
      }
      if (half == 0 && row_valid && a.lse != nullptr)
        a.lse[(int64_t)(q0 + t_idx) * a.num_qo_heads + h] =
            l_row > 0.f ? m_ref + log2f(l_row) : neg_inf();
      // the staging buffer may take the Q of the tile after next (a TMA write:
      // the generic accesses above are ordered before it)
      fence_proxy_async_smem();
      mbar_arrive(bar(B_QEMPTY + stg));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int NS, int NK, int NV>
int launch_pq(const pka_prefill_plan& plan, const PrefillArgs& args, const CUtensorMap& qmap,
              const CUtensorMap& kmap, const CUtensorMap& vmap, int sms, cudaStream_t stream) {
  const bool f16 = plan.desc.dtype == PKA_DTYPE_F16;
  auto kern = f16 ? prefill_pq_kernel<NS, NK, NV, true> : prefill_pq_kernel<NS, NK, NV, false>;
  constexpr size_t smem = PqLayout<NS, NK, NV>::kSmemBytes;
  static std::atomic<uint64_t> smem_set[2];   // per input type: devices whose limit was raised
  cudaError_t e = set_smem_once(kern, (int)smem, smem_set[f16]);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_pq)");
  const int grid = args.num_tiles < sms ? args.num_tiles : sms;
  kern<<<grid, kThreads, smem, stream>>>(args, qmap, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "prefill_pq_kernel launch");
  return PKA_OK;
}

}  // namespace

int launch_prefill_pq(const pka_prefill_plan& plan, const PrefillArgs& args,
                      const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      cudaStream_t stream) {
  if (args.num_tiles == 0) return PKA_OK;
  int dev = 0, sms = 0;
  PKA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  PKA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
               "cudaDeviceGetAttribute(SM count)");
  const char* cfg = std::getenv("PKA_PQ_CFG");
  const std::string c = cfg ? cfg : "";
  if (c == "363") return launch_pq<3, 6, 3>(plan, args, qmap, kmap, vmap, sms, stream);
  if (c == "454") return launch_pq<4, 5, 4>(plan, args, qmap, kmap, vmap, sms, stream);
  if (c == "372") return launch_pq<3, 7, 2>(plan, args, qmap, kmap, vmap, sms, stream);
  if (c == "443") return launch_pq<4, 4, 3>(plan, args, qmap, kmap, vmap, sms, stream);
  return launch_pq<4, 6, 3>(plan, args, qmap, kmap, vmap, sms, stream);
}

}  // namespace pka
