// Prefill for head_dim 128 and an even GQA group: persistent CTAs (one per
// SM), each tile two query heads of one KV head sharing every K and V tile.
//
// On the GB300 the one-head kernel is bound by the shared-memory port: per
// 64-key step it reads Q (the A operand of S = Q K^T, 32 KB), K and V (the
// B operands, 16 KB each) and takes the TMA writes of the next K and V
// (32 KB), 96 KB in all, and ncu counts 31.8 of 32 bank accesses per cycle.
// Two heads of one KV head read the same K and V, so a CTA that runs both
// copies each tile once: 80 KB per head and step instead of 96.  Such a CTA
// needs all 512 TMEM columns (two S buffers and O per head), so one runs per
// SM, and it is persistent: the next tile's Q is loaded during the current
// tile, and the tensor core computes the next tile's first scores while the
// softmax warps write the finished tile's output.
//
// Tiles (128 query rows of one request for heads h, h + 1), heaviest first,
// are walked in a snake order over the CTAs.  Roles:
//   warps 0-7  softmax: warp w takes head w / 4 of the pair and the query rows
//              of TMEM lane quarter w % 4, one thread per row (the one-head
//              kernel's softmax: row max of 64 scores, lazy rescale of O when
//              the max grew by more than 2^8, p = exp2, 16-bit P over the
//              first 32 columns of the S buffer, final O / l and LSE, the
//              output staged through the tile's own, finished Q buffer);
//   warp 8     TMA: Q of both heads (two buffers of 64 KB) and K tiles;
//   warp 9     TMA: V tiles;
//   warp 10    allocates TMEM and issues every tcgen05.mma (one elected
//              lane, four chained k-steps per asm block).
// TMEM: head e at columns 256e: S0 [0, 64), S1 [64, 128), O [128, 256).
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
constexpr int NK = 3, NV = 2;                      // K and V stages
constexpr uint32_t kQBox = 16384;                  // 128 rows x 128 bytes (64 columns)
constexpr uint32_t kKBox = 8192;                   // 64 rows x 128 bytes
constexpr uint32_t kQHead = 2 * kQBox;             // one head's Q tile
constexpr uint32_t kQStage = 2 * kQHead;           // both heads
constexpr uint32_t kKVStage = 2 * kKBox;           // one K or V tile
constexpr int kSoftmaxThreads = 256;
constexpr int kWarpK = 8, kWarpV = 9, kWarpMma = 10;
constexpr int kThreads = 32 * 11;
constexpr float kRescaleThreshold = 8.0f;

constexpr uint32_t kOffQ = 0;                          // two Q buffers
constexpr uint32_t kOffK = kOffQ + 2 * kQStage;
constexpr uint32_t kOffV = kOffK + NK * kKVStage;
constexpr uint32_t kOffBar = kOffV + NV * kKVStage;
constexpr size_t kSmemBytes = 1024 + kOffBar + 512;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// mbarriers.  A parity wait is only correct when the barrier has completed
// the phase before the awaited one; the argument for each is given where it
// is waited on.
enum {
  B_QFULL = 0,                 // [2] Q buffer b holds local tile 2k + b (TMA, tx bytes)
  B_QEMPTY = 2,                // [2] tile 2k + b's output left buffer b (256 arrivals)
  B_KFULL = 4,                 // [NK]
  B_KEMPTY = B_KFULL + NK,     // [NK] both QKs of the step that used the stage completed
  B_VFULL = B_KEMPTY + NK,     // [NV]
  B_VEMPTY = B_VFULL + NV,     // [NV] both P Vs of the step completed
  B_SFULL = B_VEMPTY + NV,     // [head][slot] S of the step is in its buffer
  B_PFULL = B_SFULL + 4,       // [head][slot] P of the step (128 arrivals)
  B_ODONE = B_PFULL + 4,       // [head][slot] P V of the step completed
  B_OFREE = B_ODONE + 4,       // [head] the softmax read a finished tile's O (128 arrivals)
  B_MMADONE = B_OFREE + 2,
  B_COUNT = B_MMADONE + 1
};
static_assert(B_COUNT * 8 + 16 <= 512, "barrier area");

template <bool F16> constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, 0, 0, F16);
template <bool F16> constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kD, 0, 1, F16);

// Q (128 rows) or K (64 rows) as the K-major operand of k-step kk: column
// block kk / 4, 32-byte step kk % 4 inside the 128-byte rows.
__device__ __forceinline__ uint64_t kmajor(uint32_t base, uint32_t block_bytes, int kk) {
  return smem_desc_sw128(base + (uint32_t)(kk >> 2) * block_bytes + (uint32_t)(kk & 3) * 32u, 16u,
                         1024u);
}
// V tile (64 keys x 128 dims) as the MN-major B operand, k-step kk = keys 16kk..
__device__ __forceinline__ uint64_t vmn(uint32_t base, int kk) {
  return smem_desc_sw128(base + (uint32_t)kk * 2048u, kKBox, 1024u);
}

// Non-blocking test of a barrier phase (try_wait may suspend the thread for a
// while before it answers "not yet").
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The plan's tile processed by CTA `cta` (of `ctas`) in its round r, or -1:
// rounds alternate direction so that every CTA gets a similar share of the
// heaviest-first list.
__device__ __forceinline__ int tile_of(int r, int cta, int ctas, int num_tiles) {
  const int idx = r * ctas + ((r & 1) ? ctas - 1 - cta : cta);
  return idx < num_tiles ? idx : -1;
}

// Walks the CTA's tiles and the 64-key steps inside them, in the order every
// role uses (t: local tile count, j: step in the tile, g: step count), with
// the next tile's description loaded one tile ahead.  Every tile has at least
// one key tile (the planner checks it).
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

template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
prefill_gh_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
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
      mbar_init(bar(B_OFREE + b), 128);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), 128);
      mbar_init(bar(B_ODONE + s), 1);
    }
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
    // ---------------- TMA: Q of both heads, K tiles ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      auto issue_q = [&](int t, const PrefillTile& tl) {
        const int qb = t & 1;
        const uint32_t dst = sbase + kOffQ + (uint32_t)qb * kQStage;
        mbar_arrive_expect_tx(bar(B_QFULL + qb), kQStage);
        for (int e = 0; e < 2; ++e)
          for (int blk = 0; blk < 2; ++blk)
            tma_load_3d(dst + (uint32_t)e * kQHead + (uint32_t)blk * kQBox, &tmq,
                        bar(B_QFULL + qb), blk * 64, tl.head + e, tl.q0 + tl.q_tile * kTileQ);
      };
      // Q of local tile t >= 2 needs buffer t & 1 back: the output of tile
      // t - 2 left it (QEMPTY completion (t >> 1) - 1 of that buffer; the next
      // one needs this load).
      auto q_parity = [](int t) { return (uint32_t)(((t >> 1) - 1) & 1); };
      StepCursor c;
      c.start(a);
      bool ok = true;
      int q_issued = 0;   // Q of local tiles 0 .. q_issued - 1 issued
      int last_k = -1;
      if (!c.done()) {
        issue_q(0, c.cur);
        q_issued = 1;
        if (c.next >= 0) {
          issue_q(1, c.nxt);
          q_issued = 2;
        }
      }
      while (!c.done()) {
        const int g = c.g, st = g % NK, t = c.t;
        // the next tile's Q: as soon as its buffer is free, and at the latest
        // before this tile's ... first K of tile t + 1 (blocking there)
        if (q_issued == t + 1 && c.next >= 0 && mbar_test(bar(B_QEMPTY + ((t + 1) & 1)), q_parity(t + 1))) {
          issue_q(t + 1, c.nxt);
          ++q_issued;
        }
        if (q_issued < t + 1) {   // Q of this tile must go out before its K tiles
          if (!mbar_wait(bar(B_QEMPTY + (t & 1)), q_parity(t), a.status)) {
            ok = false;
            break;
          }
          issue_q(t, c.cur);
          ++q_issued;
        }
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
        c.advance(a);
      }
      if (!ok) {   // give the copies already issued a bounded chance to land
        if (q_issued > 0)
          mbar_wait(bar(B_QFULL + ((q_issued - 1) & 1)), (uint32_t)(((q_issued - 1) >> 1) & 1),
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
    // The two heads advance on their own: the warp polls each head's next QK
    // and next P V and issues whichever can go, so that a head whose P is
    // late does not hold the other's work back (the tensor core runs one
    // thread's MMAs in issue order).
    //   QK of head e, step g: after P V of (e, g - 2) was issued (its S buffer
    //     then holds nothing the tensor core still reads), K of g is in, and
    //     the tile's Q is.  K's stage is released once both heads' QKs of g
    //     were issued (the commit tracks every earlier MMA of this thread).
    //   P V of head e, step g: P of (e, g) is in, V of g is, and for the first
    //     step of tile t > 0 the softmax has read O of tile t - 1 (OFREE
    //     completion t - 1 of the head; completion t needs this P V).  V's
    //     stage is released once both heads' P Vs of g were issued.
    // Every wait is a poll; a head that makes no progress for the bound of a
    // wait gives up as the blocking waits do.
    StepCursor qk[2], pv[2];
    for (int e = 0; e < 2; ++e) {
      qk[e].start(a);
      pv[e].start(a);
    }
    bool ok = true;
    uint64_t t_idle = 0;
    bool idle = false;
    while (ok && !(pv[0].done() && pv[1].done())) {
      bool progress = false;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        StepCursor& q = qk[e];
        if (!q.done() && q.g <= pv[e].g + 1) {
          const int g = q.g, t = q.t;
          const bool ready = __all_sync(
              0xffffffffu, (q.j != 0 || mbar_test(bar(B_QFULL + (t & 1)), (uint32_t)((t >> 1) & 1))) &&
                               mbar_test(bar(B_KFULL + g % NK), (uint32_t)((g / NK) & 1)));
          if (ready) {
            tc_fence_after();
            const uint32_t kb = sbase + kOffK + (uint32_t)(g % NK) * kKVStage;
            const uint32_t d = tmem + 256u * (uint32_t)e + (uint32_t)(g & 1) * 64u;
            const uint32_t qa = sbase + kOffQ + (uint32_t)(t & 1) * kQStage + (uint32_t)e * kQHead;
#pragma unroll
            for (int blk = 0; blk < 2; ++blk)   // 4 k-steps of 16 per 64-column block
              umma_ss_k4(d, kmajor(qa, kQBox, 4 * blk), kmajor(kb, kKBox, 4 * blk), kIdescQK<F16>,
                         blk > 0 ? 1u : 0u);
            umma_commit_elect(bar(B_SFULL + 2 * e + (g & 1)));
            if (qk[1 - e].g > g) umma_commit_elect(bar(B_KEMPTY + g % NK));   // both QKs of g out
            q.advance(a);
            progress = true;
          }
        }
        StepCursor& p = pv[e];
        if (!p.done() && p.g < q.g) {
          const int g = p.g, s = g & 1;
          const bool ready = __all_sync(
              0xffffffffu, mbar_test(bar(B_VFULL + g % NV), (uint32_t)((g / NV) & 1)) &&
                               mbar_test(bar(B_PFULL + 2 * e + s), (uint32_t)((g >> 1) & 1)) &&
                               (p.j != 0 || p.t == 0 ||
                                mbar_test(bar(B_OFREE + e), (uint32_t)((p.t - 1) & 1))));
          if (ready) {
            tc_fence_after();
            const uint32_t vb = sbase + kOffV + (uint32_t)(g % NV) * kKVStage;
            const uint32_t p_tm = tmem + 256u * (uint32_t)e + (uint32_t)s * 64u;   // P: 32 columns
            umma_ts_k4<2048 / 16>(tmem + 256u * (uint32_t)e + 128u, p_tm, vmn(vb, 0),
                                  kIdescPV<F16>, p.j > 0 ? 1u : 0u);
            umma_commit_elect(bar(B_ODONE + 2 * e + s));
            if (pv[1 - e].g > g) umma_commit_elect(bar(B_VEMPTY + g % NV));   // both P Vs of g out
            p.advance(a);
            progress = true;
          }
        }
      }
      if (progress) {
        idle = false;
        continue;
      }
      __nanosleep(20);   // nothing ready: leave the issue slots to the softmax warps
      if (!idle) {
        idle = true;
        t_idle = global_timer_ns();
      } else if (global_timer_ns() - t_idle > kWaitLimitNs) {
        if (lane == 0) atomicOr(a.status, STATUS_WAIT_TIMEOUT);
        ok = false;
      }
    }
    umma_commit_elect(bar(B_MMADONE));
    warp_wait(bar(B_MMADONE), 0, a.status);   // nothing of ours still runs on the tensor core
  } else {
    // ---------------- softmax: one thread per query row of one head ----------------
    const int e = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;            // query row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_base = tmem + lane_off + 256u * (uint32_t)e;
    const uint32_t o_tm = s_base + 128u;
    const float sl2 = a.scale_log2;                 // >= 0 (checked by the planner)
    bool ok = true;
    StepCursor c;
    c.start(a);
    while (ok && !c.done()) {
      const PrefillTile tl = c.cur;
      const int h = tl.head + e, mt = tl.q_tile, n_kv = tl.n_kv, kv0 = tl.kv0;
      const int q0 = tl.q0, Lq = tl.lq, Lk = tl.lk;
      const int t_fin = c.t;
      const int t = mt * kTileQ + row;
      const bool row_valid = t < Lq;
      int hi = a.causal ? min(Lk, Lk - Lq + t + 1) : Lk;   // keys [lo, hi) visible
      int lo = a.window_left >= 0 ? min(hi, max(0, Lk - Lq + t - a.window_left)) : 0;
      const unsigned span = (unsigned)(hi - lo);
      float m_ref = neg_inf(), l = 0.f;
      int g_last = c.g;
      for (int j = 0; j < n_kv; ++j) {
        const int g = c.g, s = g & 1;
        // SFULL of (head, slot) completes once per step that uses the slot, in order
        if (!(ok = warp_wait(bar(B_SFULL + 2 * e + s), (uint32_t)((g >> 1) & 1), a.status))) break;
        tc_fence_after();
        const uint32_t s_tm = s_base + (uint32_t)s * 64u;
        const int key0 = (kv0 + j) * kTileK;
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
        const float mx = mraw == neg_inf() ? neg_inf() : mraw * sl2;
        const bool grow = mx > m_ref + kRescaleThreshold;
        const float m_new = grow ? mx : m_ref;
        const float alpha = grow ? ex2(m_ref - m_new) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // O holds steps before g: wait for P V of step g - 1.  ODONE of its
          // buffer completed the phase before (P V of g - 3): S of step g is
          // full, and QK of g was issued after P V of g - 2.
          const int gp = g - 1;
          if (!(ok = warp_wait(bar(B_ODONE + 2 * e + (gp & 1)), (uint32_t)((gp >> 1) & 1),
                               a.status)))
            break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < kD / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32_sync(o_tm + (uint32_t)cc * 32u, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(o_tm + (uint32_t)cc * 32u, r);
          }
          tmem_wait_st();
        }
        m_ref = m_new;
        const float neg_m = m_ref == neg_inf() ? 0.f : -m_ref;
        const bool zero_again = masked && !(sl2 > 0.f);
        const float2 sum = zero_again
                               ? exp_tile<true, F16>(ra, rb, sl2, neg_m, w0, w1, s_tm)
                               : exp_tile<false, F16>(ra, rb, sl2, neg_m, w0, w1, s_tm);
        tmem_wait_st();
        l = l * alpha + (sum.x + sum.y);
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + 2 * e + s));
        g_last = g;
        c.advance(a);
      }
      if (!ok) break;
      // O is complete once P V of the tile's last step is (the phase before,
      // P V of g_last - 2, completed: S of g_last is full)
      if (!(ok = warp_wait(bar(B_ODONE + 2 * e + (g_last & 1)), (uint32_t)((g_last >> 1) & 1),
                           a.status)))
        break;
      tc_fence_after();
      const float inv = l > 0.f ? a.output_scale / l : 0.f;
      const int qb = t_fin & 1;   // the tile's Q buffer: every QK of the tile has completed
      if (a.out_dtype == PKA_DTYPE_F32) {
        const int64_t dst = ((int64_t)(q0 + t) * a.num_qo_heads + h) * kD;
#pragma unroll 1
        for (int cc = 0; cc < kD / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32_sync(o_tm + (uint32_t)cc * 32u, r);
          if (cc == kD / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(B_OFREE + e));   // the next tile's first P V may overwrite O
          }
          if (row_valid) {
#pragma unroll
            for (int qd = 0; qd < 2; ++qd) {
              float f[16];
#pragma unroll
              for (int x = 0; x < 16; ++x) f[x] = __uint_as_float(r[16 * qd + x]);
              store_out<16>(a.out, dst + cc * 32 + qd * 16, f, inv, a.out_dtype);
            }
          }
        }
      } else {
        // 16-bit O: each warp stages its 32 rows in its own part of the tile's
        // Q buffer (16-byte chunks XOR-swizzled by row) and writes whole rows
        // back, two per store instruction
        constexpr int kRowBytes = kD * 2, kLanesPerRow = kRowBytes / 16;
        uint8_t* wbuf = smem + kOffQ + (uint32_t)qb * kQStage + (uint32_t)e * kQHead +
                        (uint32_t)quarter * 32u * kRowBytes;
        const bool f16o = a.out_dtype == PKA_DTYPE_F16;
#pragma unroll 1
        for (int cc = 0; cc < kD / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32_sync(o_tm + (uint32_t)cc * 32u, r);
          if (cc == kD / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(B_OFREE + e));
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float lo_v = __uint_as_float(r[8 * k + 2 * x]) * inv;
              const float hi_v = __uint_as_float(r[8 * k + 2 * x + 1]) * inv;
              w[x] = f16o ? pack2<true>(lo_v, hi_v) : pack2<false>(lo_v, hi_v);
            }
            const int qc = cc * 4 + k;
            *reinterpret_cast<uint4*>(wbuf + lane * kRowBytes + ((qc ^ (lane & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        __syncwarp();
        const int qc = lane % kLanesPerRow;
#pragma unroll 4
        for (int r0 = 0; r0 < 32; r0 += 32 / kLanesPerRow) {
          const int rr = r0 + lane / kLanesPerRow;
          const int tr = mt * kTileQ + quarter * 32 + rr;
          const uint4 val =
              *reinterpret_cast<const uint4*>(wbuf + rr * kRowBytes + ((qc ^ (rr & 7)) << 4));
          if (tr < Lq)
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) +
                                      ((int64_t)(q0 + tr) * a.num_qo_heads + h) * kRowBytes +
                                      qc * 16) = val;
        }
        __syncwarp();
      }
      if (row_valid && a.lse != nullptr)
        a.lse[(int64_t)(q0 + t) * a.num_qo_heads + h] = l > 0.f ? m_ref + log2f(l) : neg_inf();
      // the Q buffer may take the tile after next (a TMA write: the generic
      // accesses above are ordered before it)
      fence_proxy_async_smem();
      mbar_arrive(bar(B_QEMPTY + qb));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_prefill_gh(const pka_prefill_plan& plan, const PrefillArgs& args,
                      const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      cudaStream_t stream) {
  if (args.num_tiles == 0) return PKA_OK;
  int dev = 0, sms = 0;
  PKA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  PKA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
               "cudaDeviceGetAttribute(SM count)");
  const bool f16 = plan.desc.dtype == PKA_DTYPE_F16;
  auto kern = f16 ? prefill_gh_kernel<true> : prefill_gh_kernel<false>;
  static std::atomic<uint64_t> smem_set[2];   // per input type: devices whose limit was raised
  cudaError_t e = set_smem_once(kern, (int)kSmemBytes, smem_set[f16]);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_gh)");
  const int grid = args.num_tiles < sms ? args.num_tiles : sms;
  kern<<<grid, kThreads, kSmemBytes, stream>>>(args, qmap, kmap, vmap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "prefill_gh_kernel launch");
  return PKA_OK;
}

}  // namespace pka
