// Paged decode attention, tensor-core variant: the plan's default for every
// query group, from one row per KV head (MHA) through GQA groups to
// speculative packed-Q verification with cudnn_batch_decode_with_kv_cache's
// q_len_per_req rows.
//
// Same work items, masks, softmax and outputs as the CUDA-core kernel; the
// two contractions run on mma.sync m16n8k16 (bf16 or f16 in, fp32 accumulate):
//  * a CTA handles one 16-row tile of the item's query rows (row r = i*group
//    + g: token i, head g of the group); blockIdx.x = item * MT + tile, so
//    the MT tiles of one item run side by side and all but the first read its
//    K/V pages from L2;
//  * its four warps each stream their own 16-token units (w, w+4, ...) with
//    TMA into a private NSTAGE-deep ring (128-byte swizzle keeps ldmatrix
//    conflict-free), exactly as in the CUDA-core kernel.  Every warp issues
//    its own copies: copies of one issuing thread complete at roughly one
//    per microsecond whatever their size, so many issuers are needed;
//  * per unit: S = Q K^T (2 n-tiles x 8 k-steps, Q in A-fragment registers),
//    mask, online softmax in base 2 on the fragments, P re-packed to 16-bit
//    A fragments in registers, O += P V (16 n-tiles, V via ldmatrix.trans);
//    a tile of at most 8 live rows (a group of at most 8 rows, or the last
//    tile of one of 8 (mod 16)) takes the transposed step instead,
//    S^T = K Q^T and O^T += V^T P^T, with the 16 keys of a unit on the
//    16-row side of the instruction and the rows on its 8-column side: half
//    the mma of a padded 16-row tile;
//  * the four warps' (m, l, O) are merged through shared memory and the CTA
//    writes final O/LSE (sink added), or, for a split request, an fp32 partial;
//    the last chunk CTA of each (request, KV head, tile) merges the partials.
// Decode is bound by HBM, not by the tensor pipe: mma takes the per-key
// arithmetic of wide groups off the FP32 pipe.
#include <cuda_bf16.h>

#include "decode_merge.cuh"
#include "decode_mma_tile.cuh"
#include "device_common.cuh"
#include "host_common.h"
#include "kernels.h"

namespace pka {

using namespace dev;

namespace {

constexpr int kWarps = 4;
constexpr int kUnit = kMmaUnitTok;
constexpr int kStageBytes = kMmaUnitBytes;
constexpr int kBoxBytes = kMmaBoxBytes;

// NARROW: every group has at most 8 rows, and only the transposed step is
// compiled; otherwise a CTA takes it when its tile has at most 8 live rows
// (the last tile of a group of 8 (mod 16) rows), else the 16-row step.
template <int NSTAGE, bool F16, bool NARROW>
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
  mma_row_key_range(kv_len, L, 0, a.causal, a.window_left, lo_first, hi_first);
  mma_row_key_range(kv_len, L, L - 1, a.causal, a.window_left, lo_last, hi_last);
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

  const float sl2 = a.scale_log2;

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
  int tcur = 0, tnext = 0, tbatch = 0;
  auto issue = [&](int k) {
    if ((k >> 5) > tbatch) {
      tcur = tnext;
      tnext = table_batch(tbatch + 2);
      ++tbatch;
    }
    const int pid = __shfl_sync(FULL, tcur, k & 31);
    const int u = unit0 + warp + k * kWarps;
    const int slot = (u % upp) * kUnit;
    const int st = k % NSTAGE;
    const uint32_t dst = stage_u32 + st * kStageBytes, bar = bar_u32 + st * 8;
    tma_load_kv_pair_elect(dst, dst + 2 * kBoxBytes, &tmk, &tmv, bar, kStageBytes, slot, hk, pid);
  };
  float* comb_o = reinterpret_cast<float*>(stages);              // [warps][16][kMmaCombStride]
  float* comb_m = comb_o + kWarps * 16 * kMmaCombStride;         // [warps][16]
  float* comb_l = comb_m + kWarps * 16;                          // [warps][16]

  // the warp's units through tile step `tw`, then its (m, l, O) into the
  // merge buffers (which reuse the stages)
  auto run = [&](auto& tw) {
    tw.init(a, rq, kv_len, hk, mt, lane);
    tcur = table_batch(0);
    tnext = table_batch(1);
    const int pre = my_units < NSTAGE ? my_units : NSTAGE;
    for (int k = 0; k < pre; ++k) issue(k);

    int k = 0;
    for (; k < my_units; ++k) {
      const int st = k % NSTAGE;
      if (!__all_sync(FULL, mbar_wait(bar_u32 + st * 8, (uint32_t)((k / NSTAGE) & 1), a.status)))
        break;
      const int tok0 = (unit0 + warp + k * kWarps) * kUnit;
      const bool full_unit = tok0 >= all_lo && tok0 + kUnit <= all_hi;
      tw.step(stage_u32 + st * kStageBytes, tok0, full_unit, sl2, lane);
      __syncwarp();
      if (k + NSTAGE < my_units) issue(k + NSTAGE);
    }
    // a wait gave up: let the copies still in flight land (bounded) before the
    // stages are reused or the CTA exits
    for (int j = k; j < my_units && j < k + NSTAGE; ++j)
      (void)mbar_wait(bar_u32 + (j % NSTAGE) * 8, (uint32_t)((j / NSTAGE) & 1), a.status);
    tw.reduce_l();
    __syncthreads();   // every warp is done with its stages
    tw.store_comb(comb_o, comb_m, comb_l, warp, lane);
  };
  // a tile of at most 8 live rows takes the transposed step
  if (NARROW || rows_b - mt * 16 <= 8) {
    MmaTileWarpT<F16> tw;
    run(tw);
  } else {
    if constexpr (!NARROW) {
      MmaTileWarp<F16> tw;
      run(tw);
    }
  }
  __syncthreads();

  // thread -> (row of the tile, 16 consecutive dims)
  mma_combine_store(a, rq, comb_o, comb_m, comb_l, 0, kWarps, mt, tid >> 3, (tid & 7) * 16, hk,
                    chunk);
  if (rq.part_base >= 0)   // a split request: the group's last chunk merges its rows
    split_merge_if_last(a, rq, hk, mt, mt * 16, min(16, rows_b - mt * 16));
}

template <int NSTAGE, bool F16, bool NARROW>
int launch_mma(const DecodeArgs& args, const CUtensorMap& kmap, const CUtensorMap& vmap,
               cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)kWarps * NSTAGE * kStageBytes + kWarps * NSTAGE * 8;
  static_assert(kWarps * 16 * (kMmaCombStride + 2) * 4 <= kWarps * NSTAGE * kStageBytes,
                "merge buffer does not fit in the stage area");
  auto kern = decode_mma_kernel<NSTAGE, F16, NARROW>;
  static std::atomic<uint64_t> smem_set{0};   // devices whose limit this launcher raised
  cudaError_t e = set_smem_once(kern, (int)smem, smem_set);
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
  if (args.rows_per_cta <= 8)   // the transposed step only: keys on the 16-row side
    return args.in_f16 ? launch_mma<2, true, true>(args, kmap, vmap, stream)
                       : launch_mma<2, false, true>(args, kmap, vmap, stream);
  return args.in_f16 ? launch_mma<2, true, false>(args, kmap, vmap, stream)
                     : launch_mma<2, false, false>(args, kmap, vmap, stream);
}

}  // namespace pka
