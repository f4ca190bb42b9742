// Standalone LSE merge of partial attention states, and the paged-gather test
// hook.
//
// attn_merge_lse: the states are normalised partial outputs over disjoint key
// subsets with their base-2 LSEs (cudnn_batch_decode_with_kv_cache, Note "LSE
// convention": the base-2 LSE is what the cascade-merge kernels consume).
// v = sum_i w_i v_i / sum_i w_i and s = m + log2 sum_i w_i with
// w_i = 2^(s_i - m), m = max_i s_i: head_dim 128 streams the states through
// shared memory (merge_states_stream_kernel), other head sizes take one warp
// per (row, head) (merge_states_kernel).
//
// paged_kv_gather: copies paged rows into a dense buffer through the decode
// kernels' own tensor map, unit coordinates and swizzled shared-memory reads,
// so the page addressing can be checked bit for bit.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "host_common.h"
#include "kernels.h"

namespace pka {

using namespace dev;

namespace {

__global__ void __launch_bounds__(256)
merge_states_kernel(const float* __restrict__ v, const float* __restrict__ s, int n, int rows,
                    int heads, int d, void* __restrict__ v_out, int out_dtype,
                    float* __restrict__ s_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t idx = (int64_t)blockIdx.x * 8 + warp;
  const int64_t per_state = (int64_t)rows * heads;
  if (idx >= per_state) return;
  float m = neg_inf();
  for (int i = 0; i < n; ++i) m = fmaxf(m, s[i * per_state + idx]);
  float wsum = 0.f;
  for (int i = 0; i < n && m != neg_inf(); ++i) wsum += ex2(s[i * per_state + idx] - m);
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m != neg_inf()) {
      for (int i = 0; i < n; ++i) {
        const float si = s[i * per_state + idx];
        if (si == neg_inf()) continue;
        const float w = ex2(si - m);
        const float4 x = *reinterpret_cast<const float4*>(v + (i * per_state + idx) * d + c);
        o.x += w * x.x;
        o.y += w * x.y;
        o.z += w * x.z;
        o.w += w * x.w;
      }
    }
    const float ov[4] = {o.x, o.y, o.z, o.w};
    store_out<4>(v_out, idx * d + c, ov, inv, out_dtype);
  }
  if (s_out != nullptr && lane == 0) s_out[idx] = wsum > 0.f ? m + log2f(wsum) : neg_inf();
}

// The same merge for head_dim 128 as a stream: one CTA takes kMergePairs
// consecutive (row, head) pairs, and each state's rows of them (32 KB,
// contiguous in [N, S, H, D]) arrive by one bulk copy into a ring of
// kMergeStages buffers (two, so that three CTAs fit an SM: measured on GB300
// against three buffers and two CTAs, and against 16 KB pieces four or six
// deep).  Warp w accumulates pairs kMergePPW * w onwards, lane l their
// dims 4l .. 4l + 3, with a running maximum per pair: a state whose LSE passes
// it rescales the sums so far by 2^(m_old - m_new), and every state is weighted
// 2^(s_i - m).  A wait that gives up sets STATUS_WAIT_TIMEOUT in *status.
constexpr int kMergePairs = 64, kMergeStages = 2, kMergeD = 128, kMergeMinBlocks = 3;
constexpr int kMergePPW = kMergePairs / 8;   // pairs per warp
constexpr uint32_t kMergeStageBytes = kMergePairs * kMergeD * 4;

__global__ void __launch_bounds__(256, kMergeMinBlocks)
merge_states_stream_kernel(const float* __restrict__ v, const float* __restrict__ s, int n,
                           int64_t per_state, void* __restrict__ v_out, int out_dtype,
                           float* __restrict__ s_out, int32_t* status) {
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~uintptr_t(127));
  const float* stages = reinterpret_cast<const float*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kMergeStages * kMergeStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t idx0 = (int64_t)blockIdx.x * kMergePairs;
  const int np = per_state - idx0 < kMergePairs ? (int)(per_state - idx0) : kMergePairs;
  const uint32_t bytes = (uint32_t)np * kMergeD * 4;
  const uint32_t stage0 = smem_u32(smem), bar0 = smem_u32(bars);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMergeStages; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int i) {   // state i's rows into stage i % kMergeStages
    const uint32_t st = (uint32_t)(i % kMergeStages);
    mbar_arrive_expect_tx(bar0 + 8 * st, bytes);
    bulk_load(stage0 + st * kMergeStageBytes, v + ((int64_t)i * per_state + idx0) * kMergeD,
              bytes, bar0 + 8 * st);
  };
  int issued = 0;
  if (threadIdx.x == 0)
    for (; issued < n && issued < kMergeStages; ++issued) issue(issued);

  const int p0 = warp * kMergePPW;   // this warp's first pair
  float acc[kMergePPW][4], m[kMergePPW], l[kMergePPW];
#pragma unroll
  for (int j = 0; j < kMergePPW; ++j) {
    acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    m[j] = neg_inf();
    l[j] = 0.f;
  }
  auto lse_of = [&](int i) -> float {   // lane j < kMergePPW: state i's LSE of pair p0 + j
    return lane < kMergePPW && p0 + lane < np ? __ldg(s + (int64_t)i * per_state + idx0 + p0 + lane)
                                      : neg_inf();
  };
  float lse_next = lse_of(0);
  int i = 0;
  for (; i < n; ++i) {
    const float lse_cur = lse_next;
    if (i + 1 < n) lse_next = lse_of(i + 1);
    const uint32_t st = (uint32_t)(i % kMergeStages);
    const bool ok = mbar_wait(bar0 + 8 * st, (uint32_t)((i / kMergeStages) & 1), status);
    if (__syncthreads_or(!ok)) break;
    const float* x = stages + st * (kMergeStageBytes / 4) + p0 * kMergeD + lane * 4;
#pragma unroll
    for (int j = 0; j < kMergePPW; ++j) {
      const float sj = __shfl_sync(FULL, lse_cur, j);
      if (sj == neg_inf()) continue;   // an empty state (or a pair past the end)
      if (sj > m[j]) {
        const float sc = ex2(m[j] - sj);   // 0 while m is still -inf
        acc[j][0] *= sc;
        acc[j][1] *= sc;
        acc[j][2] *= sc;
        acc[j][3] *= sc;
        l[j] *= sc;
        m[j] = sj;
      }
      const float w = ex2(sj - m[j]);
      l[j] += w;
      const float4 xv = *reinterpret_cast<const float4*>(x + j * kMergeD);
      acc[j][0] += w * xv.x;
      acc[j][1] += w * xv.y;
      acc[j][2] += w * xv.z;
      acc[j][3] += w * xv.w;
    }
    __syncthreads();   // every warp is done with this stage
    if (threadIdx.x == 0 && issued < n) issue(issued++);
  }
  if (i < n) {   // a wait gave up: the copies still in flight land (bounded) before exit
    if (threadIdx.x == 0)
      for (int j = i; j < issued; ++j)
        (void)mbar_wait(bar0 + 8 * (uint32_t)(j % kMergeStages),
                        (uint32_t)((j / kMergeStages) & 1), nullptr);
    return;
  }
#pragma unroll
  for (int j = 0; j < kMergePPW; ++j) {
    if (p0 + j >= np) break;
    const int64_t idx = idx0 + p0 + j;
    const float inv = l[j] > 0.f ? 1.f / l[j] : 0.f;
    store_out<4>(v_out, idx * kMergeD + lane * 4, acc[j], inv, out_dtype);
    if (s_out != nullptr && lane == 0) s_out[idx] = l[j] > 0.f ? m[j] + log2f(l[j]) : neg_inf();
  }
}

constexpr int kUnit = 16;
constexpr int kBoxBytes = 2048;

// One warp, one 16-token unit at a time: the same TMA unit load and swizzled
// reads the decode kernels use (here for one pool only).
__global__ void __launch_bounds__(32)
paged_gather_kernel(const __grid_constant__ CUtensorMap map, const int32_t* __restrict__ table,
                    int page_size, int tok_begin, int tok_end, int kv_head,
                    __nv_bfloat16* __restrict__ out, int32_t* __restrict__ status) {
  __shared__ __align__(1024) uint8_t buf[2 * kBoxBytes];
  __shared__ uint64_t bar;
  const int lane = threadIdx.x;
  const uint32_t bar_u32 = smem_u32(&bar);
  if (lane == 0) {
    mbar_init(bar_u32, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const int upp = page_size / kUnit;
  const int u_first = tok_begin / kUnit, u_last = (tok_end + kUnit - 1) / kUnit;
  uint32_t phase = 0;
  for (int u = u_first; u < u_last; ++u) {
    const int pid = __ldg(table + u / upp);
    if (lane == 0) {
      const uint32_t dst = smem_u32(buf);
      mbar_arrive_expect_tx(bar_u32, 2 * kBoxBytes);
      tma_load_kv_unit(dst, &map, bar_u32, (u % upp) * kUnit, kv_head, pid);
    }
    if (!__all_sync(0xffffffffu, mbar_wait(bar_u32, phase, status))) {
      (void)mbar_wait(bar_u32, phase, nullptr);   // the copy in flight: one more bounded wait
      return;
    }
    phase ^= 1u;
    // lane -> (row j = lane / 2 .. , chunk): 16 rows x 16 chunks = 256 chunk copies
    for (int q = lane; q < kUnit * 16; q += 32) {
      const int j = q >> 4, cg = q & 15;
      const int tok = u * kUnit + j;
      if (tok < tok_begin || tok >= tok_end) continue;
      const uint4 w = *reinterpret_cast<const uint4*>(
          buf + (cg >> 3) * kBoxBytes + swz128((uint32_t)j, (uint32_t)(cg & 7)));
      *reinterpret_cast<uint4*>(out + (int64_t)(tok - tok_begin) * 128 + cg * 8) = w;
    }
    __syncwarp();
  }
}

// One warp waits on phase 0 of an mbarrier that nothing arrives on, through
// the same bounded wait every kernel uses, with a bound of limit_ns.
__global__ void __launch_bounds__(32) wait_probe_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncwarp();
  (void)__all_sync(0xffffffffu, mbar_wait_for(b, 0, status, limit_ns));
}

// The block-table entries a run of the plan reads: for every work item of KV
// head 0, pages [page_lo, page_hi) of its request, cut at the live length when
// the plan reads lengths at run time.  An entry outside [0, num_pages) sets
// STATUS_PAGE_BOUNDS.
__global__ void __launch_bounds__(128)
check_tables_kernel(const WorkItem* __restrict__ items, const ReqInfo* __restrict__ reqs,
                    const int32_t* __restrict__ tables, int64_t row_stride,
                    const int32_t* __restrict__ seq_lens_live, int32_t page_size,
                    int32_t num_pages, int32_t* status) {
  const WorkItem it = items[blockIdx.x];
  if ((it.head_chunk & 0xffff) != 0) return;
  int hi = it.page_hi;
  if (seq_lens_live != nullptr) {
    const int live = min(__ldg(seq_lens_live + it.request), reqs[it.request].kv_len);
    hi = min(hi, (max(live, 0) + page_size - 1) / page_size);
  }
  const int32_t* row = tables + (int64_t)it.request * row_stride;
  bool bad = false;
  for (int pg = it.page_lo + (int)threadIdx.x; pg < hi; pg += blockDim.x)
    bad |= (unsigned)__ldg(row + pg) >= (unsigned)num_pages;
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, STATUS_PAGE_BOUNDS);
}

}  // namespace

int launch_check_tables(const WorkItem* items, int32_t num_items, const ReqInfo* reqs,
                        const int32_t* tables, int64_t row_stride, const int32_t* seq_lens_live,
                        int32_t page_size, int64_t num_pages, int32_t* status,
                        cudaStream_t stream) {
  if (num_items == 0) return PKA_OK;
  const int32_t np = num_pages > INT32_MAX ? INT32_MAX : (int32_t)num_pages;
  check_tables_kernel<<<num_items, 128, 0, stream>>>(items, reqs, tables, row_stride,
                                                     seq_lens_live, page_size, np, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "check_tables_kernel launch");
  return PKA_OK;
}

int launch_wait_probe(uint64_t limit_ns, int32_t* status, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "wait_probe_kernel launch");
  return PKA_OK;
}

int launch_merge_states(const float* v_states, const float* s_states, int32_t n, int32_t s,
                        int32_t h, int32_t d, void* v_out, int32_t out_dtype, float* s_out,
                        cudaStream_t stream) {
  const int64_t rows = (int64_t)s * h;
  if (rows == 0) return PKA_OK;
  if (d == kMergeD) {
    constexpr int smem = kMergeStages * kMergeStageBytes + kMergeStages * 8 + 128;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = set_smem_once(merge_states_stream_kernel, smem, smem_set);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(merge_states_stream)");
    int32_t* status = nullptr;
    const int rc = noalloc_status_word(stream, &status);
    if (rc != PKA_OK) return rc;
    const int64_t blocks = (rows + kMergePairs - 1) / kMergePairs;
    merge_states_stream_kernel<<<(unsigned)blocks, 256, smem, stream>>>(
        v_states, s_states, n, rows, v_out, out_dtype, s_out, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "merge_states_stream_kernel launch");
    return PKA_OK;
  }
  const int64_t blocks = (rows + 7) / 8;
  merge_states_kernel<<<(unsigned)blocks, 256, 0, stream>>>(v_states, s_states, n, s, h, d, v_out,
                                                           out_dtype, s_out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "merge_states_kernel launch");
  return PKA_OK;
}

int launch_paged_gather(const CUtensorMap& map, const int32_t* block_tables,
                        int64_t bt_row_stride, int32_t page_size, int32_t request,
                        int32_t kv_head, int32_t tok_begin, int32_t tok_end, void* out,
                        cudaStream_t stream) {
  if (tok_end <= tok_begin) return PKA_OK;
  paged_gather_kernel<<<1, 32, 0, stream>>>(map, block_tables + (int64_t)request * bt_row_stride,
                                            page_size, tok_begin, tok_end, kv_head,
                                            reinterpret_cast<__nv_bfloat16*>(out), nullptr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "paged_gather_kernel launch");
  return PKA_OK;
}

}  // namespace pka
