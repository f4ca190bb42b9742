// Standalone LSE merge of partial attention states, and the paged-gather test
// hook.
//
// attn_merge_lse: the states are normalised partial outputs over disjoint key
// subsets with their base-2 LSEs (cudnn_batch_decode_with_kv_cache, Note "LSE
// convention": the base-2 LSE is what the cascade-merge kernels consume).
// One warp per (row, head): m = max_i s_i, w_i = 2^(s_i - m),
// v = sum_i w_i v_i / sum_i w_i, s = m + log2 sum_i w_i.
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
