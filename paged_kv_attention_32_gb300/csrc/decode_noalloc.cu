// paged_decode_run_noalloc: the planned decode for callers that cannot
// allocate device memory -- code running where cudaMalloc is not allowed
// (inside an allocator hook, or a serving process whose device memory is a
// fixed pool owned by someone else).  Everything the run needs beyond the
// caller's inputs and outputs -- the plan's work list and the split-KV fp32
// partials -- lives in one file-scope device array of fixed size.
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "host_common.h"
#include "kernels.h"
#include "plan.h"
#include "tmap.h"

namespace pka {
namespace {

// Fixed scratch: 16 MiB on every GPU that loads the library, held until the
// process exits.  Layout per call: status word | work items | request info |
// merge counters | partial outputs | partial LSEs, each 256-byte aligned.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr size_t kStatusBytes = 256;   // the status word, padded to the alignment
constexpr int kMaxDevices = 256;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the scratch array on `dev` (the current device), looked
// up once per device.  In host code the symbol is only a stand-in: kernels
// get this address, never the symbol itself.  The set-up also clears the
// status word once, queued on `stream` ahead of the caller's work; after that
// only paged_decode_plan_check clears it, so a failed wait in any run since
// the last check stays visible.
int scratch_address(int dev, cudaStream_t stream, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(PKA_ERR_INVALID_ARG, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    e = cudaMemsetAsync(p, 0, kStatusBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(no-alloc status)");
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
  return PKA_OK;
}

}  // namespace

int noalloc_status_word(cudaStream_t stream, int32_t** out) {
  int dev = -1;
  PKA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  unsigned char* base = nullptr;
  const int rc = scratch_address(dev, stream, &base);
  if (rc != PKA_OK) return rc;
  *out = reinterpret_cast<int32_t*>(base);
  return PKA_OK;
}

}  // namespace pka

using namespace pka;

extern "C" int paged_decode_run_noalloc(const pka_plan* p, const void* q, int64_t q_stride_tok,
                                        int64_t q_stride_head, const void* k_pages,
                                        const void* v_pages, int64_t kv_stride_page,
                                        int64_t kv_stride_head, const int32_t* block_tables,
                                        int64_t bt_row_stride, const int32_t* seq_lens_kv_dev,
                                        const float* sinks, void* out, float* lse, void* stream) {
  nvtxRangePushA("pka::paged_decode_run_noalloc");
  struct PopOnExit { ~PopOnExit() { nvtxRangePop(); } } nvtx_pop;
  clear_error();
  PKA_CHECK_ARG(p != nullptr, "plan must not be NULL");
  PKA_CHECK_ARG(q && k_pages && v_pages && block_tables && out,
                "q, k_pages, v_pages, block_tables and out must not be NULL");
  PKA_CHECK_ARG(p->desc.freeze_seq_lens || seq_lens_kv_dev != nullptr,
                "seq_lens_kv_dev is required when the plan does not freeze the lengths");
  PKA_CHECK_ARG(!p->desc.return_lse || lse != nullptr, "the plan returns the LSE: lse is NULL");
  PKA_CHECK_ARG(reinterpret_cast<uintptr_t>(q) % 16 == 0 && q_stride_tok % 8 == 0 &&
                    q_stride_head % 8 == 0 && q_stride_tok >= 0 && q_stride_head >= 0,
                "q must be 16-byte aligned with non-negative strides that are multiples of 8");
  PKA_CHECK_ARG(reinterpret_cast<uintptr_t>(out) % 16 == 0, "out must be 16-byte aligned");
  PKA_CHECK_ARG(lse == nullptr || reinterpret_cast<uintptr_t>(lse) % 4 == 0,
                "lse must be 4-byte aligned");
  PKA_CHECK_ARG(kv_stride_page % 8 == 0 && kv_stride_head % 8 == 0,
                "K/V strides must be multiples of 8 elements");
  PKA_CHECK_ARG(bt_row_stride >= p->C, "bt_row_stride is smaller than the table width");

  // scratch layout for this plan
  const size_t n_items = p->items.size() * sizeof(WorkItem);
  const size_t n_reqs = p->reqs.size() * sizeof(ReqInfo);
  const size_t n_cnt = (size_t)p->num_merge_counters * sizeof(int32_t);
  const size_t off_items = kStatusBytes;
  const size_t off_reqs = off_items + up256(n_items);
  const size_t off_cnt = off_reqs + up256(n_reqs);
  const size_t off_ws = off_cnt + up256(n_cnt);
  const size_t off_lse = off_ws + (size_t)p->ws_lse_offset;
  const size_t total = off_ws + (size_t)p->workspace_bytes;
  if (total > kNoAllocScratchBytes)
    return fail(PKA_ERR_WORKSPACE_TOO_SMALL,
                "the plan needs %zu bytes of scratch; paged_decode_run_noalloc holds at most %zu "
                "(use paged_decode_run with a caller workspace)",
                total, kNoAllocScratchBytes);

  int dev = -1;
  PKA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  // a plan with a device copy was made for one device; a host-only plan runs
  // on whichever device is current
  if (p->dev_buf != nullptr)
    PKA_CHECK_ARG(dev == p->device, "plan was made on device %d, current device is %d",
                  p->device, dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* base = nullptr;
  int rc = scratch_address(dev, s, &base);
  if (rc != PKA_OK) return rc;
  // Of the rest only the merge counters must start at zero (below): every
  // partial row is written by its chunk before the group's last chunk CTA
  // reads it, and the status word is cleared only by paged_decode_plan_check
  // (it collects every run since).
  if (n_items)
    PKA_CUDA_TRY(cudaMemcpyAsync(base + off_items, p->items.data(), n_items,
                                 cudaMemcpyHostToDevice, s),
                 "cudaMemcpyAsync(no-alloc items)");
  PKA_CUDA_TRY(cudaMemcpyAsync(base + off_reqs, p->reqs.data(), n_reqs, cudaMemcpyHostToDevice, s),
               "cudaMemcpyAsync(no-alloc requests)");
  // the last chunk CTA of each split group merges it; the counters that tell it
  // so start at zero (the kernels leave them at zero, but an earlier call of
  // another plan may have used this space otherwise)
  if (n_cnt)
    PKA_CUDA_TRY(cudaMemsetAsync(base + off_cnt, 0, n_cnt, s),
                 "cudaMemsetAsync(no-alloc merge counters)");

  CUtensorMap kmap, vmap;
  rc = encode_kv_pool_map(&kmap, k_pages, p->desc.num_pages, p->Hkv, p->ps, p->D, kv_stride_page,
                          kv_stride_head);
  if (rc != PKA_OK) return rc;
  rc = encode_kv_pool_map(&vmap, v_pages, p->desc.num_pages, p->Hkv, p->ps, p->D, kv_stride_page,
                          kv_stride_head);
  if (rc != PKA_OK) return rc;

  DecodeArgs a{};
  a.q = q;
  a.q_stride_tok = q_stride_tok;
  a.q_stride_head = q_stride_head;
  a.block_tables = block_tables;
  a.bt_row_stride = bt_row_stride;
  a.seq_lens_live = p->desc.freeze_seq_lens ? nullptr : seq_lens_kv_dev;
  a.sinks = sinks;
  a.out = out;
  a.lse = p->desc.return_lse ? lse : nullptr;
  a.ws_o = reinterpret_cast<float*>(base + off_ws);
  a.ws_lse = reinterpret_cast<float*>(base + off_lse);
  a.items = reinterpret_cast<const WorkItem*>(base + off_items);
  a.reqs = reinterpret_cast<const ReqInfo*>(base + off_reqs);
  a.merge_cnt = reinterpret_cast<int32_t*>(base + off_cnt);
  a.status = reinterpret_cast<int32_t*>(base);
  a.num_items = (int32_t)p->items.size();
  a.tiles_per_item = p->kernel == PKA_KERNEL_MMA ? (p->rows_per_cta + 15) / 16 : 1;
  a.num_qo_heads = p->Hq;
  a.num_kv_heads = p->Hkv;
  a.group = p->G;
  a.page_size = p->ps;
  a.causal = p->desc.mask == PKA_MASK_CAUSAL;
  a.window_left = p->desc.window_left;
  a.rows_per_cta = p->rows_per_cta;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.bmm2_scale = p->desc.bmm2_scale;
  a.in_f16 = p->desc.dtype == PKA_DTYPE_F16;
  a.out_dtype = p->desc.out_dtype;
  return launch_decode(*p, a, kmap, vmap, s);
}
