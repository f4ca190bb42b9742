// extern "C" entry points of pka.h: argument checks, plan ownership, launch
// dispatch.  Nothing here computes attention; every step of the path runs in
// the kernels.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <new>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "host_common.h"
#include "kernels.h"
#include "plan.h"
#include "prefill.h"
#include "tmap.h"

namespace pka {

namespace {
thread_local std::string g_last_error;
}

int fail(int code, const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

void clear_error() { g_last_error.clear(); }

const char* last_error() { return g_last_error.c_str(); }

}  // namespace pka

using namespace pka;

namespace {

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// An NVTX range over an entry point, so that the plan and run calls show up by
// name on a profiler's timeline (a no-op call when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

int upload_decode_plan(pka_plan& p, cudaStream_t stream) {
  const size_t n_items = p.items.size() * sizeof(WorkItem);
  const size_t n_reqs = p.reqs.size() * sizeof(ReqInfo);
  const size_t n_cnt = (size_t)p.num_merge_counters * sizeof(int32_t);
  const size_t off_reqs = up256(n_items);
  const size_t off_status = off_reqs + up256(n_reqs);
  const size_t off_cnt = off_status + 256;   // merge counters, zero between runs
  const size_t total = off_cnt + up256(n_cnt);
  if (p.dev_buf == nullptr || total > p.dev_capacity) {
    // a replan that outgrows the buffer reallocates it with headroom
    if (p.dev_buf != nullptr) {
      PKA_CUDA_TRY(cudaFree(p.dev_buf), "cudaFree(decode plan)");
      p.dev_buf = nullptr;
      p.dev_capacity = 0;
    }
    const size_t cap = p.dev_capacity == 0 && total < 4096 ? 4096 : total + total / 2;
    PKA_CUDA_TRY(cudaGetDevice(&p.device), "cudaGetDevice");
    PKA_CUDA_TRY(cudaMalloc(&p.dev_buf, cap), "cudaMalloc(decode plan)");
    p.dev_capacity = cap;
  }
  uint8_t* base = static_cast<uint8_t*>(p.dev_buf);
  p.d_items = reinterpret_cast<const WorkItem*>(base);
  p.d_reqs = reinterpret_cast<const ReqInfo*>(base + off_reqs);
  p.d_status = reinterpret_cast<int32_t*>(base + off_status);
  p.d_merge_cnt = reinterpret_cast<int32_t*>(base + off_cnt);
  // One asynchronous copy from a pinned image of the buffer.  The image is
  // rewritten only after the copy that last read it has completed (stage_done);
  // stream order keeps the upload behind runs already queued on the same stream.
  if (p.host_stage != nullptr && p.stage_done != nullptr)
    PKA_CUDA_TRY(cudaEventSynchronize(p.stage_done), "cudaEventSynchronize(plan upload)");
  if (p.host_stage == nullptr || total > p.host_capacity) {
    if (p.host_stage != nullptr) {
      PKA_CUDA_TRY(cudaFreeHost(p.host_stage), "cudaFreeHost(plan image)");
      p.host_stage = nullptr;
      p.host_capacity = 0;
    }
    if (cudaMallocHost(&p.host_stage, p.dev_capacity) == cudaSuccess) {
      p.host_capacity = p.dev_capacity;
    } else {
      (void)cudaGetLastError();   // no pinned memory: copy from the pageable vectors
      p.host_stage = nullptr;
    }
  }
  if (p.host_stage != nullptr) {
    uint8_t* img = static_cast<uint8_t*>(p.host_stage);
    if (n_items) std::memcpy(img, p.items.data(), n_items);
    std::memcpy(img + off_reqs, p.reqs.data(), n_reqs);
    std::memset(img + off_status, 0, total - off_status);   // status word and counters
    PKA_CUDA_TRY(cudaMemcpyAsync(base, img, total, cudaMemcpyHostToDevice, stream),
                 "cudaMemcpyAsync(plan)");
    if (p.stage_done == nullptr)
      PKA_CUDA_TRY(cudaEventCreateWithFlags(&p.stage_done, cudaEventDisableTiming),
                   "cudaEventCreate(plan upload)");
    PKA_CUDA_TRY(cudaEventRecord(p.stage_done, stream), "cudaEventRecord(plan upload)");
    return PKA_OK;
  }
  // Copies from pageable host vectors are staged before cudaMemcpyAsync returns,
  // so a later replan may overwrite them.
  if (n_items)
    PKA_CUDA_TRY(cudaMemcpyAsync(base, p.items.data(), n_items, cudaMemcpyHostToDevice, stream),
                 "cudaMemcpyAsync(plan items)");
  PKA_CUDA_TRY(cudaMemcpyAsync(base + off_reqs, p.reqs.data(), n_reqs, cudaMemcpyHostToDevice,
                               stream),
               "cudaMemcpyAsync(plan requests)");
  PKA_CUDA_TRY(cudaMemsetAsync(base + off_status, 0, total - off_status, stream),
               "cudaMemsetAsync(status and counters)");
  return PKA_OK;
}

int upload_prefill_plan(pka_prefill_plan& p, cudaStream_t stream) {
  const size_t n_tiles = p.tiles.size() * sizeof(PrefillTile);
  const size_t n_ind = p.qo.size() * sizeof(int32_t);
  const size_t n_win = p.win_lo.size() * sizeof(int32_t);
  const size_t off_qo = up256(n_tiles);
  const size_t off_kv = off_qo + up256(n_ind);
  const size_t off_wlo = off_kv + up256(n_ind);
  const size_t off_whi = off_wlo + up256(n_win);
  const size_t n_map = p.row_map.size() * sizeof(int32_t);
  const size_t off_map = off_whi + up256(n_win);
  const size_t off_status = off_map + up256(n_map);
  const size_t total = off_status + 256;
  PKA_CUDA_TRY(cudaGetDevice(&p.device), "cudaGetDevice");
  PKA_CUDA_TRY(cudaMalloc(&p.dev_buf, total), "cudaMalloc(prefill plan)");
  uint8_t* base = static_cast<uint8_t*>(p.dev_buf);
  p.d_tiles = reinterpret_cast<const PrefillTile*>(base);
  p.d_qo = reinterpret_cast<const int32_t*>(base + off_qo);
  p.d_kv = reinterpret_cast<const int32_t*>(base + off_kv);
  p.d_status = reinterpret_cast<int32_t*>(base + off_status);
  if (n_tiles)
    PKA_CUDA_TRY(cudaMemcpyAsync(base, p.tiles.data(), n_tiles, cudaMemcpyHostToDevice, stream),
                 "cudaMemcpyAsync(prefill tiles)");
  PKA_CUDA_TRY(cudaMemcpyAsync(base + off_qo, p.qo.data(), n_ind, cudaMemcpyHostToDevice, stream),
               "cudaMemcpyAsync(qo_indptr)");
  PKA_CUDA_TRY(cudaMemcpyAsync(base + off_kv, p.kv.data(), n_ind, cudaMemcpyHostToDevice, stream),
               "cudaMemcpyAsync(kv_indptr)");
  if (n_win) {
    p.d_win_lo = reinterpret_cast<const int32_t*>(base + off_wlo);
    p.d_win_hi = reinterpret_cast<const int32_t*>(base + off_whi);
    PKA_CUDA_TRY(cudaMemcpyAsync(base + off_wlo, p.win_lo.data(), n_win, cudaMemcpyHostToDevice,
                                 stream),
                 "cudaMemcpyAsync(window starts)");
    PKA_CUDA_TRY(cudaMemcpyAsync(base + off_whi, p.win_hi.data(), n_win, cudaMemcpyHostToDevice,
                                 stream),
                 "cudaMemcpyAsync(window ends)");
  }
  if (n_map) {
    p.d_row_map = reinterpret_cast<const int32_t*>(base + off_map);
    PKA_CUDA_TRY(cudaMemcpyAsync(base + off_map, p.row_map.data(), n_map, cudaMemcpyHostToDevice,
                                 stream),
                 "cudaMemcpyAsync(row order)");
  }
  PKA_CUDA_TRY(cudaMemsetAsync(base + off_status, 0, 256, stream), "cudaMemsetAsync(status)");
  return PKA_OK;
}

int check_device(int plan_device) {
  int dev = -1;
  PKA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  PKA_CHECK_ARG(dev == plan_device, "plan was made on device %d, current device is %d",
                plan_device, dev);
  return PKA_OK;
}

int read_status(int32_t* d_status, cudaStream_t stream) {
  int32_t st = 0;
  PKA_CUDA_TRY(cudaMemcpyAsync(&st, d_status, sizeof(st), cudaMemcpyDeviceToHost, stream),
               "cudaMemcpyAsync(status)");
  PKA_CUDA_TRY(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  PKA_CUDA_TRY(cudaMemsetAsync(d_status, 0, sizeof(int32_t), stream), "cudaMemsetAsync(status)");
  PKA_CUDA_TRY(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  if (st & STATUS_WAIT_TIMEOUT)
    return fail(PKA_ERR_DEVICE_TIMEOUT, "a kernel gave up on a bounded wait (status 0x%x)", st);
  if (st & STATUS_PAGE_BOUNDS)
    return fail(PKA_ERR_DEVICE_BOUNDS,
                "a block-table entry a run would read is outside [0, num_pages) (status 0x%x)",
                st);
  return PKA_OK;
}

}  // namespace

extern "C" {

const char* pka_last_error(void) { return pka::last_error(); }

const char* pka_version(void) { return "pka 0.1.0 (sm_103a)"; }

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------

int paged_decode_plan(pka_plan** plan_out, const pka_decode_desc* desc,
                      const int32_t* seq_lens_kv_host, const int32_t* qo_indptr_host,
                      size_t* workspace_bytes_out, void* stream) {
  NvtxRange nvtx_range("pka::paged_decode_plan");
  clear_error();
  PKA_CHECK_ARG(plan_out != nullptr && desc != nullptr, "plan_out and desc must not be NULL");
  *plan_out = nullptr;
  pka_plan* p = new (std::nothrow) pka_plan();
  if (p == nullptr) return fail(PKA_ERR_INVALID_ARG, "out of host memory");
  int rc = build_decode_plan(*p, *desc, seq_lens_kv_host, qo_indptr_host);
  if (rc == PKA_OK && !(desc->flags & PKA_PLAN_HOST_ONLY))
    rc = upload_decode_plan(*p, static_cast<cudaStream_t>(stream));
  if (rc != PKA_OK) {
    paged_decode_plan_destroy(p);
    return rc;
  }
  if (workspace_bytes_out) *workspace_bytes_out = (size_t)p->workspace_bytes;
  *plan_out = p;
  return PKA_OK;
}

int paged_decode_plan_update(pka_plan* p, int32_t batch_size, const int32_t* seq_lens_kv_host,
                             const int32_t* qo_indptr_host, size_t* workspace_bytes_out,
                             void* stream) {
  NvtxRange nvtx_range("pka::paged_decode_plan_update");
  clear_error();
  PKA_CHECK_ARG(p != nullptr, "plan must not be NULL");
  pka_decode_desc d = p->desc;
  d.batch_size = batch_size;
  pka_plan fresh;
  int rc = build_decode_plan(fresh, d, seq_lens_kv_host, qo_indptr_host);
  if (rc != PKA_OK) return rc;   // the old plan stays as it was
  if (!(p->desc.flags & PKA_PLAN_HOST_ONLY)) {
    int dev = -1;
    PKA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
    PKA_CHECK_ARG(dev == p->device, "plan was made on device %d, current device is %d", p->device,
                  dev);
  }
  fresh.dev_buf = p->dev_buf;
  fresh.dev_capacity = p->dev_capacity;
  fresh.device = p->device;
  fresh.host_stage = p->host_stage;
  fresh.host_capacity = p->host_capacity;
  fresh.stage_done = p->stage_done;
  p->dev_buf = nullptr;
  p->host_stage = nullptr;
  p->stage_done = nullptr;
  *p = std::move(fresh);
  if (!(p->desc.flags & PKA_PLAN_HOST_ONLY)) {
    rc = upload_decode_plan(*p, static_cast<cudaStream_t>(stream));
    if (rc != PKA_OK) return rc;
  }
  if (workspace_bytes_out) *workspace_bytes_out = (size_t)p->workspace_bytes;
  return PKA_OK;
}

void paged_decode_plan_destroy(pka_plan* plan) {
  if (plan == nullptr) return;
  if (plan->stage_done != nullptr) {
    cudaEventSynchronize(plan->stage_done);   // the image is not freed under a pending copy
    cudaEventDestroy(plan->stage_done);
  }
  if (plan->host_stage != nullptr) cudaFreeHost(plan->host_stage);
  if (plan->dev_buf != nullptr) cudaFree(plan->dev_buf);
  delete plan;
}

int paged_decode_plan_info(const pka_plan* p, pka_plan_info* info) {
  clear_error();
  PKA_CHECK_ARG(p != nullptr && info != nullptr, "plan and info must not be NULL");
  info->num_items = (int32_t)p->items.size();
  info->chunk_pages = p->chunk_pages;
  info->num_split = p->num_split;
  info->partial_rows = p->partial_rows;
  info->workspace_bytes = p->workspace_bytes;
  info->kernel = p->kernel;
  info->rows_per_cta = p->rows_per_cta;
  info->num_sms = p->desc.num_sms;
  info->split_waves = p->desc.split_waves;
  info->min_chunk_tokens = p->desc.min_chunk_tokens;
  info->total_q = p->total_q;
  return PKA_OK;
}

int paged_decode_plan_export(const pka_plan* p, int32_t* items, int32_t* n_chunks,
                             int32_t* part_base, int32_t* page_lo, int32_t* page_hi,
                             int32_t* order) {
  clear_error();
  PKA_CHECK_ARG(p != nullptr, "plan must not be NULL");
  if (items) {
    for (size_t i = 0; i < p->items.size(); ++i) {
      const WorkItem& w = p->items[i];
      items[5 * i + 0] = w.request;
      items[5 * i + 1] = w.head_chunk & 0xffff;
      items[5 * i + 2] = w.head_chunk >> 16;
      items[5 * i + 3] = w.page_lo;
      items[5 * i + 4] = w.page_hi;
    }
  }
  for (int32_t b = 0; b < p->B; ++b) {
    if (n_chunks) n_chunks[b] = p->reqs[b].n_chunks;
    if (part_base) part_base[b] = p->reqs[b].part_base;
    if (page_lo) page_lo[b] = p->page_lo[b];
    if (page_hi) page_hi[b] = p->page_hi[b];
    if (order) order[b] = p->order[b];
  }
  return PKA_OK;
}

int paged_decode_run(const pka_plan* p, const void* q, int64_t q_stride_tok,
                     int64_t q_stride_head, const void* k_pages, const void* v_pages,
                     int64_t kv_stride_page, int64_t kv_stride_head,
                     const int32_t* block_tables, int64_t bt_row_stride,
                     const int32_t* seq_lens_kv_dev, const float* sinks, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("pka::paged_decode_run");
  clear_error();
  PKA_CHECK_ARG(p != nullptr, "plan must not be NULL");
  PKA_CHECK_ARG(p->dev_buf != nullptr, "plan was built with PKA_PLAN_HOST_ONLY and cannot run");
  PKA_CHECK_ARG(q && k_pages && v_pages && block_tables && out,
                "q, k_pages, v_pages, block_tables and out must not be NULL");
  PKA_CHECK_ARG(p->desc.freeze_seq_lens || seq_lens_kv_dev != nullptr,
                "seq_lens_kv_dev is required when the plan does not freeze the lengths");
  PKA_CHECK_ARG(!p->desc.return_lse || lse != nullptr, "the plan returns the LSE: lse is NULL");
  PKA_CHECK_ARG(aligned(q, 16) && q_stride_tok % 8 == 0 && q_stride_head % 8 == 0,
                "q must be 16-byte aligned with strides that are multiples of 8 elements");
  PKA_CHECK_ARG(q_stride_tok >= 0 && q_stride_head >= 0, "q strides must be non-negative");
  PKA_CHECK_ARG(aligned(out, 16), "out must be 16-byte aligned");
  PKA_CHECK_ARG(lse == nullptr || aligned(lse, 4), "lse must be 4-byte aligned");
  PKA_CHECK_ARG(kv_stride_page % 8 == 0 && kv_stride_head % 8 == 0,
                "K/V strides must be multiples of 8 elements");
  PKA_CHECK_ARG(bt_row_stride >= p->C, "bt_row_stride (%lld) is smaller than the table width %d",
                (long long)bt_row_stride, p->C);
  if (p->workspace_bytes > 0) {
    if (workspace == nullptr || workspace_bytes < (size_t)p->workspace_bytes)
      return fail(PKA_ERR_WORKSPACE_TOO_SMALL, "workspace of %zu bytes, the plan needs %lld",
                  workspace_bytes, (long long)p->workspace_bytes);
    PKA_CHECK_ARG(aligned(workspace, 256), "workspace must be 256-byte aligned");
  }
  int rc = check_device(p->device);
  if (rc != PKA_OK) return rc;

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
  a.ws_o = static_cast<float*>(workspace);
  a.ws_lse = workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                  p->ws_lse_offset)
                       : nullptr;
  a.items = p->d_items;
  a.reqs = p->d_reqs;
  a.merge_cnt = p->d_merge_cnt;
  a.status = p->d_status;
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
  return launch_decode(*p, a, kmap, vmap, static_cast<cudaStream_t>(stream));
}

namespace {
// The device address of `host` when it is page-locked host memory the current
// device can address (a kernel may then read or write it in place over the
// host link), else nullptr.
void* host_mapped(const void* host) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}
}  // namespace

int paged_decode_step_host(pka_plan* p, int32_t batch_size, const pka_decode_host_io* io,
                           const void* k_pages, const void* v_pages, int64_t kv_stride_page,
                           int64_t kv_stride_head, const float* sinks, void* workspace,
                           size_t workspace_bytes, size_t* workspace_bytes_out,
                           int32_t synchronize, void* stream) {
  NvtxRange nvtx_range("pka::paged_decode_step_host");
  clear_error();
  PKA_CHECK_ARG(p != nullptr && io != nullptr, "plan and io must not be NULL");
  PKA_CHECK_ARG(p->dev_buf != nullptr, "plan was built with PKA_PLAN_HOST_ONLY and cannot run");
  PKA_CHECK_ARG(io->q_host && io->block_tables_host && io->seq_lens_kv_host && io->out_host &&
                    io->q_dev && io->block_tables_dev && io->out_dev,
                "the q, block-table, length and output buffers must not be NULL");
  PKA_CHECK_ARG(k_pages && v_pages, "k_pages and v_pages must not be NULL");
  PKA_CHECK_ARG(p->desc.freeze_seq_lens || io->seq_lens_kv_dev != nullptr,
                "seq_lens_kv_dev is required when the plan does not freeze the lengths");
  PKA_CHECK_ARG(!p->desc.return_lse || (io->lse_host != nullptr && io->lse_dev != nullptr),
                "the plan returns the LSE: lse_host and lse_dev are required");
  PKA_CHECK_ARG(io->bt_row_stride >= p->C,
                "bt_row_stride (%lld) is smaller than the table width %d",
                (long long)io->bt_row_stride, p->C);
  // A device array given as its host array itself is used in place: the
  // kernel reads (or writes) the page-locked host memory directly, and the
  // step copies nothing for it.
  const void* q_use = io->q_dev;
  const int32_t* bt_use = io->block_tables_dev;
  const int32_t* len_use = io->seq_lens_kv_dev;
  void* out_use = io->out_dev;
  float* lse_use = io->lse_dev;
  const bool q_in = io->q_dev == io->q_host;
  const bool bt_in = io->block_tables_dev == io->block_tables_host;
  const bool len_in = io->seq_lens_kv_dev != nullptr && io->seq_lens_kv_dev == io->seq_lens_kv_host;
  const bool out_in = io->out_dev == io->out_host;
  const bool lse_in = io->lse_dev != nullptr && io->lse_dev == io->lse_host;
  if (q_in || bt_in || len_in || out_in || lse_in) {
    int rc0 = check_device(p->device);
    if (rc0 != PKA_OK) return rc0;
  }
  if (q_in) q_use = host_mapped(io->q_host);
  if (bt_in) bt_use = static_cast<const int32_t*>(host_mapped(io->block_tables_host));
  if (len_in) len_use = static_cast<const int32_t*>(host_mapped(io->seq_lens_kv_host));
  if (out_in) out_use = host_mapped(io->out_host);
  if (lse_in) lse_use = static_cast<float*>(host_mapped(io->lse_host));
  PKA_CHECK_ARG(q_use && bt_use && out_use && (!lse_in || lse_use) && (!len_in || len_use),
                "a device array given as its host array must be page-locked host memory that "
                "the device can address");
  PKA_CHECK_ARG(aligned(q_use, 16) && aligned(out_use, 16) &&
                    (lse_use == nullptr || aligned(lse_use, 4)),
                "q_dev and out_dev must be 16-byte aligned, lse_dev 4-byte aligned");
  PKA_CHECK_ARG(aligned(k_pages, 16) && aligned(v_pages, 16) && kv_stride_page % 8 == 0 &&
                    kv_stride_head % 8 == 0,
                "K/V pools must be 16-byte aligned with strides that are multiples of 8");
  PKA_CHECK_ARG(workspace == nullptr || aligned(workspace, 256),
                "workspace must be 256-byte aligned");
  PKA_CHECK_ARG(batch_size >= 1, "batch_size must be >= 1 (got %d)", batch_size);
  int rc = check_device(p->device);
  if (rc != PKA_OK) return rc;

  // The input copies go first: their sizes follow from the host arrays alone,
  // so the GPU moves them while the host re-plans.  The query rows are counted
  // as the planner counts them (packed when qo_indptr is given).
  int64_t total_q = (int64_t)batch_size * p->desc.q_len;
  if (io->qo_indptr_host != nullptr) {
    const int32_t* ind = io->qo_indptr_host;
    PKA_CHECK_ARG(ind[0] == 0, "qo_indptr[0] must be 0 (got %d)", ind[0]);
    for (int32_t b = 0; b < batch_size; ++b)
      PKA_CHECK_ARG(ind[b + 1] > ind[b], "request %d has %lld query rows; packed rows must be >= 1",
                    b, (long long)ind[b + 1] - ind[b]);
    total_q = ind[batch_size];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)total_q * (size_t)p->Hq;
  const size_t out_elem = p->desc.out_dtype == PKA_DTYPE_F32 ? 4 : 2;
  if (!q_in)
    PKA_CUDA_TRY(cudaMemcpyAsync(io->q_dev, io->q_host, rows * p->D * 2, cudaMemcpyHostToDevice,
                                 s),
                 "cudaMemcpyAsync (q)");
  if (!bt_in)
    PKA_CUDA_TRY(cudaMemcpyAsync(io->block_tables_dev, io->block_tables_host,
                                 (size_t)batch_size * (size_t)io->bt_row_stride * sizeof(int32_t),
                                 cudaMemcpyHostToDevice, s),
                 "cudaMemcpyAsync (block tables)");
  if (!p->desc.freeze_seq_lens && !len_in)
    PKA_CUDA_TRY(cudaMemcpyAsync(io->seq_lens_kv_dev, io->seq_lens_kv_host,
                                 (size_t)batch_size * sizeof(int32_t), cudaMemcpyHostToDevice, s),
                 "cudaMemcpyAsync (lengths)");

  rc = paged_decode_plan_update(p, batch_size, io->seq_lens_kv_host, io->qo_indptr_host,
                                workspace_bytes_out, stream);
  if (rc != PKA_OK) return rc;
  if (p->total_q != total_q)
    return fail(PKA_ERR_INVALID_ARG, "the plan counts %d query rows, the step copied %lld",
                p->total_q, (long long)total_q);
  if (p->workspace_bytes > 0 && (workspace == nullptr || workspace_bytes < (size_t)p->workspace_bytes))
    return fail(PKA_ERR_WORKSPACE_TOO_SMALL, "workspace of %zu bytes, the plan needs %lld",
                workspace_bytes, (long long)p->workspace_bytes);
  rc = paged_decode_run(p, q_use, (int64_t)p->Hq * p->D, p->D, k_pages, v_pages, kv_stride_page,
                        kv_stride_head, bt_use, io->bt_row_stride, len_use, sinks, out_use,
                        p->desc.return_lse ? lse_use : nullptr, workspace, workspace_bytes,
                        stream);
  if (rc != PKA_OK) return rc;
  if (!out_in)
    PKA_CUDA_TRY(cudaMemcpyAsync(io->out_host, io->out_dev, rows * p->D * out_elem,
                                 cudaMemcpyDeviceToHost, s),
                 "cudaMemcpyAsync (out)");
  if (p->desc.return_lse && !lse_in)
    PKA_CUDA_TRY(cudaMemcpyAsync(io->lse_host, io->lse_dev, rows * sizeof(float),
                                 cudaMemcpyDeviceToHost, s),
                 "cudaMemcpyAsync (lse)");
  if (synchronize) PKA_CUDA_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  return PKA_OK;
}

int paged_decode_plan_check(const pka_plan* p, void* stream) {
  clear_error();
  PKA_CHECK_ARG(p != nullptr, "plan must not be NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->desc.flags & PKA_PLAN_HOST_ONLY) {
    // a host-only plan runs only through paged_decode_run_noalloc, whose
    // kernels report into the status word of its fixed scratch
    int32_t* word = nullptr;
    const int rc = noalloc_status_word(s, &word);
    if (rc != PKA_OK) return rc;
    return read_status(word, s);
  }
  PKA_CHECK_ARG(p->d_status != nullptr, "plan has no device state");
  return read_status(p->d_status, s);
}

// ---------------------------------------------------------------------------
// merge
// ---------------------------------------------------------------------------

int attn_merge_lse(const float* v_states, const float* s_states, int32_t num_states,
                   int32_t num_rows, int32_t num_heads, int32_t head_dim, void* v_out,
                   int32_t out_dtype, float* s_out, void* stream) {
  NvtxRange nvtx_range("pka::attn_merge_lse");
  clear_error();
  PKA_CHECK_ARG(v_states && s_states && v_out, "v_states, s_states and v_out must not be NULL");
  PKA_CHECK_ARG(num_states >= 1, "num_states must be >= 1");
  PKA_CHECK_ARG(num_rows >= 0 && num_heads >= 1, "bad row/head counts");
  PKA_CHECK_ARG(head_dim >= 4 && head_dim % 4 == 0 && head_dim <= 1024,
                "head_dim must be a multiple of 4 in [4, 1024]");
  if (out_dtype != PKA_DTYPE_BF16 && out_dtype != PKA_DTYPE_F16 && out_dtype != PKA_DTYPE_F32)
    return fail(PKA_ERR_UNSUPPORTED, "out_dtype must be bf16, f16 or f32");
  PKA_CHECK_ARG(aligned(v_states, 16) && aligned(v_out, 16),
                "v_states and v_out must be 16-byte aligned");
  return launch_merge_states(v_states, s_states, num_states, num_rows, num_heads, head_dim, v_out,
                             out_dtype, s_out, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// prefill
// ---------------------------------------------------------------------------

int batch_prefill_plan(pka_prefill_plan** plan_out, const pka_prefill_desc* desc,
                       const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                       size_t* workspace_bytes_out, int32_t* num_tiles_out, void* stream) {
  NvtxRange nvtx_range("pka::batch_prefill_plan");
  clear_error();
  PKA_CHECK_ARG(plan_out != nullptr && desc != nullptr, "plan_out and desc must not be NULL");
  *plan_out = nullptr;
  pka_prefill_plan* p = new (std::nothrow) pka_prefill_plan();
  if (p == nullptr) return fail(PKA_ERR_INVALID_ARG, "out of host memory");
  int rc = build_prefill_plan(*p, *desc, qo_indptr_host, kv_indptr_host);
  if (rc == PKA_OK && !(desc->flags & PKA_PLAN_HOST_ONLY))
    rc = upload_prefill_plan(*p, static_cast<cudaStream_t>(stream));
  if (rc != PKA_OK) {
    batch_prefill_plan_destroy(p);
    return rc;
  }
  if (workspace_bytes_out) *workspace_bytes_out = 0;
  if (num_tiles_out) *num_tiles_out = (int32_t)p->tiles.size();
  *plan_out = p;
  return PKA_OK;
}

int batch_prefill_plan_fixed(pka_prefill_plan** plan_out, const pka_prefill_desc* desc,
                             int32_t seq_len_q, int32_t seq_len_kv,
                             const int32_t* window_starts_host, const int32_t* window_ends_host,
                             size_t* workspace_bytes_out, int32_t* num_tiles_out, void* stream) {
  NvtxRange nvtx_range("pka::batch_prefill_plan_fixed");
  clear_error();
  PKA_CHECK_ARG(plan_out != nullptr && desc != nullptr, "plan_out and desc must not be NULL");
  *plan_out = nullptr;
  PKA_CHECK_ARG(desc->batch_size >= 1, "batch_size must be >= 1");
  PKA_CHECK_ARG(seq_len_q >= 1 && seq_len_kv >= 1, "seq_len_q and seq_len_kv must be >= 1");
  PKA_CHECK_ARG((int64_t)desc->batch_size * std::max(seq_len_q, seq_len_kv) <= INT32_MAX,
                "batch_size * seq_len exceeds 2^31 - 1 rows");
  std::vector<int32_t> qo(desc->batch_size + 1), kv(desc->batch_size + 1);
  for (int32_t b = 0; b <= desc->batch_size; ++b) {
    qo[b] = b * seq_len_q;
    kv[b] = b * seq_len_kv;
  }
  pka_prefill_plan* p = new (std::nothrow) pka_prefill_plan();
  if (p == nullptr) return fail(PKA_ERR_INVALID_ARG, "out of host memory");
  int rc = build_prefill_plan(*p, *desc, qo.data(), kv.data(), window_starts_host,
                              window_ends_host);
  if (rc == PKA_OK && !(desc->flags & PKA_PLAN_HOST_ONLY))
    rc = upload_prefill_plan(*p, static_cast<cudaStream_t>(stream));
  if (rc != PKA_OK) {
    batch_prefill_plan_destroy(p);
    return rc;
  }
  if (workspace_bytes_out) *workspace_bytes_out = 0;
  if (num_tiles_out) *num_tiles_out = (int32_t)p->tiles.size();
  *plan_out = p;
  return PKA_OK;
}

void batch_prefill_plan_destroy(pka_prefill_plan* plan) {
  if (plan == nullptr) return;
  if (plan->dev_buf != nullptr) cudaFree(plan->dev_buf);
  delete plan;
}

int batch_prefill_run(const pka_prefill_plan* p, const void* q, int64_t q_stride_tok,
                      int64_t q_stride_head, const void* k, const void* v, int64_t kv_stride_tok,
                      int64_t kv_stride_head, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("pka::batch_prefill_run");
  clear_error();
  (void)workspace;
  (void)workspace_bytes;
  PKA_CHECK_ARG(p != nullptr, "plan must not be NULL");
  PKA_CHECK_ARG(p->dev_buf != nullptr, "plan was built with PKA_PLAN_HOST_ONLY and cannot run");
  PKA_CHECK_ARG(q && k && v && out, "q, k, v and out must not be NULL");
  PKA_CHECK_ARG(!p->desc.return_lse || lse != nullptr, "the plan returns the LSE: lse is NULL");
  PKA_CHECK_ARG(aligned(out, 16), "out must be 16-byte aligned");
  PKA_CHECK_ARG(q_stride_tok % 8 == 0 && q_stride_head % 8 == 0 && kv_stride_tok % 8 == 0 &&
                    kv_stride_head % 8 == 0,
                "strides must be multiples of 8 elements");
  int rc = check_device(p->device);
  if (rc != PKA_OK) return rc;
  if (p->tiles.empty()) return PKA_OK;
  // q: (d, head, token) with 128-token boxes; k/v: (d, head, token) likewise
  CUtensorMap qmap, kmap, vmap;
  {
    const uint64_t dims[3] = {(uint64_t)p->D, (uint64_t)p->Hq, (uint64_t)p->total_q};
    const uint64_t strides[2] = {(uint64_t)q_stride_head * 2, (uint64_t)q_stride_tok * 2};
    const uint32_t box[3] = {64, 1, 128};
    rc = encode_bf16_map(&qmap, q, 3, dims, strides, box);
    if (rc != PKA_OK) return rc;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p->D, (uint64_t)p->Hkv, (uint64_t)p->total_kv};
    const uint64_t strides[2] = {(uint64_t)kv_stride_head * 2, (uint64_t)kv_stride_tok * 2};
    const uint32_t box[3] = {64, 1, 64};   // one 64-key tile per 64-column block
    rc = encode_bf16_map(&kmap, k, 3, dims, strides, box);
    if (rc != PKA_OK) return rc;
    rc = encode_bf16_map(&vmap, v, 3, dims, strides, box);
    if (rc != PKA_OK) return rc;
  }
  PrefillArgs a{};
  a.q = q;
  a.q_stride_tok = q_stride_tok;
  a.q_stride_head = q_stride_head;
  a.out = out;
  a.lse = p->desc.return_lse ? lse : nullptr;
  a.tiles = p->d_tiles;
  a.qo_indptr = p->d_qo;
  a.kv_indptr = p->d_kv;
  a.status = p->d_status;
  a.num_tiles = (int32_t)p->tiles.size();
  a.num_qo_heads = p->Hq;
  a.num_kv_heads = p->Hkv;
  a.group = p->G;
  a.causal = p->desc.mask == PKA_MASK_CAUSAL;
  a.window_left = p->desc.window_left;
  a.window_lo = p->d_win_lo;
  a.window_hi = p->d_win_hi;
  a.row_map = p->d_row_map;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.output_scale = p->desc.output_scale;
  a.out_dtype = p->desc.out_dtype;
  return launch_prefill_1h(*p, a, qmap, kmap, vmap, static_cast<cudaStream_t>(stream));
}

int batch_prefill_plan_check(const pka_prefill_plan* p, void* stream) {
  clear_error();
  PKA_CHECK_ARG(p != nullptr && p->d_status != nullptr, "plan has no device state");
  return read_status(p->d_status, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// test hook
// ---------------------------------------------------------------------------

int paged_kv_gather(const void* pages, int64_t num_pages, int64_t stride_page,
                    int64_t stride_head, int32_t num_kv_heads, int32_t page_size,
                    int32_t head_dim, const int32_t* block_tables, int64_t bt_row_stride,
                    int32_t request, int32_t kv_head, int32_t tok_begin, int32_t tok_end,
                    void* out, void* stream) {
  clear_error();
  PKA_CHECK_ARG(pages && block_tables && out, "pages, block_tables and out must not be NULL");
  if (head_dim != 128) return fail(PKA_ERR_UNSUPPORTED, "head_dim must be 128");
  if (page_size < 16 || page_size > 256 || page_size % 16 != 0)
    return fail(PKA_ERR_UNSUPPORTED, "page_size must be a multiple of 16 in [16, 256]");
  PKA_CHECK_ARG(kv_head >= 0 && kv_head < num_kv_heads, "kv_head out of range");
  PKA_CHECK_ARG(request >= 0 && tok_begin >= 0 && tok_end >= tok_begin, "bad token range");
  PKA_CHECK_ARG(aligned(out, 16), "out must be 16-byte aligned");
  CUtensorMap map;
  int rc = encode_kv_pool_map(&map, pages, num_pages, num_kv_heads, page_size, head_dim,
                              stride_page, stride_head);
  if (rc != PKA_OK) return rc;
  return launch_paged_gather(map, block_tables, bt_row_stride, page_size, request, kv_head,
                             tok_begin, tok_end, out, static_cast<cudaStream_t>(stream));
}

int paged_decode_check_tables(const pka_plan* p, const int32_t* block_tables,
                              int64_t bt_row_stride, const int32_t* seq_lens_kv_dev,
                              void* stream) {
  NvtxRange nvtx_range("pka::paged_decode_check_tables");
  clear_error();
  PKA_CHECK_ARG(p != nullptr && p->d_status != nullptr, "plan has no device state");
  PKA_CHECK_ARG(block_tables != nullptr, "block_tables must not be NULL");
  PKA_CHECK_ARG(bt_row_stride >= p->C, "bt_row_stride (%lld) is smaller than the table width %d",
                (long long)bt_row_stride, p->C);
  int rc = check_device(p->device);
  if (rc != PKA_OK) return rc;
  return launch_check_tables(p->d_items, (int32_t)p->items.size(), p->d_reqs, block_tables,
                             bt_row_stride, p->desc.freeze_seq_lens ? nullptr : seq_lens_kv_dev,
                             p->ps, p->desc.num_pages, p->d_status,
                             static_cast<cudaStream_t>(stream));
}

int pka_wait_timeout_probe(const pka_plan* plan, int32_t* status_dev, int64_t limit_ns,
                           void* stream) {
  clear_error();
  if (plan != nullptr && (plan->desc.flags & PKA_PLAN_HOST_ONLY)) {
    const int rc = noalloc_status_word(static_cast<cudaStream_t>(stream), &status_dev);
    if (rc != PKA_OK) return rc;
  } else if (plan != nullptr) {
    PKA_CHECK_ARG(plan->d_status != nullptr, "plan has no device state");
    status_dev = plan->d_status;
  }
  PKA_CHECK_ARG(status_dev != nullptr && aligned(status_dev, 4),
                "status_dev must be a 4-byte aligned device pointer");
  PKA_CHECK_ARG(limit_ns >= 1000000 && limit_ns <= 2000000000,
                "limit_ns must be in [1e6, 2e9] (got %lld)", (long long)limit_ns);
  return launch_wait_probe((uint64_t)limit_ns, status_dev, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
