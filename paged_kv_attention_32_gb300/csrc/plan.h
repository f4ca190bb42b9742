// Plan objects and the argument blocks handed to the kernels.  Shared by the
// host planner, the C-ABI layer and the kernel launchers; plain C++ types
// only, so that host-only translation units can include it.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "pka.h"

namespace pka {

// Per-request data the decode kernels read (32 bytes, one aligned load).
struct ReqInfo {
  int32_t q_start;    // first packed query row
  int32_t q_len;      // query rows of the request
  int32_t kv_len;     // key count seen by the planner (upper bound when not frozen)
  int32_t part_base;  // first fp32 partial row, -1 when the request is not split
  int32_t n_chunks;   // chunks the request's key range was cut into
  int32_t cnt_base;   // split requests: first of its merge counters (one per KV head and tile)
  int32_t pad1, pad2;
};

// One decode work item = one CTA: (request, kv head, chunk, pages [lo, hi)).
// Stored as int4 {request, (chunk << 16) | kv_head, page_lo, page_hi}.
struct WorkItem {
  int32_t request;
  int32_t head_chunk;
  int32_t page_lo;
  int32_t page_hi;
};

// Everything a decode kernel launch needs besides the two tensor maps.
struct DecodeArgs {
  const void* q;
  int64_t q_stride_tok;
  int64_t q_stride_head;
  const int32_t* block_tables;
  int64_t bt_row_stride;
  const int32_t* seq_lens_live;  // nullptr for a frozen plan
  const float* sinks;            // nullptr: no sink
  void* out;
  float* lse;                    // nullptr: no LSE output
  float* ws_o;                   // fp32 partial outputs [partial_rows, D]
  float* ws_lse;                 // fp32 partial base-2 LSE [partial_rows]
  const WorkItem* items;
  const ReqInfo* reqs;
  int32_t* merge_cnt;            // split requests: chunk CTAs done per (request, KV head, tile)
  int32_t* status;               // device error word (0 = fine)
  int32_t num_items;
  int32_t tiles_per_item;        // CTAs per work item (16-row tiles of the mma kernel, else 1)
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t group;                 // Hq / Hkv
  int32_t page_size;
  int32_t causal;
  int32_t window_left;
  int32_t rows_per_cta;          // group * max_q_len
  float scale_log2;              // scale * log2(e), folded into q
  float bmm2_scale;
  int32_t in_f16;                // q/K/V are IEEE half (else bf16)
  int32_t out_dtype;             // PKA_DTYPE_BF16 / F16 / F32
};

// Device error word bits (OR-ed by kernels, read by paged_decode_status).
enum : int32_t {
  STATUS_WAIT_TIMEOUT = 1,  // an mbarrier wait hit its iteration limit
  STATUS_PAGE_BOUNDS = 2,   // paged_decode_check_tables found an entry outside [0, num_pages)
};

}  // namespace pka

// The opaque decode plan of the C ABI.
struct pka_plan {
  pka_decode_desc desc;       // normalised copy (defaults filled in)
  int32_t B = 0, Hq = 0, Hkv = 0, G = 0, D = 0, ps = 0, C = 0;
  int32_t total_q = 0, max_q_len = 0, rows_per_cta = 0;
  int32_t kernel = 0, chunk_pages = 0, num_split = 0, partial_rows = 0;
  int64_t workspace_bytes = 0;
  int64_t ws_lse_offset = 0;  // byte offset of the partial LSEs in the workspace
  float scale = 0.f;
  std::vector<pka::ReqInfo> reqs;
  std::vector<int32_t> page_lo, page_hi, order;
  std::vector<pka::WorkItem> items;
  int32_t num_merge_counters = 0;   // split requests: Hkv x tiles per item each
  // one device allocation holding items | reqs | status word | merge counters
  void* dev_buf = nullptr;
  size_t dev_capacity = 0;    // bytes of dev_buf (reused by paged_decode_plan_update)
  const pka::WorkItem* d_items = nullptr;
  const pka::ReqInfo* d_reqs = nullptr;
  int32_t* d_status = nullptr;
  int32_t* d_merge_cnt = nullptr;
  int device = -1;
  // pinned host image of dev_buf: a replan writes it and uploads it with one
  // asynchronous copy; stage_done marks when that copy has read it
  void* host_stage = nullptr;
  size_t host_capacity = 0;
  cudaEvent_t stage_done = nullptr;
};

namespace pka {

// Fills `plan` (host arrays only) following the written plan specification:
// visited pages per request, chunk choice under the CTA target, longest-first
// item order, partial-row bases and workspace size.  Returns PKA_OK or an
// error code (message recorded).
int build_decode_plan(pka_plan& plan, const pka_decode_desc& desc, const int32_t* seq_lens_kv,
                      const int32_t* qo_indptr);

}  // namespace pka
