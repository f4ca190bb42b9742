// Kernel launchers (defined in the .cu files, called by the C-ABI layer).
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "plan.h"

namespace pka {

// Decode kernel (CUDA-core or mma variant, as the plan chose); the partials of
// a split request are merged inside it by the last chunk CTA of each group.
int launch_decode(const pka_plan& plan, const DecodeArgs& args, const CUtensorMap& kmap,
                  const CUtensorMap& vmap, cudaStream_t stream);

// Standalone merge of [N, S, H, D] fp32 states by their base-2 LSEs.
int launch_merge_states(const float* v_states, const float* s_states, int32_t n, int32_t s,
                        int32_t h, int32_t d, void* v_out, int32_t out_dtype, float* s_out,
                        cudaStream_t stream);

// Checks the block-table entries a run of the plan reads (see pka.h,
// paged_decode_check_tables); a bad one sets STATUS_PAGE_BOUNDS in *status.
int launch_check_tables(const WorkItem* items, int32_t num_items, const ReqInfo* reqs,
                        const int32_t* tables, int64_t row_stride, const int32_t* seq_lens_live,
                        int32_t page_size, int64_t num_pages, int32_t* status,
                        cudaStream_t stream);

// One warp waiting on a barrier nothing completes, bounded by limit_ns: the
// timeout bit ends up in *status (device int32).
int launch_wait_probe(uint64_t limit_ns, int32_t* status, cudaStream_t stream);

// Device address of the status word of paged_decode_run_noalloc's fixed
// scratch on the current device (set up on first use, on `stream`).
int noalloc_status_word(cudaStream_t stream, int32_t** out);

// Test hook: paged rows -> dense rows through the decode kernels' addressing.
int launch_paged_gather(const CUtensorMap& map, const int32_t* block_tables,
                        int64_t bt_row_stride, int32_t page_size, int32_t request,
                        int32_t kv_head, int32_t tok_begin, int32_t tok_end, void* out,
                        cudaStream_t stream);

}  // namespace pka
