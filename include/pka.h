/*
 * pka.h -- C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * Operations (FlashInfer API documentation pages they follow):
 *   paged_decode_plan / paged_decode_run
 *       batched decode attention over a paged KV cache:
 *       "flashinfer.attention.prims_ts.batch_decode_with_paged_kv_cache"
 *       (plan-before-capture, fixed or packed query, mask_type, window_left,
 *       bmm1_scale / bmm2_scale) and
 *       "flashinfer.cudnn.cudnn_batch_decode_with_kv_cache"
 *       (HND k_cache / v_cache, q_len_per_req causal rows, sinks, the base-2
 *       LSE of the Note "LSE convention").
 *   attn_merge_lse
 *       merge of partial attention states by base-2 LSE (the "cascade-merge"
 *       input named in the LSE convention of cudnn_batch_decode_with_kv_cache).
 *   batch_prefill_plan / batch_prefill_run
 *       packed ragged causal context attention:
 *       "flashinfer.attention.prims_ts.batch_prefill".
 *   paged_decode_step_host
 *       one decode step from host buffers: copies in, re-plan, run, copies
 *       out, queued in order on one stream.
 *   paged_decode_check_tables
 *       validation of the block-table entries a decode run reads.
 *   paged_kv_gather
 *       test hook: copies paged K or V rows to a dense buffer through the same
 *       page addressing the decode kernels use.
 *   pka_wait_timeout_probe
 *       test hook: runs the kernels' bounded wait until it gives up, so that
 *       the timeout report can be checked without faulting or hanging.
 *
 * Conventions shared by every entry point
 *   - Return value: PKA_OK (0) or a negative PKA_ERR_* code.  The message of
 *     the last error on the calling thread is returned by pka_last_error().
 *   - All arguments are checked on the host before any kernel is launched; an
 *     invalid argument launches no kernel (paged_decode_step_host may have
 *     queued its input copies by then, see there).  No kernel traps or asserts.
 *   - Device pointers are raw CUDA device addresses of the current device.
 *     `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - Element strides are in elements, not bytes.
 *   - q/K/V are bf16 (PKA_DTYPE_BF16) or IEEE half (PKA_DTYPE_F16), one type
 *     for all three, chosen by the plan's `dtype` (cudnn_batch_decode_with_kv_cache,
 *     q: float16 or bfloat16); the output is bf16, f16 or fp32, chosen by the
 *     plan's `out_dtype` (out_dtype of batch_decode_with_paged_kv_cache and
 *     batch_prefill).  head_dim is 128 for decode and 128 or 256 for prefill
 *     (batch_prefill allows those two head sizes).
 *   - The caller owns every device buffer (q, pools, tables, lengths, out,
 *     lse, workspace).  The library owns only the opaque plan objects.
 *   - paged_decode_run and batch_prefill_run allocate nothing, never
 *     synchronise and never read device memory on the host, so they may be
 *     captured in a CUDA graph.  Plans must be created before capture.
 *   - Prefill, like decode, is split into a host plan (batch_prefill_plan,
 *     made from host copies of the indptr arrays, before any capture) and a
 *     run (batch_prefill_run): batch_decode_with_paged_kv_cache's planner note
 *     asks for exactly this split so that the run stays capturable.
 */
#ifndef PKA_H
#define PKA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define PKA_OK 0
#define PKA_ERR_INVALID_ARG (-1)          /* a shape, length or pointer check failed   */
#define PKA_ERR_UNSUPPORTED (-2)          /* valid on the pages, not built here        */
#define PKA_ERR_WORKSPACE_TOO_SMALL (-3)  /* workspace_bytes below the plan's need     */
#define PKA_ERR_CUDA (-4)                 /* a CUDA runtime/driver call failed         */
#define PKA_ERR_DEVICE_BOUNDS (-5)        /* a block-table entry outside the pool      */
#define PKA_ERR_DEVICE_TIMEOUT (-6)       /* a kernel gave up on a bounded wait        */

/* ---- enums ------------------------------------------------------------- */
#define PKA_DTYPE_BF16 0
#define PKA_DTYPE_F16 1
#define PKA_DTYPE_F32 2

#define PKA_MASK_DENSE 0   /* mask_type 'dense': only padding is masked            */
#define PKA_MASK_CAUSAL 1  /* mask_type 'causal': bottom-right aligned diagonal     */
#define PKA_MASK_VARIABLE_WINDOW 2 /* prefill, fixed shape only: per-query inclusive key
                                      bounds (batch_prefill, mask_type 'variable_window') */

#define PKA_PLAN_HOST_ONLY 1  /* build the plan on the host only (no device copy);
                                 such a plan can be inspected but not run        */

#define PKA_KERNEL_CUDA_CORE 0  /* decode kernel on CUDA cores (FFMA2 + shuffles) */
#define PKA_KERNEL_MMA 1        /* decode kernel on tensor cores (mma m16n8k16)   */

/* Message of the last error raised on the calling thread ("" if none). */
const char* pka_last_error(void);

/* Library version string. */
const char* pka_version(void);

/* ======================================================================== */
/* Paged decode                                                              */
/* ======================================================================== */

/*
 * Problem description for a decode plan.
 *
 * batch_size         B, number of requests.
 * num_qo_heads       Hq.  num_kv_heads Hkv.  Hq % Hkv == 0 is required
 *                    (GQA/MQA: query head h reads KV head h / (Hq/Hkv);
 *                    cudnn_batch_decode_with_kv_cache, Note).
 * head_dim           D; must be 128.
 * page_size          tokens per page: a multiple of 16 in [16, 256].
 * max_pages_per_seq  C, the number of entries in each block_tables row.
 * num_pages          pages in each of the K and V pools.
 * dtype              PKA_DTYPE_BF16 or PKA_DTYPE_F16: q and the K/V pools.
 * q_len              fixed query rows per request, used when the plan gets no
 *                    qo_indptr (batch_decode_with_paged_kv_cache, seq_len_q).
 * max_q_len          packed mode: per-request capacity (0 = derive from
 *                    qo_indptr); fixed mode: 0 or equal to q_len, anything
 *                    else is PKA_ERR_INVALID_ARG (same page, max_seq_len_q).
 * mask               PKA_MASK_DENSE or PKA_MASK_CAUSAL.  Causal row i of a
 *                    request with L rows and n keys sees keys 0 .. n-L+i
 *                    (cudnn_batch_decode_with_kv_cache, q_len_per_req).
 * window_left        -1 disables; W >= 0 keeps the W keys before the row's
 *                    diagonal position n-L+i plus that position
 *                    (same page, window_left).  With mask DENSE the window is
 *                    anchored at the same diagonal position.
 * scale              softmax scale on q.k; NaN selects 1/sqrt(D)
 *                    (bmm1_scale / scale).
 * bmm2_scale         multiplies O (not the LSE).
 * return_lse         nonzero: paged_decode_run writes the base-2 LSE.
 * freeze_seq_lens    nonzero: the plan keeps the host lengths and run ignores
 *                    its seq_lens_kv_dev argument.  Zero: run reads the live
 *                    lengths from seq_lens_kv_dev; each must be >= its q_len
 *                    and <= the length the plan saw (lengths above that are
 *                    clamped to it), and the window start is then found at
 *                    run time (batch_decode_with_paged_kv_cache, planner note:
 *                    a captured run either reads a length tensor that stays
 *                    in place or uses lengths kept in the plan).
 * num_sms            SM count the planner balances for; 0 = the device's.
 * split_waves        target CTAs = split_waves * num_sms; 0 = the environment
 *                    variable PKA_SPLIT_WAVES if set to a positive integer, else 2.
 * min_chunk_tokens   smallest split chunk in tokens; 0 = PKA_MIN_CHUNK_TOKENS,
 *                    else 256.
 * mma_min_rows       the tensor-core kernel is used when
 *                    (Hq/Hkv) * max_q_len >= mma_min_rows (or > 8, the rows
 *                    the CUDA-core kernel holds); 0 = PKA_MMA_MIN_ROWS, else 1
 *                    (the tensor-core kernel always; a higher value keeps
 *                    narrower groups on the CUDA-core kernel).
 *                    paged_decode_plan_info reports the values used.
 * flags              PKA_PLAN_HOST_ONLY or 0.
 * out_dtype          PKA_DTYPE_BF16, PKA_DTYPE_F16 or PKA_DTYPE_F32: O of
 *                    paged_decode_run (batch_decode_with_paged_kv_cache,
 *                    out_dtype; a zeroed descriptor means bf16).
 */
typedef struct pka_decode_desc {
  int32_t batch_size;
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t max_pages_per_seq;
  int64_t num_pages;
  int32_t dtype;
  int32_t q_len;
  int32_t max_q_len;
  int32_t mask;
  int32_t window_left;
  float scale;
  float bmm2_scale;
  int32_t return_lse;
  int32_t freeze_seq_lens;
  int32_t num_sms;
  int32_t split_waves;
  int32_t min_chunk_tokens;
  int32_t mma_min_rows;
  int32_t flags;
  int32_t out_dtype;
} pka_decode_desc;

typedef struct pka_plan pka_plan; /* opaque decode plan */

/* Summary of a decode plan. */
typedef struct pka_plan_info {
  int32_t num_items;        /* work items = CTAs of the decode kernel              */
  int32_t chunk_pages;      /* split chunk length in pages                          */
  int32_t num_split;        /* requests cut into more than one chunk                */
  int32_t partial_rows;     /* fp32 partial rows in the workspace                   */
  int64_t workspace_bytes;  /* bytes paged_decode_run needs in `workspace`          */
  int32_t kernel;           /* PKA_KERNEL_CUDA_CORE or PKA_KERNEL_MMA               */
  int32_t rows_per_cta;     /* query rows per KV head, (Hq/Hkv) * max_q_len: one
                               CTA holds them all (CUDA-core kernel, <= 8) or one
                               16-row tile of them (tensor-core kernel, <= 65536) */
  int32_t num_sms;          /* SM count the plan balanced for                       */
  int32_t split_waves;
  int32_t min_chunk_tokens;
  int32_t total_q;          /* query rows in the batch                              */
} pka_plan_info;

/*
 * Build a decode plan from host copies of the lengths.
 *
 * seq_lens_kv_host  [B] int32 host array, 1 <= kv_len <= C*page_size and
 *                   kv_len >= the request's q_len (cudnn_batch_decode_with_kv_cache,
 *                   q_len_per_req: no request may have fewer keys than query rows).
 * qo_indptr_host    NULL (fixed q_len) or [B+1] int32 host array, cumulative
 *                   query offsets starting at 0, every q_len >= 1 (packed mode,
 *                   batch_decode_with_paged_kv_cache, qo_indptr).
 * workspace_bytes_out  receives the workspace size paged_decode_run needs
 *                   (0 when no request is split).
 * stream            stream for the upload of the plan's device arrays.
 *
 * The plan (host arrays plus one device buffer for the work list) is owned
 * by the library until paged_decode_plan_destroy.  Planning reads lengths on
 * the host, so do it before graph capture.
 */
int paged_decode_plan(pka_plan** plan_out, const pka_decode_desc* desc,
                      const int32_t* seq_lens_kv_host, const int32_t* qo_indptr_host,
                      size_t* workspace_bytes_out, void* stream);

/*
 * Re-plan an existing plan for a new batch (new lengths, query offsets and
 * batch size; every other descriptor field stays), as a serving loop does
 * each step.  The plan's device buffer is reused when the new work list fits
 * (no allocation, no device synchronisation), else reallocated with headroom.
 * The new work list goes up in one asynchronous copy from a pinned host image
 * that the plan keeps; the call first waits (on the host) until the previous
 * upload of this plan has read that image, which it normally has long since.
 * The upload is ordered on `stream` after earlier runs queued there; a run
 * on another stream must be ordered by the caller.  On error the plan is
 * unchanged.  workspace_bytes_out as for paged_decode_plan.
 */
int paged_decode_plan_update(pka_plan* plan, int32_t batch_size, const int32_t* seq_lens_kv_host,
                             const int32_t* qo_indptr_host, size_t* workspace_bytes_out,
                             void* stream);

/* Free a plan (NULL is ignored).  Must not be called while a run that uses
 * the plan may still execute on the device; waits for the plan's last upload. */
void paged_decode_plan_destroy(pka_plan* plan);

/* Fill `info` with the plan's summary. */
int paged_decode_plan_info(const pka_plan* plan, pka_plan_info* info);

/*
 * Copy the plan's host arrays out (for bit-exact tests of the planner).
 * items     [num_items * 5] int32: (request, kv_head, chunk, page_lo, page_hi)
 *           in launch order; page_lo/page_hi index the request's table row.
 * n_chunks, part_base, page_lo, page_hi  [B] int32 each (part_base -1 when
 *           the request is not split).
 * order     [B] int32: requests in launch order.
 * Any output pointer may be NULL.
 */
int paged_decode_plan_export(const pka_plan* plan, int32_t* items, int32_t* n_chunks,
                             int32_t* part_base, int32_t* page_lo, int32_t* page_hi,
                             int32_t* order);

/*
 * Run the planned decode.
 *
 * q               the plan's dtype (bf16 or f16), rows [total_q] x heads [Hq] x D;
 *                 element (t, h, d) at
 *                 q + t*q_stride_tok + h*q_stride_head + d.  D innermost and
 *                 dense; other strides free (cudnn_batch_decode_with_kv_cache,
 *                 Note: q may be a strided view, e.g. part of a fused QKV output).
 *                 Strides must be multiples of 8 elements.
 * k_pages, v_pages  HND pools: element (page, kv_head, slot, d) at
 *                 base + page*kv_stride_page + kv_head*kv_stride_head + slot*D + d
 *                 (k_cache / v_cache shapes (total_num_pages, num_heads_kv,
 *                 page_size, head_dim)).  Strides multiples of 8 elements,
 *                 bases 16-byte aligned.  A combined K/V tensor is passed as
 *                 two base pointers with its strides.
 * block_tables    int32 [B, C] device, row b at block_tables + b*bt_row_stride;
 *                 token t of request b is in page block_tables[b, t/page_size],
 *                 slot t % page_size (batch_decode_with_paged_kv_cache,
 *                 block_tables).  Entries past a request's last page are not read.
 * seq_lens_kv_dev int32 [B] device; read only when the plan is not frozen
 *                 (may be NULL for a frozen plan).
 * sinks           NULL or fp32 [Hq] device: per-head sink logits joining each
 *                 row's softmax denominator with a zero value row
 *                 (cudnn_batch_decode_with_kv_cache, sinks).
 * out             the plan's out_dtype (bf16, f16 or fp32), [total_q, Hq, D]
 *                 contiguous, 16-byte aligned.
 * lse             NULL or fp32 [total_q, Hq] contiguous: log2 of the sum over
 *                 the row's valid keys of exp(scale * q.k) -- the sink is not
 *                 included (Note "LSE convention").  Required when the plan
 *                 has return_lse.
 * workspace       device scratch of at least the plan's workspace_bytes
 *                 (256-byte aligned); holds fp32 split-KV partials.
 *
 * A request cut into chunks is merged inside the decode kernel: the chunk CTA
 * that finishes last combines the partials, counted on counters in the plan's
 * device buffer (zero between runs).  Runs that use one plan must therefore
 * not overlap on the GPU (queue them on one stream, or order the streams).
 */
int paged_decode_run(const pka_plan* plan, const void* q, int64_t q_stride_tok,
                     int64_t q_stride_head, const void* k_pages, const void* v_pages,
                     int64_t kv_stride_page, int64_t kv_stride_head,
                     const int32_t* block_tables, int64_t bt_row_stride,
                     const int32_t* seq_lens_kv_dev, const float* sinks, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Host-buffer I/O of one decode step (paged_decode_step_host).  Host arrays
 * should be pinned (page-locked) for the copies to be asynchronous; device
 * staging arrays are the caller's and hold at least the sizes below.
 *
 * In place: a device array may be given as its host array itself (the same
 * pointer: q_dev == q_host, block_tables_dev == block_tables_host,
 * seq_lens_kv_dev == seq_lens_kv_host, out_dev == out_host, lse_dev ==
 * lse_host).  It must then be page-locked host memory that the device can
 * address (checked with cudaPointerGetAttributes, else PKA_ERR_INVALID_ARG):
 * the step copies nothing for it, and the kernels read (q, table rows, live
 * lengths) or write (O, LSE) it where it is, over the host link (NVLink-C2C
 * on a Grace-Blackwell node).  Such arrays must not be touched by the host
 * while the step runs.
 *
 * q_host, q_dev            [total_q, Hq, D] dense, the plan's input type.
 * block_tables_host, _dev  [batch_size, bt_row_stride] int32 (as for
 *                          paged_decode_run); the whole rows are copied.
 * seq_lens_kv_host         [batch_size] int32: the step's key lengths, which
 *                          the step re-plans on.
 * seq_lens_kv_dev          [batch_size] int32 device, or NULL when the plan
 *                          freezes the lengths (they then travel in the plan).
 * qo_indptr_host           [batch_size + 1] int32, or NULL for the plan's
 *                          fixed q_len.
 * out_dev, out_host        [total_q, Hq, D] dense, the plan's output type.
 * lse_dev, lse_host        [total_q, Hq] fp32; required when the plan returns
 *                          the LSE, else ignored.
 */
typedef struct pka_decode_host_io {
  const void* q_host;
  const int32_t* block_tables_host;
  const int32_t* seq_lens_kv_host;
  const int32_t* qo_indptr_host;
  void* out_host;
  float* lse_host;
  void* q_dev;
  int32_t* block_tables_dev;
  int32_t* seq_lens_kv_dev;
  void* out_dev;
  float* lse_dev;
  int64_t bt_row_stride;
} pka_decode_host_io;

/*
 * One decode step from host buffers, as a serving loop runs it: copy q, the
 * block table rows (and the live lengths) host -> device, re-plan `plan` on
 * the step's lengths (paged_decode_plan_update), run the decode over the
 * device-resident K/V pools (arguments as for paged_decode_run, with dense q),
 * and copy O (and the LSE) device -> host, all queued on `stream` in that
 * order (the input copies first, so that the GPU moves them while the host
 * re-plans).  With `synchronize` nonzero the call returns once O is in host
 * memory; otherwise the caller synchronises `stream` before reading it.
 * workspace_bytes_out (may be NULL) receives the re-planned workspace size.
 * The io, the pointers and the query rows (qo_indptr_host) are checked
 * before anything is queued.  A re-plan that fails leaves the plan unchanged,
 * with only the input copies queued.  PKA_ERR_WORKSPACE_TOO_SMALL means the
 * plan was re-planned (its upload queued after the input copies) but needs
 * more workspace than given: the run and the output copies were not queued.
 */
int paged_decode_step_host(pka_plan* plan, int32_t batch_size, const pka_decode_host_io* io,
                           const void* k_pages, const void* v_pages, int64_t kv_stride_page,
                           int64_t kv_stride_head, const float* sinks, void* workspace,
                           size_t workspace_bytes, size_t* workspace_bytes_out,
                           int32_t synchronize, void* stream);

/*
 * Wait for `stream`, then read and clear the plan's device status word, which
 * kernels set instead of trapping: returns PKA_OK; PKA_ERR_DEVICE_TIMEOUT when
 * some kernel of an earlier run gave up on a bounded (2 s) wait (the outputs
 * of that run are then not valid); or PKA_ERR_DEVICE_BOUNDS when
 * paged_decode_check_tables found a block-table entry outside [0, num_pages).
 * For a PKA_PLAN_HOST_ONLY plan the word read is the one that
 * paged_decode_run_noalloc's kernels report into on the current device,
 * shared by every no-allocation run there: it collects them all since the
 * last check.  Reading it allocates nothing.  Synchronises; not for capture.
 */
int paged_decode_plan_check(const pka_plan* plan, void* stream);

/*
 * Validate, on the device, the block-table entries that paged_decode_run with
 * this plan would read: for every request, the pages its visited keys lie in
 * (the window's start on; up to the live length from seq_lens_kv_dev when the
 * plan does not freeze the lengths, which may then be NULL only if frozen).
 * An entry outside [0, num_pages) sets the plan's status word, which the next
 * paged_decode_plan_check reports as PKA_ERR_DEVICE_BOUNDS.  A run never reads
 * outside the pools: an out-of-range entry's copy reads zeros (TMA bounds), so
 * this check is what makes such a table visible.  One small launch, reading
 * only the entries; allocates nothing; does not synchronise.
 */
int paged_decode_check_tables(const pka_plan* plan, const int32_t* block_tables,
                              int64_t bt_row_stride, const int32_t* seq_lens_kv_dev,
                              void* stream);

/*
 * paged_decode_run without any device allocation.  The pages have no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc themselves -- code inside an allocator hook, or a serving
 * process whose device memory is a fixed pool it does not control.  Together
 * with a plan built with PKA_PLAN_HOST_ONLY the whole decode allocates
 * nothing on the device.
 *
 * Arguments are those of paged_decode_run without the workspace.  The plan's
 * work list and the split-KV fp32 partials go to one fixed 16 MiB device
 * array inside the library (held on every GPU that loads the library until
 * the process exits); a plan that needs more returns
 * PKA_ERR_WORKSPACE_TOO_SMALL -- use paged_decode_run for it.
 *
 * - The first call on a device looks up that array's device address
 *   (cudaGetSymbolAddress) with the device current; make that first call
 *   before any stream capture.
 * - Every call on a device shares the one array and overwrites what the
 *   previous call left there; calls whose executions overlap on the GPU (on
 *   different streams, or from different threads) race and give wrong
 *   results.  Serialise them.
 * - The call copies the plan's host arrays into the array with
 *   cudaMemcpyAsync; it calls no allocating routine.
 * - Kernels that give up on a bounded wait report it in a status word at the
 *   start of the array (cleared once at the first call on the device, then
 *   only by a check): paged_decode_plan_check on a PKA_PLAN_HOST_ONLY plan
 *   reads and clears it, reporting every no-allocation run since the last
 *   check.
 * - A plan with a device copy must be run on the device it was made on; a
 *   host-only plan runs on the current device.
 */
int paged_decode_run_noalloc(const pka_plan* plan, const void* q, int64_t q_stride_tok,
                             int64_t q_stride_head, const void* k_pages, const void* v_pages,
                             int64_t kv_stride_page, int64_t kv_stride_head,
                             const int32_t* block_tables, int64_t bt_row_stride,
                             const int32_t* seq_lens_kv_dev, const float* sinks, void* out,
                             float* lse, void* stream);

/* ======================================================================== */
/* LSE merge                                                                 */
/* ======================================================================== */

/*
 * Merge num_states partial attention results of the same rows.
 *
 * v_states   fp32 [num_states, num_rows, num_heads, head_dim] contiguous:
 *            each state's normalised output over its own key subset.
 * s_states   fp32 [num_states, num_rows, num_heads] contiguous: each state's
 *            base-2 LSE (-inf for an empty subset).
 * v_out      [num_rows, num_heads, head_dim] contiguous, out_dtype
 *            PKA_DTYPE_BF16, PKA_DTYPE_F16 or PKA_DTYPE_F32:
 *            sum_i 2^(s_i - m) v_i / sum_i 2^(s_i - m), m = max_i s_i.
 * s_out      NULL or fp32 [num_rows, num_heads]: m + log2 sum_i 2^(s_i - m).
 * Rows whose states are all -inf get v = 0 and s = -inf.
 * head_dim must be a multiple of 4 (<= 1024); num_states >= 1; v_states and
 * v_out 16-byte aligned.  With head_dim 128 the states stream through shared
 * memory by bulk copies under bounded waits; a wait that gives up (the copies
 * read only the caller's arrays, so this means a failing device) leaves v_out
 * and s_out unwritten and sets the timeout bit of the device status word of
 * the library's fixed scratch, which paged_decode_plan_check on a
 * PKA_PLAN_HOST_ONLY plan reads.  The first call on a device sets that word
 * up (one cudaMemsetAsync on `stream`).
 */
int attn_merge_lse(const float* v_states, const float* s_states, int32_t num_states,
                   int32_t num_rows, int32_t num_heads, int32_t head_dim, void* v_out,
                   int32_t out_dtype, float* s_out, void* stream);

/* ======================================================================== */
/* Ragged causal prefill                                                     */
/* ======================================================================== */

/*
 * batch_size, num_qo_heads, num_kv_heads as for decode; head_dim 128 or 256.
 * mask         PKA_MASK_CAUSAL (bottom-right aligned) or PKA_MASK_DENSE.
 * window_left  -1 disables; W >= 0 keeps, for query row i of a request with
 *              Lq rows and Lk keys, the keys from Lk - Lq + i - W on (the plain
 *              sliding window of the decode entry points; batch_prefill lists
 *              window_left, and its head-paired GQA policy is not built).
 * sm_scale     NaN selects 1/sqrt(D) (batch_prefill, sm_scale).
 * output_scale multiplies O (batch_prefill, output_scale).
 * return_lse   nonzero: batch_prefill_run writes the base-2 LSE.
 * num_sms      0 = the device's.   flags  PKA_PLAN_HOST_ONLY or 0.
 * dtype        PKA_DTYPE_BF16 or PKA_DTYPE_F16: q, k and v.
 * out_dtype    PKA_DTYPE_BF16, PKA_DTYPE_F16 or PKA_DTYPE_F32: O (batch_prefill,
 *              out_dtype; a zeroed descriptor means bf16).
 */
typedef struct pka_prefill_desc {
  int32_t batch_size;
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t dtype;
  int32_t mask;
  int32_t window_left;
  float sm_scale;
  float output_scale;
  int32_t return_lse;
  int32_t num_sms;
  int32_t flags;
  int32_t out_dtype;
} pka_prefill_desc;

typedef struct pka_prefill_plan pka_prefill_plan; /* opaque prefill plan */

/*
 * Build the tile schedule of a packed ragged prefill (mask CAUSAL or DENSE;
 * PKA_MASK_VARIABLE_WINDOW needs the fixed-shape planner below).
 * qo_indptr_host, kv_indptr_host  [B+1] int32 host arrays, cumulative offsets
 *           starting at 0 (batch_prefill, qo_indptr / kv_indptr).  For a
 *           causal mask every request needs kv_len >= q_len.
 * workspace_bytes_out  receives 0 (the prefill needs no workspace).
 * num_tiles_out  NULL or receives the number of CTAs batch_prefill_run launches.
 */
int batch_prefill_plan(pka_prefill_plan** plan_out, const pka_prefill_desc* desc,
                       const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                       size_t* workspace_bytes_out, int32_t* num_tiles_out, void* stream);

/*
 * Build the tile schedule of a fixed-shape prefill (batch_prefill with
 * [B, S, H, D] storage and no offset tensors): q [B, seq_len_q, Hq, D] and k, v
 * [B, seq_len_kv, Hkv, D], run by batch_prefill_run as a packed batch whose B
 * requests all have seq_len_q queries and seq_len_kv keys (token t of request
 * b is row b * seq_len + t).
 * mask       PKA_MASK_CAUSAL, PKA_MASK_DENSE or PKA_MASK_VARIABLE_WINDOW.
 * window_starts_host, window_ends_host  with PKA_MASK_VARIABLE_WINDOW: [B,
 *            seq_len_q] int32 host arrays of inclusive key bounds, 0 <= start
 *            <= end < seq_len_kv (batch_prefill, variable_window_token_starts /
 *            _ends; query row q of request b sees keys start[b, q] .. end[b, q]);
 *            the plan keeps a device copy.  NULL with the other masks.
 * Errors: INVALID_ARG for bounds outside that range, a bound array missing or
 * given with another mask, seq_len_q < 1, seq_len_kv < 1.
 */
int batch_prefill_plan_fixed(pka_prefill_plan** plan_out, const pka_prefill_desc* desc,
                             int32_t seq_len_q, int32_t seq_len_kv,
                             const int32_t* window_starts_host, const int32_t* window_ends_host,
                             size_t* workspace_bytes_out, int32_t* num_tiles_out, void* stream);

void batch_prefill_plan_destroy(pka_prefill_plan* plan);

/* As paged_decode_plan_check, for the prefill plan's device status word. */
int batch_prefill_plan_check(const pka_prefill_plan* plan, void* stream);

/*
 * Run the planned prefill.
 * q      the plan's dtype (bf16 or f16), packed [total_q, Hq, D]: (t, h, d) at
 *        q + t*q_stride_tok + h*q_stride_head + d.
 * k, v   the plan's dtype, packed [total_kv, Hkv, D]: (t, h, d) at
 *        base + t*kv_stride_tok + h*kv_stride_head + d.
 *        All strides multiples of 8 elements, bases 16-byte aligned.
 * out    the plan's out_dtype (bf16, f16 or fp32), [total_q, Hq, D] contiguous,
 *        16-byte aligned.
 * lse    NULL or fp32 [total_q, Hq] contiguous base-2 LSE (required with return_lse).
 * workspace, workspace_bytes  unused (the prefill needs none); may be NULL, 0.
 */
int batch_prefill_run(const pka_prefill_plan* plan, const void* q, int64_t q_stride_tok,
                      int64_t q_stride_head, const void* k, const void* v, int64_t kv_stride_tok,
                      int64_t kv_stride_head, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, void* stream);

/* ======================================================================== */
/* Test hook                                                                 */
/* ======================================================================== */

/*
 * Copy tokens [tok_begin, tok_end) of request `request`, KV head `kv_head`,
 * from an HND pool (layout as for paged_decode_run) into `out`
 * (bf16 [tok_end - tok_begin, head_dim] contiguous), through the same tensor
 * map, page coordinates and shared-memory swizzle the decode kernels use.
 * The caller guarantees that every table entry read is a valid page.
 */
int paged_kv_gather(const void* pages, int64_t num_pages, int64_t stride_page,
                    int64_t stride_head, int32_t num_kv_heads, int32_t page_size,
                    int32_t head_dim, const int32_t* block_tables, int64_t bt_row_stride,
                    int32_t request, int32_t kv_head, int32_t tok_begin, int32_t tok_end,
                    void* out, void* stream);

/*
 * Exercise the bounded wait every kernel uses: one warp waits on a barrier
 * phase that nothing completes, gives up after limit_ns nanoseconds (1e6 to
 * 2e9), ORs the timeout bit (1) into a status word and returns; the context
 * stays usable.  The status word is the decode plan's own when `plan` is not
 * NULL (paged_decode_plan_check then returns PKA_ERR_DEVICE_TIMEOUT, and
 * clears it) -- for a PKA_PLAN_HOST_ONLY plan the word of
 * paged_decode_run_noalloc's scratch on the current device -- else
 * *status_dev (device int32, caller-owned).  Does not synchronise.
 */
int pka_wait_timeout_probe(const pka_plan* plan, int32_t* status_dev, int64_t limit_ns,
                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKA_H */
