// Ragged causal prefill: plan object, tile schedule and kernel launcher.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "pka.h"

namespace pka {

// One unit of prefill work: a 128-row query tile of one request for one
// query head, with the request's offsets (32 bytes, two aligned loads).
struct alignas(16) PrefillTile {
  int32_t head;     // query head
  int32_t q_tile;   // 128-row tile index inside the request
  int32_t n_kv;     // KV tiles (64 keys) the tile visits
  int32_t kv0;      // first of them (past 0 only with a window)
  int32_t q0;       // the request's first packed query row (qo_indptr[b])
  int32_t lq;       // its query rows
  int32_t k0;       // its first packed key row (kv_indptr[b])
  int32_t lk;       // its keys
};

struct PrefillArgs {
  const void* q;
  int64_t q_stride_tok;
  int64_t q_stride_head;
  void* out;
  float* lse;
  const PrefillTile* tiles;
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  int32_t* status;
  int32_t num_tiles;
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t causal;
  int32_t window_left;   // -1: no window
  const int32_t* window_lo;   // variable_window: first key of each query row, else nullptr
  const int32_t* window_hi;   // variable_window: last key (inclusive) of each query row
  const int32_t* row_map;     // nullptr, or per packed position the request-local query row
                              // placed there (tiles then hold rows of similar windows)
  float scale_log2;
  float output_scale;
  int32_t out_dtype;       // PKA_DTYPE_BF16 / F16 / F32
};

}  // namespace pka

struct pka_prefill_plan {
  pka_prefill_desc desc;
  int32_t B = 0, Hq = 0, Hkv = 0, G = 0, D = 0;
  int32_t total_q = 0, total_kv = 0;
  float scale = 0.f;
  std::vector<int32_t> qo, kv;
  std::vector<int32_t> win_lo, win_hi;   // variable_window bounds per query row (host)
  std::vector<int32_t> row_map;          // empty, or the query row order inside the tiles
  std::vector<pka::PrefillTile> tiles;
  void* dev_buf = nullptr;
  const pka::PrefillTile* d_tiles = nullptr;
  const int32_t* d_qo = nullptr;
  const int32_t* d_kv = nullptr;
  const int32_t* d_win_lo = nullptr;
  const int32_t* d_win_hi = nullptr;
  const int32_t* d_row_map = nullptr;
  int32_t* d_status = nullptr;
  int device = -1;
};

namespace pka {

// Builds the host tile schedule (heaviest tiles first).  win_lo / win_hi:
// per-query-row inclusive key bounds of mask PKA_MASK_VARIABLE_WINDOW (one
// entry per packed query row), nullptr with the other masks.
int build_prefill_plan(pka_prefill_plan& plan, const pka_prefill_desc& desc, const int32_t* qo,
                       const int32_t* kv, const int32_t* win_lo = nullptr,
                       const int32_t* win_hi = nullptr);

// Launches the prefill kernel (one query head and 128 rows per CTA, 64-key
// tiles; head_dim 128 or 256) over the plan's tiles.
int launch_prefill_1h(const pka_prefill_plan& plan, const PrefillArgs& args,
                      const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      cudaStream_t stream);

}  // namespace pka
