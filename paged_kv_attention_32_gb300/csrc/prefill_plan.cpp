// Host tile schedule of the ragged causal prefill (batch_prefill with packed
// qo_indptr / kv_indptr).  One tile = 128 query rows of one request for one
// query head, with the run of 64-key tiles its rows can see
// (causal diagonal, optional left window); tiles are ordered heaviest first
// (most KV tiles to visit), so that the hardware block scheduler hands the
// long causal rows out before the short ones (longest-processing-time order).
#include <algorithm>
#include <climits>
#include <cmath>
#include <numeric>

#include "host_common.h"
#include "prefill.h"

namespace pka {

namespace {
constexpr int kTileQ = 128;     // query rows per CTA
constexpr int kTileK = 64;      // keys per K/V tile
}  // namespace

int build_prefill_plan(pka_prefill_plan& p, const pka_prefill_desc& d_in, const int32_t* qo,
                       const int32_t* kv, const int32_t* win_lo, const int32_t* win_hi) {
  pka_prefill_desc d = d_in;
  PKA_CHECK_ARG(qo != nullptr && kv != nullptr, "qo_indptr_host and kv_indptr_host are required");
  PKA_CHECK_ARG(d.batch_size >= 1, "batch_size must be >= 1");
  PKA_CHECK_ARG(d.num_qo_heads >= 1 && d.num_kv_heads >= 1, "head counts must be >= 1");
  PKA_CHECK_ARG(d.num_qo_heads % d.num_kv_heads == 0,
                "num_qo_heads (%d) must be a multiple of num_kv_heads (%d)", d.num_qo_heads,
                d.num_kv_heads);
  if (d.dtype != PKA_DTYPE_BF16 && d.dtype != PKA_DTYPE_F16)
    return fail(PKA_ERR_UNSUPPORTED, "q/K/V must be bf16 or f16 (dtype %d)", d.dtype);
  PKA_CHECK_ARG(d.out_dtype == PKA_DTYPE_BF16 || d.out_dtype == PKA_DTYPE_F16 ||
                    d.out_dtype == PKA_DTYPE_F32,
                "out_dtype must be bf16, f16 or f32 (got %d)", d.out_dtype);
  if (d.head_dim != 128 && d.head_dim != 256)
    return fail(PKA_ERR_UNSUPPORTED, "prefill head_dim must be 128 or 256 (got %d)", d.head_dim);
  PKA_CHECK_ARG(d.mask == PKA_MASK_DENSE || d.mask == PKA_MASK_CAUSAL ||
                    d.mask == PKA_MASK_VARIABLE_WINDOW,
                "unknown mask %d", d.mask);
  const bool varwin = d.mask == PKA_MASK_VARIABLE_WINDOW;
  PKA_CHECK_ARG(varwin == (win_lo != nullptr && win_hi != nullptr),
                varwin ? "variable_window needs both bound arrays (fixed-shape planner)"
                       : "window bounds are given only with mask variable_window");
  PKA_CHECK_ARG(d.window_left >= -1, "window_left must be -1 or >= 0 (got %d)", d.window_left);
  if (std::isnan(d.sm_scale)) d.sm_scale = 1.0f / std::sqrt((float)d.head_dim);
  PKA_CHECK_ARG(std::isfinite(d.sm_scale) && std::isfinite(d.output_scale),
                "sm_scale and output_scale must be finite");
  if (d.sm_scale < 0.f)
    return fail(PKA_ERR_UNSUPPORTED, "prefill sm_scale must be >= 0 (got %g)", (double)d.sm_scale);
  PKA_CHECK_ARG(qo[0] == 0 && kv[0] == 0, "indptr arrays must start at 0");
  const int32_t B = d.batch_size;
  for (int32_t b = 0; b < B; ++b)
    PKA_CHECK_ARG(qo[b + 1] >= qo[b] && kv[b + 1] >= kv[b],
                  "indptr arrays must be non-decreasing (request %d)", b);
  p.desc = d;
  p.B = B;
  p.Hq = d.num_qo_heads;
  p.Hkv = d.num_kv_heads;
  p.G = p.Hq / p.Hkv;
  p.D = d.head_dim;
  p.scale = d.sm_scale;
  p.qo.assign(qo, qo + B + 1);
  p.kv.assign(kv, kv + B + 1);
  p.win_lo.clear();
  p.win_hi.clear();
  if (varwin) {
    p.win_lo.assign(win_lo, win_lo + qo[B]);
    p.win_hi.assign(win_hi, win_hi + qo[B]);
  }
  p.tiles.clear();
  p.row_map.clear();
  if (varwin) {
    // Tiles of rows with similar windows compute fewer invisible scores: each
    // request's rows are ordered by their last key, cut into bands of a few
    // tiles, and ordered by their first key inside a band.  The band size that
    // needs the fewest key tiles is taken (it grows with the spread of the
    // windows), and the order only where it needs fewer than the rows' own.
    for (int32_t b = 0; b < B; ++b) {
      const int64_t lk = (int64_t)kv[b + 1] - kv[b];
      for (int64_t r = qo[b]; r < qo[b + 1]; ++r)
        PKA_CHECK_ARG(win_lo[r] >= 0 && win_lo[r] <= win_hi[r] && win_hi[r] < lk,
                      "request %d row %lld: window bounds [%d, %d] outside 0 <= start <= end < "
                      "%lld", b, (long long)(r - qo[b]), win_lo[r], win_hi[r], (long long)lk);
    }
    std::vector<int32_t> order, best;
    bool any = false;
    p.row_map.resize(qo[B]);
    for (int32_t b = 0; b < B; ++b) {
      const int64_t lq = (int64_t)qo[b + 1] - qo[b];
      const int32_t* s0 = win_lo + qo[b];
      const int32_t* e0 = win_hi + qo[b];
      auto key_tiles = [&](auto row_at) {
        int64_t n = 0;
        for (int64_t m = 0; m * kTileQ < lq; ++m) {
          int64_t lo = INT64_MAX, hi = 0;
          for (int64_t r = m * kTileQ; r < std::min<int64_t>(lq, (m + 1) * kTileQ); ++r) {
            const int32_t i = row_at(r);
            lo = std::min<int64_t>(lo, s0[i]);
            hi = std::max<int64_t>(hi, (int64_t)e0[i] + 1);
          }
          n += ceil_div(hi, kTileK) - lo / kTileK;
        }
        return n;
      };
      int64_t best_n = key_tiles([&](int64_t r) { return (int32_t)r; });
      best.clear();
      for (int band : {2, 3, 4, 6, 8, 16}) {
        order.resize(lq);
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t x, int32_t y) { return e0[x] < e0[y]; });
        for (int64_t r0 = 0; r0 < lq; r0 += (int64_t)band * kTileQ)
          std::stable_sort(order.begin() + r0,
                           order.begin() + std::min<int64_t>(lq, r0 + (int64_t)band * kTileQ),
                           [&](int32_t x, int32_t y) { return s0[x] < s0[y]; });
        const int64_t n = key_tiles([&](int64_t r) { return order[r]; });
        if (n < best_n) {
          best_n = n;
          best = order;
        }
      }
      for (int64_t r = 0; r < lq; ++r) p.row_map[qo[b] + r] = best.empty() ? (int32_t)r : best[r];
      any = any || !best.empty();
    }
    if (!any) p.row_map.clear();
  }
  for (int32_t b = 0; b < B; ++b) {
    const int64_t lq = (int64_t)qo[b + 1] - qo[b], lk = (int64_t)kv[b + 1] - kv[b];
    PKA_CHECK_ARG(lq >= 0 && lk >= 0, "indptr arrays must be non-decreasing (request %d)", b);
    if (d.mask == PKA_MASK_CAUSAL)
      PKA_CHECK_ARG(lk >= lq, "request %d: causal prefill needs kv_len >= q_len", b);
    PKA_CHECK_ARG(lq == 0 || lk > 0, "request %d has queries but no keys", b);
    const int64_t n_qt = ceil_div(lq, kTileQ);
    for (int64_t m = 0; m < n_qt; ++m) {
      // keys the tile's rows see: up to the last row's bottom-right causal
      // diagonal, from the first row's window edge (plain sliding window)
      const int64_t first_row = m * kTileQ;
      const int64_t last_row = std::min<int64_t>(lq, (m + 1) * kTileQ) - 1;
      int64_t hi = d.mask == PKA_MASK_CAUSAL ? lk - lq + last_row + 1 : lk;
      int64_t lo =
          d.window_left >= 0 ? std::max<int64_t>(0, lk - lq + first_row - d.window_left) : 0;
      if (varwin) {   // the union of the tile's rows' bounds
        lo = lk;
        hi = 0;
        for (int64_t pos = first_row; pos <= last_row; ++pos) {
          const int64_t r = p.row_map.empty() ? pos : p.row_map[qo[b] + pos];
          const int32_t s = win_lo[qo[b] + r], e = win_hi[qo[b] + r];
          lo = std::min<int64_t>(lo, s);
          hi = std::max<int64_t>(hi, (int64_t)e + 1);
        }
      }
      const int32_t kv0 = (int32_t)(lo / kTileK);
      const int32_t n_kv = (int32_t)(ceil_div(hi, kTileK) - kv0);
      PKA_CHECK_ARG(n_kv >= 1, "request %d: a query tile with no key tile", b);
      for (int32_t h = 0; h < p.Hq; ++h)
        p.tiles.push_back(PrefillTile{h, (int32_t)m, n_kv, kv0, qo[b], (int32_t)lq, kv[b],
                                      (int32_t)lk});
    }
  }
  std::stable_sort(p.tiles.begin(), p.tiles.end(),
                   [](const PrefillTile& a, const PrefillTile& b) { return a.n_kv > b.n_kv; });
  p.total_q = qo[B];
  p.total_kv = kv[B];
  PKA_CHECK_ARG(p.tiles.size() < (size_t)INT32_MAX, "too many prefill tiles");
  return PKA_OK;
}

}  // namespace pka
