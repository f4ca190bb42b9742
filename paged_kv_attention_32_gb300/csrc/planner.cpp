// Host planner of the paged decode: reads the lengths on the host (the
// one-shot planner of batch_decode_with_paged_kv_cache reads seq_lens_kv on
// the host to derive exact plan bounds), cuts long key ranges into chunks so
// that enough CTAs exist to fill the GPU, and orders the work longest first.
//
// The chunking rule is this library's own design (the pages leave it open):
//   - request b visits pages [kv_lo / ps, ceil(n / ps)), kv_lo being the left
//     window edge of its first row when the plan is frozen, else 0;
//   - with T = split_waves * num_sms target CTAs, no request is split when
//     B * Hkv >= T; otherwise the chunk c is the smallest page count in
//     [min(c_min, max np), max np] with Hkv * sum_b ceil(np_b / c) <= T;
//   - when nothing is split that way, the requests past the first wave of
//     resident CTAs (S = 3 per SM for the mma kernel, 2 for the CUDA-core
//     one; longest-first prefix with at most S CTAs) start only as that wave
//     ends, so they are cut into k = S / R chunks (R = their CTAs) of
//     max(ceil(np / k), min(c_min, np)) pages when k > 1: one short round on
//     every SM instead of a long one on a few;
//   - and, for the mma kernel with one 16-row tile per request, a request
//     longer than 3/5 of a resident slot's average load (A = Hkv * sum np / S
//     pages) is cut into ceil(np / (3A/5)) chunks of at least min(c_min, np)
//     pages: its warps stream at a latency-bound rate, so long CTAs would
//     finish last (measured on GB300; requests of several tiles, and the
//     CUDA-core kernel, run best uncut);
//   - items run longest request first, then chunk, then KV head.
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cmath>
#include <numeric>

#include "host_common.h"
#include "plan.h"

namespace pka {

namespace {
constexpr int32_t kDefaultWaves = 2;
constexpr int32_t kDefaultMinChunkTokens = 256;
// rows per KV head from which the mma.sync kernel runs: measured on GB300
// (B = 64, kv_len U[512, 8192]), with the plan's cut of long single-tile
// requests it beats the CUDA-core kernel at 1, 2 and 4 rows per KV head, bf16
// and half alike (1.105 / 1.069 / 1.005 of the copy peak against 1.075 / 1.015
// / 0.95), so it runs by default; the CUDA-core kernel is kept for a threshold
// set higher
constexpr int32_t kDefaultMmaMinRows = 1;
constexpr int32_t kMaxCudaCoreRows = 8;   // rows one warp of the CUDA-core kernel holds
// query rows per KV head the tensor-core kernel takes: one CTA per 16-row
// tile of every item (4096 tiles); the pages put no bound on the group or on
// q_len_per_req, this only keeps the launch arithmetic in 32 bits
constexpr int32_t kMaxMmaRows = 65536;

// A positive integer from the environment variable `name`, else `fallback`.
int32_t env_int(const char* name, int32_t fallback) {
  const char* v = std::getenv(name);
  if (v == nullptr || *v == '\0') return fallback;
  char* end = nullptr;
  const long x = std::strtol(v, &end, 10);
  return (end != nullptr && *end == '\0' && x > 0 && x <= INT32_MAX) ? (int32_t)x : fallback;
}
}  // namespace

int build_decode_plan(pka_plan& p, const pka_decode_desc& d_in, const int32_t* seq,
                      const int32_t* indptr) {
  pka_decode_desc d = d_in;
  PKA_CHECK_ARG(d.batch_size >= 1, "batch_size must be >= 1 (got %d)", d.batch_size);
  PKA_CHECK_ARG(seq != nullptr, "seq_lens_kv_host is NULL");
  PKA_CHECK_ARG(d.num_qo_heads >= 1 && d.num_kv_heads >= 1, "head counts must be >= 1");
  PKA_CHECK_ARG(d.num_qo_heads % d.num_kv_heads == 0,
                "num_qo_heads (%d) must be a multiple of num_kv_heads (%d)", d.num_qo_heads,
                d.num_kv_heads);
  if (d.dtype != PKA_DTYPE_BF16 && d.dtype != PKA_DTYPE_F16)
    return fail(PKA_ERR_UNSUPPORTED, "q/K/V must be bf16 or f16 (dtype %d)", d.dtype);
  PKA_CHECK_ARG(d.out_dtype == PKA_DTYPE_BF16 || d.out_dtype == PKA_DTYPE_F16 ||
                    d.out_dtype == PKA_DTYPE_F32,
                "out_dtype must be bf16, f16 or f32 (got %d)", d.out_dtype);
  if (d.head_dim != 128)
    return fail(PKA_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", d.head_dim);
  if (d.page_size < 16 || d.page_size > 256 || d.page_size % 16 != 0)
    return fail(PKA_ERR_UNSUPPORTED, "page_size must be a multiple of 16 in [16, 256] (got %d)",
                d.page_size);
  PKA_CHECK_ARG(d.max_pages_per_seq >= 1, "max_pages_per_seq must be >= 1");
  PKA_CHECK_ARG(d.num_pages >= 1 && d.num_pages <= (int64_t)INT32_MAX,
                "num_pages must be in [1, 2^31-1]");
  PKA_CHECK_ARG(d.mask == PKA_MASK_DENSE || d.mask == PKA_MASK_CAUSAL, "unknown mask %d", d.mask);
  PKA_CHECK_ARG(d.window_left >= -1, "window_left must be -1 or >= 0");
  if (std::isnan(d.scale)) d.scale = 1.0f / std::sqrt((float)d.head_dim);
  PKA_CHECK_ARG(std::isfinite(d.scale), "scale must be finite");
  PKA_CHECK_ARG(std::isfinite(d.bmm2_scale), "bmm2_scale must be finite");
  // a field left 0 takes the environment's value (PKA_SPLIT_WAVES, PKA_MIN_CHUNK_TOKENS,
  // PKA_MMA_MIN_ROWS), else the default; the plan records what it used
  if (d.split_waves <= 0) d.split_waves = env_int("PKA_SPLIT_WAVES", kDefaultWaves);
  if (d.min_chunk_tokens <= 0)
    d.min_chunk_tokens = env_int("PKA_MIN_CHUNK_TOKENS", kDefaultMinChunkTokens);
  if (d.mma_min_rows <= 0) d.mma_min_rows = env_int("PKA_MMA_MIN_ROWS", kDefaultMmaMinRows);
  if (d.num_sms <= 0) {
    int dev = 0, sms = 0;
    PKA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
    PKA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                 "cudaDeviceGetAttribute(SM count)");
    d.num_sms = sms;
  }

  const int32_t B = d.batch_size, ps = d.page_size, Hkv = d.num_kv_heads, Hq = d.num_qo_heads;
  p.desc = d;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.D = d.head_dim;
  p.ps = ps;
  p.C = d.max_pages_per_seq;
  p.scale = d.scale;

  // ---- query rows per request (fixed or packed) ----
  std::vector<int32_t> qstart(B + 1), qlen(B);
  if (indptr == nullptr) {
    PKA_CHECK_ARG(d.q_len >= 1, "q_len must be >= 1 in fixed-query mode (got %d)", d.q_len);
    PKA_CHECK_ARG(d.max_q_len == 0 || d.max_q_len == d.q_len,
                  "fixed-query mode needs max_q_len == q_len (got %d vs %d)", d.max_q_len,
                  d.q_len);
    for (int32_t b = 0; b <= B; ++b) qstart[b] = b * d.q_len;
    for (int32_t b = 0; b < B; ++b) qlen[b] = d.q_len;
  } else {
    PKA_CHECK_ARG(indptr[0] == 0, "qo_indptr[0] must be 0 (got %d)", indptr[0]);
    int32_t cap = d.max_q_len;
    if (d.q_len > 1) {
      PKA_CHECK_ARG(cap == 0 || cap == d.q_len,
                    "q_len (%d) is an alias of max_q_len (%d) in packed mode and must agree",
                    d.q_len, cap);
      cap = d.q_len;
    }
    for (int32_t b = 0; b < B; ++b) {
      int64_t l = (int64_t)indptr[b + 1] - indptr[b];
      PKA_CHECK_ARG(l >= 1, "request %d has %lld query rows; packed rows must be >= 1", b,
                    (long long)l);
      PKA_CHECK_ARG(cap == 0 || l <= cap, "request %d has %lld query rows, above max_q_len %d",
                    b, (long long)l, cap);
      qstart[b] = indptr[b];
      qlen[b] = (int32_t)l;
    }
    qstart[B] = indptr[B];
  }
  int32_t max_q = *std::max_element(qlen.begin(), qlen.end());
  p.total_q = qstart[B];
  p.max_q_len = max_q;

  // ---- kernel choice ----
  const int64_t rows = (int64_t)p.G * max_q;
  if (rows > kMaxMmaRows)
    return fail(PKA_ERR_UNSUPPORTED,
                "(Hq/Hkv) * max_q_len = %lld query rows per KV head exceeds %d", (long long)rows,
                kMaxMmaRows);
  p.rows_per_cta = (int32_t)rows;
  p.kernel = (rows >= d.mma_min_rows || rows > kMaxCudaCoreRows) ? PKA_KERNEL_MMA
                                                                    : PKA_KERNEL_CUDA_CORE;

  // ---- visited pages per request ----
  const bool windowed = d.window_left >= 0 && d.freeze_seq_lens;
  std::vector<int64_t> npages(B);
  p.page_lo.assign(B, 0);
  p.page_hi.assign(B, 0);
  for (int32_t b = 0; b < B; ++b) {
    const int64_t n = seq[b];
    PKA_CHECK_ARG(n >= 1, "seq_lens_kv[%d] = %lld must be >= 1", b, (long long)n);
    PKA_CHECK_ARG(n >= qlen[b], "request %d: kv_len %lld < q_len %d (every request needs "
                  "kv_len >= q_len)", b, (long long)n, qlen[b]);
    PKA_CHECK_ARG(n <= (int64_t)p.C * ps, "request %d: kv_len %lld exceeds the table capacity "
                  "%d pages x %d", b, (long long)n, p.C, ps);
    const int64_t kv_lo = windowed ? std::max<int64_t>(0, n - qlen[b] - d.window_left) : 0;
    p.page_lo[b] = (int32_t)(kv_lo / ps);
    p.page_hi[b] = (int32_t)ceil_div(n, ps);
    npages[b] = p.page_hi[b] - p.page_lo[b];
  }

  // ---- chunk choice: count CTAs (the mma kernel runs one CTA per 16-row tile) ----
  std::vector<int64_t> tiles(B, 1);
  if (p.kernel == PKA_KERNEL_MMA)
    for (int32_t b = 0; b < B; ++b) tiles[b] = ceil_div((int64_t)p.G * qlen[b], 16);
  int64_t tiles_sum = 0;
  for (int32_t b = 0; b < B; ++b) tiles_sum += tiles[b];
  const int64_t max_np = *std::max_element(npages.begin(), npages.end());
  const int64_t target = (int64_t)d.split_waves * d.num_sms;
  int64_t chunk = max_np;
  if (tiles_sum * Hkv < target) {
    const int64_t c_min = ceil_div(d.min_chunk_tokens, ps);
    for (int64_t c = std::min(c_min, max_np); c <= max_np; ++c) {
      int64_t cnt = 0;
      for (int32_t b = 0; b < B; ++b) cnt += tiles[b] * ceil_div(npages[b], c);
      if (cnt * Hkv <= target) {
        chunk = c;
        break;
      }
    }
  }
  p.chunk_pages = (int32_t)chunk;

  // ---- longest request first; chunk length per request ----
  p.order.resize(B);
  std::iota(p.order.begin(), p.order.end(), 0);
  // longest first, ties in request order (a stable order without the stable
  // sort's buffer)
  std::sort(p.order.begin(), p.order.end(), [&](int32_t a, int32_t b) {
    return npages[a] > npages[b] || (npages[a] == npages[b] && a < b);
  });
  std::vector<int64_t> cb(B, chunk);
  if (tiles_sum * Hkv >= target) {
    const int64_t slots = (int64_t)(p.kernel == PKA_KERNEL_MMA ? 3 : 2) * d.num_sms;
    // the tail: order[first_tail ..], past the longest-first prefix that fits
    int64_t acc = 0, rest = 0;
    int32_t first_tail = B;
    for (int32_t i = 0; i < B; ++i) {
      const int32_t b = p.order[i];
      if (first_tail == B && acc + Hkv * tiles[b] <= slots) {
        acc += Hkv * tiles[b];
      } else {
        if (first_tail == B) first_tail = i;
        rest += Hkv * tiles[b];
      }
    }
    const int64_t k = rest ? slots / rest : 1;
    const int64_t c_min = ceil_div(d.min_chunk_tokens, ps);
    if (k > 1)
      for (int32_t i = first_tail; i < B; ++i) {
        const int32_t b = p.order[i];
        cb[b] = std::max(ceil_div(npages[b], k), std::min(c_min, npages[b]));
      }
    // tensor-core kernel, one 16-row tile per request: a request longer than
    // 3/5 of a resident slot's average load A = Hkv * sum np / S is cut into
    // ceil(np / (3A/5)) chunks (integer form: np * 5S > 3 * Hkv * sum np)
    if (p.kernel == PKA_KERNEL_MMA && p.rows_per_cta <= 16) {
      int64_t load = 0;
      for (int32_t b = 0; b < B; ++b) load += (int64_t)Hkv * npages[b];
      for (int32_t b = 0; b < B; ++b) {
        const int64_t num = npages[b] * 5 * slots, den = 3 * load;
        if (num > den) {
          const int64_t parts = ceil_div(num, den);
          cb[b] = std::min(cb[b], std::max(ceil_div(npages[b], parts), std::min(c_min, npages[b])));
        }
      }
    }
  }

  // ---- items ----
  std::vector<int32_t> nch(B);
  for (int32_t b = 0; b < B; ++b) nch[b] = (int32_t)ceil_div(npages[b], cb[b]);
  int64_t n_items = 0;
  for (int32_t b = 0; b < B; ++b) n_items += (int64_t)nch[b] * Hkv;
  PKA_CHECK_ARG(n_items <= (int64_t)INT32_MAX, "too many work items");
  for (int32_t b = 0; b < B; ++b)
    PKA_CHECK_ARG(nch[b] < 65536, "request %d needs %d chunks (limit 65535)", b, nch[b]);
  PKA_CHECK_ARG(Hkv < 65536, "num_kv_heads must be < 65536");
  p.items.resize((size_t)n_items);
  WorkItem* item = p.items.data();
  for (int32_t b : p.order) {
    const int64_t c = cb[b];
    const int32_t lo0 = p.page_lo[b], hi0 = p.page_hi[b], n = nch[b];
    for (int32_t ci = 0; ci < n; ++ci) {
      const int32_t lo = lo0 + (int32_t)(ci * c);
      const int32_t hi = (int32_t)std::min<int64_t>(lo0 + (ci + 1) * c, hi0);
      for (int32_t hk = 0; hk < Hkv; ++hk) *item++ = WorkItem{b, (ci << 16) | hk, lo, hi};
    }
  }

  // ---- split requests: partial rows, merge counters, workspace ----
  // The last chunk CTA of each (request, KV head, tile) merges that group's
  // partials; a counter per group tells it that it is the last.
  const int32_t tiles_per_item =
      p.kernel == PKA_KERNEL_MMA ? (int32_t)ceil_div(p.rows_per_cta, 16) : 1;
  p.reqs.assign(B, ReqInfo{});
  int64_t prow = 0, counters = 0;
  int32_t n_split = 0;
  for (int32_t b = 0; b < B; ++b) {
    ReqInfo& r = p.reqs[b];
    r.q_start = qstart[b];
    r.q_len = qlen[b];
    r.kv_len = seq[b];
    r.n_chunks = nch[b];
    r.cnt_base = -1;
    if (nch[b] > 1) {
      r.part_base = (int32_t)prow;
      prow += (int64_t)nch[b] * qlen[b] * Hq;
      r.cnt_base = (int32_t)counters;
      counters += (int64_t)Hkv * tiles_per_item;
      ++n_split;
    } else {
      r.part_base = -1;
    }
    PKA_CHECK_ARG(prow <= (int64_t)INT32_MAX && counters <= (int64_t)INT32_MAX,
                  "too many partial rows");
  }
  p.num_merge_counters = (int32_t)counters;
  p.num_split = n_split;
  p.partial_rows = (int32_t)prow;
  const int64_t o_bytes = ceil_div(prow * p.D * 4, 256) * 256;
  p.ws_lse_offset = o_bytes;
  p.workspace_bytes = prow ? o_bytes + prow * 4 : 0;
  return PKA_OK;
}

}  // namespace pka
