#include "tmap.h"

#include <mutex>

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "host_common.h"

namespace pka {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                  cudaEnableDefault, &q);
  if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

int encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) {
    if (g_encode_err != cudaSuccess) return cuda_fail(g_encode_err, "cuTensorMapEncodeTiled lookup");
    return fail(PKA_ERR_CUDA, "cuTensorMapEncodeTiled not found in the driver");
  }
  PKA_CHECK_ARG(((uintptr_t)base & 15) == 0, "tensor base %p is not 16-byte aligned", base);
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) {
    PKA_CHECK_ARG(strides[i] % 16 == 0, "tensor stride %llu bytes is not a multiple of 16",
                  (unsigned long long)strides[i]);
    gstride[i] = strides[i];
  }
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                        const_cast<void*>(base), gdim, gstride, bdim, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PKA_OK;
}

namespace {
int encode_pool_map_uncached(CUtensorMap* map, const void* pool, int64_t num_pages,
                             int32_t num_heads, int32_t page_size, int32_t head_dim,
                             int64_t stride_page, int64_t stride_head) {
  // The 128 columns are split as (d_lo 0..63, d_hi 0..1) and d_hi is placed
  // after the slot dimension: (d_lo, slot, d_hi, head, page).  A box of
  // {64, 16, 2, 1, 1} then lands in shared memory as the two 64-column halves
  // of 16 token rows one after the other -- a whole 16-token unit in one copy.
  const uint64_t dims[5] = {64, (uint64_t)page_size, 2, (uint64_t)num_heads, (uint64_t)num_pages};
  const uint64_t strides[4] = {(uint64_t)head_dim * 2, 128, (uint64_t)stride_head * 2,
                               (uint64_t)stride_page * 2};
  const uint32_t box[5] = {64, 16, 2, 1, 1};
  return encode_bf16_map(map, pool, 5, dims, strides, box);
}

// A pool map is a pure function of the pool's address, shape and strides, so
// the maps of the last few pools a thread ran on are kept (a serving loop runs
// the same K and V pools every step) and reused without the driver call.
struct PoolMapKey {
  const void* pool;
  int64_t num_pages, stride_page, stride_head;
  int32_t num_heads, page_size;
  bool operator==(const PoolMapKey& o) const {
    return pool == o.pool && num_pages == o.num_pages && stride_page == o.stride_page &&
           stride_head == o.stride_head && num_heads == o.num_heads && page_size == o.page_size;
  }
};
constexpr int kPoolMapCache = 4;
struct PoolMapCache {
  PoolMapKey key[kPoolMapCache] = {};
  CUtensorMap map[kPoolMapCache];
  bool used[kPoolMapCache] = {};
  int next = 0;
};
thread_local PoolMapCache t_pool_maps;
}  // namespace

int encode_kv_pool_map(CUtensorMap* map, const void* pool, int64_t num_pages, int32_t num_heads,
                       int32_t page_size, int32_t head_dim, int64_t stride_page,
                       int64_t stride_head) {
  PKA_CHECK_ARG(stride_head > 0 && stride_page > 0, "K/V strides must be positive");
  PKA_CHECK_ARG(head_dim == 128, "the K/V pool map takes head_dim 128 (got %d)", head_dim);
  const PoolMapKey key{pool, num_pages, stride_page, stride_head, num_heads, page_size};
  PoolMapCache& c = t_pool_maps;
  for (int i = 0; i < kPoolMapCache; ++i)
    if (c.used[i] && c.key[i] == key) {
      *map = c.map[i];
      return PKA_OK;
    }
  const int rc = encode_pool_map_uncached(map, pool, num_pages, num_heads, page_size, head_dim,
                                          stride_page, stride_head);
  if (rc == PKA_OK) {
    c.key[c.next] = key;
    c.map[c.next] = *map;
    c.used[c.next] = true;
    c.next = (c.next + 1) % kPoolMapCache;
  }
  return rc;
}

}  // namespace pka
