// TMA tensor-map encoding (host).  The driver's cuTensorMapEncodeTiled is a
// pure host-side encoder: it touches no device state, so it may run while a
// stream is being captured.
#pragma once

#include <cstdint>

#include <cuda.h>

namespace pka {

// Encodes a bf16 tiled tensor map with 128-byte swizzle.
//   rank        2..5
//   dims        extent of each dimension, innermost first (elements)
//   strides     byte stride of dimensions 1..rank-1 (multiples of 16)
//   box         box extent per dimension; box[0] * 2 bytes must be <= 128
// Returns PKA_OK or an error code with the message recorded.
int encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box);

// Tensor map over an HND page pool (page, kv_head, slot, d), D = 128, as the
// 5-D view (d_lo, slot, d_hi, head, page): one box is a 16-token unit of one
// (page, head) block, 4 KB, stored as its two 64-column halves.
int encode_kv_pool_map(CUtensorMap* map, const void* pool, int64_t num_pages, int32_t num_heads,
                       int32_t page_size, int32_t head_dim, int64_t stride_page,
                       int64_t stride_head);

}  // namespace pka
