// pa_index.cuh - the block-table lookup shared by every kernel and the gather hook.
#pragma once

#include <cstdint>

namespace pa {

// Physical page holding cache position `pos` of sequence b
// (block_table row b, logical block pos / page_size).
__device__ __forceinline__ int page_of(const int32_t* block_table, int max_blocks, int b, int pos,
                                       int page_size) {
  return block_table[(int64_t)b * max_blocks + pos / page_size];
}

}  // namespace pa
