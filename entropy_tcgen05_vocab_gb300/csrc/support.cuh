// support.cuh -- reading a row's sampling support inside an epilogue.
//
// The support (the per-row vocabulary mask of the pages' sampling_mask) is a
// bitmask of uint32 words per h row: token v is in the row's support iff bit
// v % 32 of word v / 32 is set.  An epilogue warp folds 32 columns at a time,
// so each chunk needs exactly one word.  SupportRow loads that word one chunk
// ahead, and at the end of a tile the first word of the warp's next tile, so
// the load latency hides behind the MMAs of that tile.
#pragma once

#include <cstdint>

namespace flp {

struct SupportRow {
  const uint32_t *row;  // this row's words, or null (no token is in the support)
  int V;
  int pre_col;          // column whose word `pre` holds; -1 if none
  uint32_t pre;

  __device__ __forceinline__ void reset(const uint32_t *r, int vocab) {
    row = r;
    V = vocab;
    pre_col = -1;
    pre = 0u;
  }
  // Word of the 32-column chunk starting at column cb (0 past the vocabulary).
  __device__ __forceinline__ uint32_t load(int cb) const {
    return (row != nullptr && cb < V) ? __ldg(row + (cb >> 5)) : 0u;
  }
  // Word of a tile's first chunk: the prefetched one if it is that chunk.
  __device__ __forceinline__ uint32_t first(int col0) const {
    return col0 == pre_col ? pre : load(col0);
  }
  __device__ __forceinline__ void prefetch(int col) {
    pre = load(col);
    pre_col = col;
  }
  // Bits of the chunk at cb that are inside the vocabulary.
  __device__ __forceinline__ uint32_t clip(uint32_t w, int cb) const {
    return cb + 32 <= V ? w : (w & ((1u << (V - cb)) - 1u));
  }
};

}  // namespace flp
