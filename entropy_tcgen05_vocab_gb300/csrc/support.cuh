// support.cuh -- reading a row's sampling support inside an epilogue.
//
// The support (the per-row vocabulary mask of the pages' sampling_mask) is a
// bitmask of uint32 words per h row: token v is in the row's support iff bit
// v % 32 of word v / 32 is set.  An epilogue warp folds 32 columns at a time,
// so each chunk needs exactly one word.  The words of a warp's columns in a
// tile are loaded together at the end of the previous tile, so their latency
// (an HBM round trip: the words are read once) hides behind that tile's
// MMAs instead of stalling each chunk.
#pragma once

#include <cstdint>

namespace flp {

struct SupportRow {
  static constexpr int kWords = 8;  // chunks a warp folds per tile, held ahead
  const uint32_t *row;  // this row's words, or null (no token is in the support)
  int V;
  int pre_col;          // first column of the words held in w; -1 if none
  uint32_t w[kWords];

  __device__ __forceinline__ void reset(const uint32_t *r, int vocab) {
    row = r;
    V = vocab;
    pre_col = -1;
  }
  // Word of the 32-column chunk starting at column cb (0 past the vocabulary).
  __device__ __forceinline__ uint32_t load(int cb) const {
    return (row != nullptr && cb < V) ? __ldg(row + (cb >> 5)) : 0u;
  }
  // Loads the words of the kWords chunks from column col on.
  __device__ __forceinline__ void prefetch(int col) {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = load(col + 32 * i);
    pre_col = col;
  }
  // Call once at the start of a tile whose first column is col0.
  __device__ __forceinline__ void start(int col0) {
    if (col0 != pre_col) prefetch(col0);
  }
  // Word of chunk c of the tile started at col0; chunks are taken in order
  // c = 0, 1, ... (the held words shift down, so no register is indexed
  // dynamically).
  __device__ __forceinline__ uint32_t next(int col0, int c) {
    if (c >= kWords) return load(col0 + 32 * c);
    const uint32_t x = w[0];
#pragma unroll
    for (int i = 0; i + 1 < kWords; ++i) w[i] = w[i + 1];
    return x;
  }
  // Bits of the chunk at cb that are inside the vocabulary.
  __device__ __forceinline__ uint32_t clip(uint32_t word, int cb) const {
    return cb + 32 <= V ? word : (word & ((1u << (V - cb)) - 1u));
  }
};

}  // namespace flp
