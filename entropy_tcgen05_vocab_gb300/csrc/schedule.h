// schedule.h -- the work decomposition shared by the host planner and the
// scoring kernels (compiled by nvcc for both sides).
#pragma once

#ifndef __CUDACC__
#error "schedule.h is compiled by nvcc only"
#endif

namespace flp {

// Indices of the device status words at the start of the workspace.
constexpr int kStatBadTarget = 0;
constexpr int kStatBadRow = 1;
constexpr int kStatTimeout = 2;
constexpr int kStatEmptySupport = 3;

// MXFP4 operand in the blocked layout: for column block kb (64 wide) and row
// v < v_pad, 32 bytes of E2M1 codes at packed + (kb * v_pad + v) * 32 (byte b:
// element 2b in the low nibble, 2b + 1 in the high one) and two E8M0 scale
// codes at scales + (kb * v_pad + v) * 2 (elements 0..31, 32..63).
struct MxOperand {
  const unsigned char *packed;
  const unsigned char *scales;
  long long v_pad;
};

// Work item = (row tile, vocabulary split).  Items are ordered band by band:
// within a band of `band` row tiles, all items of split 0 (row tiles
// fastest), then split 1, ...  The last band may hold fewer row tiles.
struct Schedule {
  int n;                // scored rows
  int V;                // vocabulary size
  int row_tiles;        // ceil(n / 128)
  int vocab_tiles;      // ceil(V / BN)
  int splits;           // vocabulary splits
  int tiles_per_split;  // vocabulary tiles per split (the last split may be shorter)
  int band;             // row tiles per band
  int items;            // row_tiles * splits
  int k_blocks;         // ceil(H / 64)
  unsigned long long wait_ns;  // limit of the kernels' barrier waits (0: the default, 4 s)

  __host__ __device__ __forceinline__ void item(int L, int &mt, int &s, int &vt0,
                                                int &vt1) const {
    const int per_band = band * splits;
    const int b = L / per_band;
    const int rem = L - b * per_band;
    const int left = row_tiles - b * band;
    const int rows_in_band = band < left ? band : left;
    s = rem / rows_in_band;
    mt = b * band + (rem - s * rows_in_band);
    vt0 = s * tiles_per_split;
    vt1 = vt0 + tiles_per_split < vocab_tiles ? vt0 + tiles_per_split : vocab_tiles;
  }
};

}  // namespace flp
