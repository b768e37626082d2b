// kernels_support.cu -- packing a sampling-support mask into bit words.
//
// The pages' sampling_mask is a per-row mask over the vocabulary (one entry
// per token).  The scoring kernels read it as 32 tokens per uint32 word:
// bit v % 32 of word v / 32 of row r is set iff mask[r, v] != 0.  One warp
// builds one word per step: lane j reads byte 32w + j of the row (a 32-byte
// coalesced read) and the warp's ballot is the word.
#include <cuda_runtime.h>

#include "launch.h"

namespace flp {

__global__ void pack_support_kernel(const uint8_t *__restrict__ mask, int64_t T, int64_t V,
                                    int64_t ld_mask, uint32_t *__restrict__ support,
                                    int64_t ld_support) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = T * ld_support;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < total;
       i += warps) {
    const int64_t r = i / ld_support;
    const int64_t w = i - r * ld_support;
    const int64_t v = w * 32 + lane;
    const bool on = v < V && mask[r * ld_mask + v] != 0;
    const uint32_t word = __ballot_sync(0xffffffffu, on);
    if (lane == 0) support[i] = word;
  }
}

cudaError_t launch_pack_support(const uint8_t *mask, int64_t T, int64_t V, int64_t ld_mask,
                                uint32_t *support, int64_t ld_support, int num_sms,
                                cudaStream_t stream) {
  const int64_t words = T * ld_support;
  if (words == 0) return cudaSuccess;
  int64_t blocks = (words + 7) / 8;  // 8 warps per block
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  pack_support_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(mask, T, V, ld_mask,
                                                                        support, ld_support);
  return cudaGetLastError();
}

}  // namespace flp
