// kernels_mx.cu -- MXFP4 quantisation of a teacher head (DeepSeek-V4 book
// ch. 19, "1. FP4 in OPD": the inference-only teacher forwards run on 4-bit
// MXFP4 weights).
//
// OCP Microscaling FP4, per 32 consecutive elements of a row:
//   scale code  s = floor(log2 max|x|) - 2 + 127, clamped to [0, 254]
//               (2 is the exponent of E2M1's largest value, 6); 0 for an
//               all-zero block
//   element     the E2M1 value nearest to x / 2^(s - 127), ties to the even
//               code, saturated at 6; a zero magnitude is stored as +0.
// E2M1 magnitudes by code: 0, 0.5, 1, 1.5, 2, 3, 4, 6.  The grid spacing is
// 0.5 below 2, 1 in [2, 4) and 2 from 4, so rounding to nearest-even in units
// of the spacing of the value's octave is the E2M1 rounding.
// Output: the blocked layout of MxOperand (rows past V zero).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "launch.h"

namespace flp {

namespace {
__device__ __forceinline__ float load_elem(const void *W, bool bf16, int64_t i) {
  if (bf16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(W)[i]);
  return __half2float(static_cast<const __half *>(W)[i]);
}

// E2M1 code (0..7) of a magnitude a >= 0 given in units of the block scale.
__device__ __forceinline__ uint32_t e2m1_code(float a) {
  const float spacing = a < 2.f ? 0.5f : (a < 4.f ? 1.f : 2.f);
  const float q = fminf(rintf(a / spacing) * spacing, 6.f);
  if (q < 2.f) return static_cast<uint32_t>(q * 2.f);   // 0, 0.5, 1, 1.5 -> 0..3
  if (q < 4.f) return static_cast<uint32_t>(q) + 2u;    // 2, 3 -> 4, 5
  return q == 4.f ? 6u : 7u;                            // 4, 6
}
}  // namespace

// One thread per (row, 32-element block).
__global__ void mxfp4_quantize_kernel(const void *__restrict__ W, bool bf16, int64_t V,
                                      int64_t H, int64_t ld_w, int64_t v_pad,
                                      uint8_t *__restrict__ packed, uint8_t *__restrict__ scales) {
  const int64_t nblk = H / 32;
  const int64_t total = v_pad * nblk;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t v = t / nblk;
    const int64_t j = t - v * nblk;          // 32-element block of the row
    const int64_t kb = j >> 1;               // 64-wide column block
    const int64_t blk = kb * v_pad + v;
    uint4 out = make_uint4(0, 0, 0, 0);
    uint32_t code = 0;
    if (v < V) {
      float x[32];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = load_elem(W, bf16, v * ld_w + j * 32 + i);
        amax = fmaxf(amax, fabsf(x[i]));
      }
      const int fe = static_cast<int>((__float_as_uint(amax) >> 23) & 255u);  // biased exponent
      code = amax > 0.f ? static_cast<uint32_t>(max(fe - 2, 0)) : 0u;
      code = min(code, 254u);
      // 1 / 2^(code - 127) = 2^(127 - code): a normal float for code <= 253
      const float inv = __uint_as_float((254u - min(code, 253u)) << 23);
      uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        uint32_t c = e2m1_code(fabsf(x[i]) * inv);
        if (c != 0u && x[i] < 0.f) c |= 8u;
        w[i >> 3] |= c << (4 * (i & 7));
      }
      out = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4 *>(packed + blk * 32 + (j & 1) * 16) = out;
    scales[blk * 2 + (j & 1)] = static_cast<uint8_t>(code);
  }
}

// The same quantisation into the head layout of the block-scaled KL: codes
// [V, H/2] row-major (byte b of a row: elements 2b, low nibble, and 2b + 1),
// and for each 224-row vocabulary tile vt and 128-wide k-chunk kc two
// 512-byte scale atoms, rows vt * 224 + 128 a .. + 127 for atom a, row r's
// scale of step j at byte (r % 32) * 16 + (r / 32) * 4 + j.  One thread per
// (row, 32-element block) over the rows of whole tiles; rows past V get
// scale 0 (atom bytes of rows past a tile's 224 are left to the caller).
__global__ void mx_head_quantize_kernel(const void *__restrict__ W, bool bf16, int64_t V,
                                        int64_t H, int64_t ld_w, int64_t rows_out,
                                        uint8_t *__restrict__ codes, uint8_t *__restrict__ atoms) {
  const int64_t nblk = H / 32;
  const int64_t kc_n = H / 128;
  const int64_t total = rows_out * nblk;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t v = t / nblk;
    const int64_t j = t - v * nblk;
    uint32_t code = 0;
    if (v < V) {
      float x[32];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = load_elem(W, bf16, v * ld_w + j * 32 + i);
        amax = fmaxf(amax, fabsf(x[i]));
      }
      const int fe = static_cast<int>((__float_as_uint(amax) >> 23) & 255u);
      code = amax > 0.f ? static_cast<uint32_t>(max(fe - 2, 0)) : 0u;
      code = min(code, 254u);
      const float inv = __uint_as_float((254u - min(code, 253u)) << 23);
      uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        uint32_t c = e2m1_code(fabsf(x[i]) * inv);
        if (c != 0u && x[i] < 0.f) c |= 8u;
        w[i >> 3] |= c << (4 * (i & 7));
      }
      *reinterpret_cast<uint4 *>(codes + v * (H / 2) + j * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const int64_t vt = v / kMxBN, i = v - vt * kMxBN, a = i >> 7, r = i & 127;
    atoms[((vt * kc_n + (j >> 2)) * 2 + a) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3)] =
        static_cast<uint8_t>(code);
  }
}

cudaError_t launch_mx_head_quantize(const void *W, bool bf16, int64_t V, int64_t H, int64_t ld_w,
                                    uint8_t *codes, uint8_t *atoms, int num_sms,
                                    cudaStream_t stream) {
  const int64_t rows_out = (V + kMxBN - 1) / kMxBN * kMxBN;
  const int64_t total = rows_out * (H / 32);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  mx_head_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      W, bf16, V, H, ld_w, rows_out, codes, atoms);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_quantize(const void *W, bool bf16, int64_t V, int64_t H, int64_t ld_w,
                                  int64_t v_pad, uint8_t *packed, uint8_t *scales, int num_sms,
                                  cudaStream_t stream) {
  const int64_t total = v_pad * (H / 32);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  mxfp4_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      W, bf16, V, H, ld_w, v_pad, packed, scales);
  return cudaGetLastError();
}

}  // namespace flp
