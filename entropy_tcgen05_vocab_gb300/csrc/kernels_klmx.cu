// kernels_klmx.cu -- KL(teacher || student) with the teacher forward on the
// block-scaled tensor cores (DeepSeek-V4 book ch. 19, "1. FP4 in OPD": the
// inference-only teacher runs in native low precision; "TileLang KL kernel":
// the exact full-vocabulary KL with neither logit tensor in memory).
//
// A call quantises the teacher's hidden rows to MXFP8 (mxfp8_quantize_kernel,
// gathering the scored rows on the way), then runs mx_kl_pipeline_kernel:
// student logits from bf16/fp16 MMAs, teacher logits from block-scaled
// E4M3 x E2M1 MMAs against the MXFP4 head, both folded by the KL epilogue.
//
// OCP Microscaling MXFP8 with E4M3 elements, per 32 consecutive elements of
// a row:
//   scale code  s = floor(log2 max|x|) - 8 + 127, clamped to [0, 254] (8 is
//               the exponent of E4M3's largest finite value, 448); 0 for an
//               all-zero block
//   element     the E4M3 value nearest to x / 2^(s - 127), ties to the even
//               code, magnitudes above 448 saturated to 448; zero as +0.
// x / 2^(s - 127) is an exact power-of-two scaling in FP32 (results below
// FP32's normal range are far below E4M3's smallest step and round to 0 in
// either case), and the conversion to E4M3 is the hardware's
// round-to-nearest-even conversion with saturation to the largest finite
// value.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kl_epilogue.cuh"
#include "launch.h"
#include "launch_util.cuh"
#include "mx_pipeline.cuh"

namespace flp {

namespace {

// Two FP32 values -> two E4M3 codes (RNE, saturating), `hi` in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Clears the sign of every byte whose magnitude bits are zero (-0 -> +0).
__device__ __forceinline__ uint32_t plus_zero4(uint32_t w) {
  uint32_t out = w;
#pragma unroll
  for (int b = 0; b < 4; ++b)
    if (((w >> (8 * b)) & 0x7Fu) == 0u) out &= ~(0xFFu << (8 * b));
  return out;
}

}  // namespace

// One thread per (output row, 32-element block).  Output row i reads input
// row row_idx[i] (or i without row_idx); a row index outside [0, T) reads as
// zeros.  ATOMS: scales go to the atom layout of the block-scaled pipeline
// (atom (i / 128) * (H / 128) + b / 4, byte (i % 128 % 32) * 16 +
// (i % 128 / 32) * 4 + b % 4) and rows R .. rows_out - 1 get scale code 0;
// otherwise scales[i * (H / 32) + b].  codes [R, H] row-major.
template <bool ATOMS>
__global__ void mxfp8_quantize_kernel(const void *__restrict__ X, bool bf16, int64_t R, int64_t H,
                                      int64_t ld, const int64_t *__restrict__ row_idx, int64_t T,
                                      uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
                                      int64_t rows_out) {
  const int64_t nblk = H / 32;
  const int64_t total = rows_out * nblk;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = t / nblk;
    const int64_t b = t - i * nblk;
    uint32_t code = 0;
    if (i < R) {
      int64_t src = row_idx ? row_idx[i] : i;
      const bool valid = src >= 0 && src < T;
      float x[32];
      if (valid) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(X) +
                                                         src * ld + b * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 u = p[q];
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint16_t lo = static_cast<uint16_t>(w[e] & 0xFFFFu);
            const uint16_t hi = static_cast<uint16_t>(w[e] >> 16);
            if (bf16) {
              x[q * 8 + 2 * e] = __uint_as_float(static_cast<uint32_t>(lo) << 16);
              x[q * 8 + 2 * e + 1] = __uint_as_float(static_cast<uint32_t>(hi) << 16);
            } else {
              x[q * 8 + 2 * e] = __half2float(__ushort_as_half(lo));
              x[q * 8 + 2 * e + 1] = __half2float(__ushort_as_half(hi));
            }
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = 0.f;
      }
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(x[k]));
      const int fe = static_cast<int>((__float_as_uint(amax) >> 23) & 255u);
      code = amax > 0.f ? static_cast<uint32_t>(max(fe - 8, 0)) : 0u;
      code = min(code, 254u);
      const float inv = __uint_as_float((254u - min(code, 253u)) << 23);  // 2^(127 - code)
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t p0 = e4m3x2(x[4 * q + 1] * inv, x[4 * q] * inv);
        const uint32_t p1 = e4m3x2(x[4 * q + 3] * inv, x[4 * q + 2] * inv);
        w[q] = plus_zero4(p0 | (p1 << 16));
      }
      uint4 *o = reinterpret_cast<uint4 *>(codes + i * H + b * 32);
      o[0] = make_uint4(w[0], w[1], w[2], w[3]);
      o[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    if (ATOMS) {
      const int64_t r = i & 127;
      const int64_t atom = (i >> 7) * (H / 128) + (b >> 2);
      scales[atom * 512 + (r & 31) * 16 + (r >> 5) * 4 + (b & 3)] = static_cast<uint8_t>(code);
    } else if (i < R) {
      scales[i * nblk + b] = static_cast<uint8_t>(code);
    }
  }
}

cudaError_t launch_mxfp8_quantize(const void *X, bool bf16, int64_t R, int64_t H, int64_t ld,
                                  const int64_t *row_idx, int64_t T, uint8_t *codes,
                                  uint8_t *scales, bool atoms, int num_sms, cudaStream_t stream) {
  const int64_t rows_out = atoms ? (R + 127) / 128 * 128 : R;
  const int64_t total = rows_out * (H / 32);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  if (atoms)
    mxfp8_quantize_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        X, bf16, R, H, ld, row_idx, T, codes, scales, rows_out);
  else
    mxfp8_quantize_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        X, bf16, R, H, ld, row_idx, T, codes, scales, rows_out);
  return cudaGetLastError();
}

using KlBsEpi = KlEpiT<kMxBN, 16>;
#define KL_BS_KERNEL mx_kl_pipeline_kernel<KlBsEpi>

cudaError_t launch_kl_blockscaled(const KlBsArgs &a, cudaStream_t stream) {
  KlBsEpi::Params p{};
  p.n = a.sch.n;
  p.V = a.sch.V;
  p.pmt = a.pmt;
  p.pst = a.pst;
  p.pct = a.pct;
  p.pms = a.pms;
  p.pss = a.pss;
  p.counters = a.counters;
  p.splits = a.sch.splits * (kMxEpiWarps / 4);  // partial slots per row
  p.row_idx = a.row_idx;
  p.T = a.T;
  p.out_kl = a.out_kl;
  p.status = a.status;
  const uint32_t idesc_s = idesc_f16(a.bf16, kBM * 2, kMxBN, false, false);
  const uint32_t idesc_t = idesc_mx_e4m3_e2m1(kBM * 2, kMxBN);
  return launch_persistent(KL_BS_KERNEL, a.grid, kMxThreads, MxPipeLayout::kSmemBytes, 2, stream,
                           a.tmAs, a.tmBs, a.tmAt, a.tmBt, a.tmSfa, a.tmSfb, a.sch, idesc_s,
                           idesc_t, p, a.status);
}

int kl_bs_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64)
    return resident_units(KL_BS_KERNEL, kMxThreads, MxPipeLayout::kSmemBytes, 2, num_sms);
  if (!cached[dev])
    cached[dev] = resident_units(KL_BS_KERNEL, kMxThreads, MxPipeLayout::kSmemBytes, 2, num_sms);
  return cached[dev];
}

}  // namespace flp
