// kernels_fwd.cu -- forward scoring: response-row gather and the fused
// logits-tile -> online log-sum-exp/entropy pipeline, whose epilogue also
// merges the per-split partial states of a row into log-prob and entropy
// (the last warp to finish a 32-row group merges it).
//
// Arithmetic (miles PR #2764 summary, "Implementation breakdown" item 2:
// upcast first, temperature in FP32 after the upcast; entropy from the same
// values).  The tensor cores accumulate z = h W^T in FP32; nothing is rounded
// to model precision.  The epilogue works in base 2 on y = z * (log2 e / tau)
// (one FP32 multiply per logit: z/tau and the change of base folded), so
// every exponential is one ex2 on the special-function unit:
//   m = max y,  S = sum 2^(y-m),  B = sum 2^(y-m) (y-m)
// When m grows to m' the running sums are rescaled with a = 2^(m-m'):
//   S <- a S,  B <- a (B + (m-m') S).
// Then ln 2 (m + log2 S) = LSE(z/tau) and ln 2 (log2 S - B/S) = entropy.
//
// With a sampling support (SUP) only the support's columns enter m, S and B:
// the log-prob and entropy are those of softmax(z/tau) restricted to the
// support and renormalised, and a target outside it has log-prob -inf.  A
// column off the support has its logit replaced by a sentinel zs with
// y_s = zs * log2(e)/tau = -2^120 (finite), and the running max starts at
// y_s / 2 instead of -FLT_MAX: the sentinel never raises m, and every
// off-support term is 2^(y_s - m) <= 2^(y_s / 2) = 0 with a finite exponent,
// so it adds exactly 0 to S and B.  One select per logit; the fold itself is
// the unrestricted one.
#include <algorithm>
#include <cfloat>

#include <cuda.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "launch_util.cuh"
#include "lse_epilogue.cuh"
#include "vocab_pipeline.cuh"

namespace flp {

// ---------------------------------------------------------------- row gather
// hs[i, :] = h[row_idx[i], :] in 16-byte units, one warp per row.  Rows with
// an out-of-range index are zero-filled (the merge reports them).
__global__ void gather_rows_kernel(const uint4 *__restrict__ h, int64_t ld_h16,
                                   const int64_t *__restrict__ row_idx, int64_t n, int64_t T,
                                   int64_t H16, uint4 *__restrict__ hs) {
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < n;
       i += warps) {
    const int64_t r = row_idx[i];
    uint4 *dst = hs + i * H16;
    if (r < 0 || r >= T) {
      for (int64_t k = lane; k < H16; k += 32) dst[k] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4 *src = h + r * ld_h16;
    for (int64_t k = lane; k < H16; k += 32) dst[k] = __ldg(src + k);
  }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_gather(const void *h, int64_t ld_h, const int64_t *row_idx, int64_t n,
                          int64_t T, int64_t H, void *hs, int num_sms, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t warps_needed = n;
  int64_t blocks = (warps_needed + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  gather_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint4 *>(h), ld_h / 8, row_idx, n, T, H / 8, static_cast<uint4 *>(hs));
  return cudaGetLastError();
}

static_assert(kFwdTileCols == 2 * kFwdBN, "two MMAs per tile");
using FwdLayout = PipeLayout<kFwdBN, kFwdStages, 2, kFwdCG, 1, true>;
#define FWD_KERNEL(KMAX, SUP) \
  vocab_pipeline_kernel<kFwdBN, kFwdStages, 2, LseEpi<KMAX, SUP>, kFwdCG, 1, kFwdEpiWarps, true>
constexpr int kFwdThreads = pipe_threads(kFwdEpiWarps);

// Few scored rows: single CTAs on 128-row x kFwdBN-column tiles, two
// accumulator buffers, four epilogue warps.
using Fwd1Layout = PipeLayout<kFwdBN, kFwd1Stages, 1, 1, 2, false>;
#define FWD1_KERNEL(KMAX, SUP) \
  vocab_pipeline_kernel<kFwdBN, kFwd1Stages, 1, LseEpi<KMAX, SUP>, 1, 2, kFwd1EpiWarps, false>
constexpr int kFwd1Threads = pipe_threads(kFwd1EpiWarps);

// FEW: the single-CTA kernel, else the CTA-pair one.
template <int KMAX, bool SUP, bool FEW>
static cudaError_t launch_fwd_k(const FwdArgs &a, cudaStream_t stream) {
  typename LseEpi<KMAX, SUP>::Params p;
  p.targets = a.targets;
  p.K = a.K;
  p.row_idx = a.row_idx;
  p.T = a.T;
  p.n = a.sch.n;
  p.V = a.sch.V;
  p.sl = a.scale_log2;
  // y of the sentinel: -2^120, or as close as a finite float logit gets
  p.zsent = static_cast<float>(
      std::max(-1.329227995784916e36 / static_cast<double>(a.scale_log2), -0.5 * FLT_MAX));
  p.pm = a.pm;
  p.ps = a.ps;
  p.pb = a.pb;
  p.zt = a.zt;
  p.counters = a.counters;
  // partial slots per row
  p.splits = a.sch.splits * ((FEW ? kFwd1EpiWarps : kFwdEpiWarps) / 4);
  p.inv_tau = a.inv_tau;
  p.out_logp = a.out_logp;
  p.out_ent = a.out_ent;
  p.out_lse = a.out_lse;
  p.out_ez = a.out_ez;
  p.status = a.status;
  p.support = a.support;
  p.ld_support = a.ld_support;
  p.tile_cols = FEW ? kFwdBN : kFwdTileCols;
  if constexpr (FEW) {
    const uint32_t idesc = idesc_f16(a.bf16, kBM, kFwdBN, false, false);
    return launch_persistent(FWD1_KERNEL(KMAX, SUP), a.grid, kFwd1Threads, Fwd1Layout::kSmemBytes,
                             1, stream, a.tmA, a.tmB, a.tmA, a.tmB, a.sch, idesc, p, a.status);
  } else {
    const uint32_t idesc = idesc_f16(a.bf16, kBM * kFwdCG, kFwdBN, false, false);
    return launch_persistent(FWD_KERNEL(KMAX, SUP), a.grid, kFwdThreads, FwdLayout::kSmemBytes,
                             kFwdCG, stream, a.tmA, a.tmB, a.tmA, a.tmB, a.sch, idesc, p, a.status);
  }
}

template <bool FEW>
static cudaError_t launch_fwd_any(const FwdArgs &a, cudaStream_t stream) {
  if (a.support) {
    if (a.K != 1) return cudaErrorInvalidValue;  // the host API never asks for this
    return launch_fwd_k<1, true, FEW>(a, stream);
  }
  if (a.K == 1) return launch_fwd_k<1, false, FEW>(a, stream);
  return launch_fwd_k<kMaxTargets, false, FEW>(a, stream);
}

cudaError_t launch_fwd_scoring(const FwdArgs &a, cudaStream_t stream) {
  return launch_fwd_any<false>(a, stream);
}

cudaError_t launch_fwd_scoring_1cta(const FwdArgs &a, cudaStream_t stream) {
  return launch_fwd_any<true>(a, stream);
}

int fwd_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const auto kern = FWD_KERNEL(1, false);
  if (dev < 0 || dev >= 64) return resident_units(kern, kFwdThreads, FwdLayout::kSmemBytes, kFwdCG, num_sms);
  if (!cached[dev]) cached[dev] = resident_units(kern, kFwdThreads, FwdLayout::kSmemBytes, kFwdCG, num_sms);
  return cached[dev];
}

int fwd_smem_bytes() { return FwdLayout::kSmemBytes; }

int fwd1_units(int num_sms) { return num_sms; }

}  // namespace flp
