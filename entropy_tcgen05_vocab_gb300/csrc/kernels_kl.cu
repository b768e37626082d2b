// kernels_kl.cu -- full-vocabulary KL(teacher || student) without either
// logit tensor in memory (DeepSeek-V4 book ch. 19, "Never materialize
// logits" and "TileLang KL kernel": the teacher's logits are rebuilt from its
// cached hidden states through its prediction head and the exact KL is taken
// directly).
//
// Both heads run on the same (row tile, vocabulary tile): the pipeline issues
// two tcgen05 GEMMs per K step into two TMEM accumulators, z_s = h_s W_s^T and
// z_t = h_t W_t^T.  The epilogue keeps, per row, in base 2 (y = z log2 e):
//   teacher  m_t = max y_t,  S_t = sum 2^(y_t - m_t),
//            C_t = sum 2^(y_t - m_t) (z_t - z_s)      (natural units)
//   student  m_s = max y_s,  S_s = sum 2^(y_s - m_s)
// rescaling S and C by 2^(m - m') when a running max grows.  The last warp
// to finish a 32-row group merges the group's split partials and finishes
//   KL = sum_v p_t (log p_t - log p_s) = C_t / S_t - LSE_t + LSE_s,
//   LSE = ln 2 (m + log2 S).
#include <cuda.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "launch_util.cuh"
#include "vocab_pipeline.cuh"

namespace flp {

namespace {
constexpr float kLn2f = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;
}  // namespace

struct KlEpi {
  struct Params {
    int n;
    int V;
    float *pmt, *pst, *pct, *pms, *pss;  // [splits][n]
    uint32_t *counters;                   // [ceil(n/32)] items finished per 32-row group
    int splits;
    const int64_t *row_idx;
    int64_t T;
    float *out_kl;
    uint32_t *status;
    MxOperand mx;  // teacher head in MXFP4 (read by the MX pipeline's producer)
  };
  const Params p;
  float mt, st0, st1, ct0, ct1, ms, ss0, ss1;

  __device__ __forceinline__ explicit KlEpi(const Params &pp) : p(pp) {}

  __device__ __forceinline__ void begin(int /*mt*/, int /*row*/) {
    mt = ms = -FLT_MAX;
    st0 = st1 = ct0 = ct1 = ss0 = ss1 = 0.f;
  }

  __device__ __forceinline__ void rescale(float cmax_t, float cmax_s) {
    const float nt = fmaxf(mt, cmax_t * kLog2e);
    if (nt > mt) {
      const float a = ex2(mt - nt);
      st0 *= a;
      st1 *= a;
      ct0 *= a;
      ct1 *= a;
      mt = nt;
    }
    const float ns = fmaxf(ms, cmax_s * kLog2e);
    if (ns > ms) {
      const float a = ex2(ms - ns);
      ss0 *= a;
      ss1 *= a;
      ms = ns;
    }
  }

  __device__ __forceinline__ void fold_full(const float (&xs)[32], const float (&xt)[32]) {
    float cs = xs[0], ct = xt[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) {
      cs = fmaxf(cs, xs[j]);
      ct = fmaxf(ct, xt[j]);
    }
    rescale(ct, cs);
    const float nmt = -mt, nms = -ms;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float et0 = ex2(fmaf(xt[j], kLog2e, nmt));
      const float et1 = ex2(fmaf(xt[j + 1], kLog2e, nmt));
      st0 += et0;
      st1 += et1;
      ct0 = fmaf(et0, xt[j] - xs[j], ct0);
      ct1 = fmaf(et1, xt[j + 1] - xs[j + 1], ct1);
      ss0 += ex2(fmaf(xs[j], kLog2e, nms));
      ss1 += ex2(fmaf(xs[j + 1], kLog2e, nms));
    }
  }

  __device__ __forceinline__ void fold_masked(const float (&xs)[32], const float (&xt)[32],
                                              int nv) {
    float cs = -FLT_MAX, ct = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < nv) {
        cs = fmaxf(cs, xs[j]);
        ct = fmaxf(ct, xt[j]);
      }
    }
    rescale(ct, cs);
    const float nmt = -mt, nms = -ms;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < nv) {
        const float et = ex2(fmaf(xt[j], kLog2e, nmt));
        st0 += et;
        ct0 = fmaf(et, xt[j] - xs[j], ct0);
        ss0 += ex2(fmaf(xs[j], kLog2e, nms));
      }
    }
  }

  __device__ __forceinline__ void tile(uint32_t taddr, int col0, int nchunks) {
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int cb = col0 + c * 32;
      if (cb >= p.V) break;  // same for the whole warp
      float xs[32], xt[32];
      tmem_ld32(taddr + c * 32, xs);
      tmem_ld32(taddr + kKlBN + c * 32, xt);
      if (cb + 32 <= p.V)
        fold_full(xs, xt);
      else
        fold_masked(xs, xt, p.V - cb);
    }
  }

  __device__ __forceinline__ void end(int split, int row) {
    if (row < p.n) {
      const size_t o = static_cast<size_t>(split) * p.n + row;
      p.pmt[o] = mt;
      p.pst[o] = st0 + st1;
      p.pct[o] = ct0 + ct1;
      p.pms[o] = ms;
      p.pss[o] = ss0 + ss1;
    }
    if (last_arrival(p.counters + (row >> 5), static_cast<uint32_t>(p.splits)) && row < p.n)
      merge_row(row);
  }

  // Merge the split partials of one row and finish the KL.
  __device__ __forceinline__ void merge_row(int i) const {
    const int n = p.n;
    float Mt = -FLT_MAX, Ms = -FLT_MAX;
    for (int s = 0; s < p.splits; ++s) {
      const size_t o = static_cast<size_t>(s) * n + i;
      Mt = fmaxf(Mt, __ldcg(p.pmt + o));
      Ms = fmaxf(Ms, __ldcg(p.pms + o));
    }
    float St = 0.f, Ct = 0.f, Ss = 0.f;
    for (int s = 0; s < p.splits; ++s) {
      const size_t o = static_cast<size_t>(s) * n + i;
      const float at = exp2f(__ldcg(p.pmt + o) - Mt);
      St = fmaf(__ldcg(p.pst + o), at, St);
      Ct = fmaf(__ldcg(p.pct + o), at, Ct);
      Ss = fmaf(__ldcg(p.pss + o), exp2f(__ldcg(p.pms + o) - Ms), Ss);
    }
    float kl = Ct / St - kLn2f * ((Mt - Ms) + (log2f(St) - log2f(Ss)));
    if (p.row_idx) {
      const int64_t r = p.row_idx[i];
      if (r < 0 || r >= p.T) {
        atomicAdd(p.status + kStatBadRow, 1u);
        kl = __int_as_float(0x7fc00000);
      }
    }
    p.out_kl[i] = kl;
  }
};

using KlLayout = PipeLayout<kKlBN, kKlStages, 2, kKlCG, kKlAcc>;
using KlMxLayout = PipeLayout<kKlBN, kKlStages, 2, kKlCG, kKlAcc, false, true>;
// With the MX teacher head, four epilogue warps (the eight converter warps
// take the place of the other four).
constexpr int kKlMxEpiWarps = 4;
#define KL_KERNEL vocab_pipeline_kernel<kKlBN, kKlStages, 2, KlEpi, kKlCG, kKlAcc, kKlEpiWarps>
// the teacher head's B operand decoded from MXFP4 in shared memory
#define KL_MX_KERNEL \
  vocab_pipeline_kernel<kKlBN, kKlStages, 2, KlEpi, kKlCG, kKlAcc, kKlMxEpiWarps, false, true>
constexpr int kKlThreads = pipe_threads(kKlEpiWarps);
constexpr int kKlMxThreads = pipe_threads(kKlMxEpiWarps, true);

cudaError_t launch_kl(const KlArgs &a, cudaStream_t stream) {
  KlEpi::Params p;
  p.n = a.sch.n;
  p.V = a.sch.V;
  p.pmt = a.pmt;
  p.pst = a.pst;
  p.pct = a.pct;
  p.pms = a.pms;
  p.pss = a.pss;
  p.counters = a.counters;
  // partial slots per row
  p.splits = a.sch.splits * ((a.mx.packed ? kKlMxEpiWarps : kKlEpiWarps) / 4);
  p.row_idx = a.row_idx;
  p.T = a.T;
  p.out_kl = a.out_kl;
  p.status = a.status;
  p.mx = a.mx;
  const uint32_t idesc = idesc_f16(a.bf16, kBM * kKlCG, kKlBN, false, false);
  if (a.mx.packed)  // tmBt is unused: the teacher's B comes from the MXFP4 operand
    return launch_persistent(KL_MX_KERNEL, a.grid, kKlMxThreads, KlMxLayout::kSmemBytes, kKlCG,
                             stream, a.tmAs, a.tmBs, a.tmAt, a.tmBs, a.sch, idesc, p, a.status);
  return launch_persistent(KL_KERNEL, a.grid, kKlThreads, KlLayout::kSmemBytes, kKlCG, stream, a.tmAs, a.tmBs,
                           a.tmAt, a.tmBt, a.sch, idesc, p, a.status);
}

int kl_mx_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64)
    return resident_units(KL_MX_KERNEL, kKlMxThreads, KlMxLayout::kSmemBytes, kKlCG, num_sms);
  if (!cached[dev])
    cached[dev] = resident_units(KL_MX_KERNEL, kKlMxThreads, KlMxLayout::kSmemBytes, kKlCG, num_sms);
  return cached[dev];
}

int kl_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return resident_units(KL_KERNEL, kKlThreads, KlLayout::kSmemBytes, kKlCG, num_sms);
  if (!cached[dev]) cached[dev] = resident_units(KL_KERNEL, kKlThreads, KlLayout::kSmemBytes, kKlCG, num_sms);
  return cached[dev];
}

}  // namespace flp
