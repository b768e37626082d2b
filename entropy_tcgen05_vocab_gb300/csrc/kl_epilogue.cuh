// kl_epilogue.cuh -- the epilogue of the KL pipelines: folds the student and
// teacher logit tiles straight out of TMEM into per-row running states and
// merges the vocabulary splits (DeepSeek-V4 book ch. 19, "TileLang KL
// kernel": the exact full-vocabulary KL with neither logit tensor in memory).
//
// Per row, in base 2 (y = z log2 e):
//   teacher  m_t = max y_t,  S_t = sum 2^(y_t - m_t),
//            C_t = sum 2^(y_t - m_t) (z_t - z_s)      (natural units)
//   student  m_s = max y_s,  S_s = sum 2^(y_s - m_s)
// rescaling S and C by 2^(m - m') when a running max grows.  The last warp
// to finish a 32-row group merges the group's split partials and finishes
//   KL = sum_v p_t (log p_t - log p_s) = C_t / S_t - LSE_t + LSE_s,
//   LSE = ln 2 (m + log2 S).
// TBN: TMEM column offset of the teacher accumulator from the student's.
// CW: columns read and folded per step (32 or 16).
#pragma once

#include <cfloat>
#include <cstdint>

#include "ptx.cuh"
#include "schedule.h"
#include "vocab_pipeline.cuh"

namespace flp {

namespace kl_detail {
constexpr float kLn2f = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;
}  // namespace kl_detail

template <int TBN, int CW>
struct KlEpiT {
  static_assert(CW == 32 || CW == 16, "fold 32 or 16 columns at a time");
  static constexpr int kChunk = CW;
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

  __device__ __forceinline__ explicit KlEpiT(const Params &pp) : p(pp) {}

  __device__ __forceinline__ void begin(int /*mt*/, int /*row*/) {
    mt = ms = -FLT_MAX;
    st0 = st1 = ct0 = ct1 = ss0 = ss1 = 0.f;
  }

  __device__ __forceinline__ void rescale(float cmax_t, float cmax_s) {
    const float nt = fmaxf(mt, cmax_t * kl_detail::kLog2e);
    if (nt > mt) {
      const float a = ex2(mt - nt);
      st0 *= a;
      st1 *= a;
      ct0 *= a;
      ct1 *= a;
      mt = nt;
    }
    const float ns = fmaxf(ms, cmax_s * kl_detail::kLog2e);
    if (ns > ms) {
      const float a = ex2(ms - ns);
      ss0 *= a;
      ss1 *= a;
      ms = ns;
    }
  }

  __device__ __forceinline__ void fold_full(const float (&xs)[CW], const float (&xt)[CW]) {
    float cs = xs[0], ct = xt[0];
#pragma unroll
    for (int j = 1; j < CW; ++j) {
      cs = fmaxf(cs, xs[j]);
      ct = fmaxf(ct, xt[j]);
    }
    rescale(ct, cs);
    const float nmt = -mt, nms = -ms;
#pragma unroll
    for (int j = 0; j < CW; j += 2) {
      const float et0 = ex2(fmaf(xt[j], kl_detail::kLog2e, nmt));
      const float et1 = ex2(fmaf(xt[j + 1], kl_detail::kLog2e, nmt));
      st0 += et0;
      st1 += et1;
      ct0 = fmaf(et0, xt[j] - xs[j], ct0);
      ct1 = fmaf(et1, xt[j + 1] - xs[j + 1], ct1);
      ss0 += ex2(fmaf(xs[j], kl_detail::kLog2e, nms));
      ss1 += ex2(fmaf(xs[j + 1], kl_detail::kLog2e, nms));
    }
  }

  __device__ __forceinline__ void fold_masked(const float (&xs)[CW], const float (&xt)[CW],
                                              int nv) {
    float cs = -FLT_MAX, ct = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < CW; ++j) {
      if (j < nv) {
        cs = fmaxf(cs, xs[j]);
        ct = fmaxf(ct, xt[j]);
      }
    }
    rescale(ct, cs);
    const float nmt = -mt, nms = -ms;
#pragma unroll
    for (int j = 0; j < CW; ++j) {
      if (j < nv) {
        const float et = ex2(fmaf(xt[j], kl_detail::kLog2e, nmt));
        st0 += et;
        ct0 = fmaf(et, xt[j] - xs[j], ct0);
        ss0 += ex2(fmaf(xs[j], kl_detail::kLog2e, nms));
      }
    }
  }

  __device__ __forceinline__ void tile(uint32_t taddr, int col0, int nchunks) {
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int cb = col0 + c * CW;
      if (cb >= p.V) break;  // same for the whole warp
      float xs[CW], xt[CW];
      if constexpr (CW == 32) {
        tmem_ld32(taddr + c * CW, xs);
        tmem_ld32(taddr + TBN + c * CW, xt);
      } else {
        tmem_ld16(taddr + c * CW, xs);
        tmem_ld16(taddr + TBN + c * CW, xt);
      }
      if (cb + CW <= p.V)
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
    float kl = Ct / St - kl_detail::kLn2f * ((Mt - Ms) + (log2f(St) - log2f(Ss)));
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

}  // namespace flp
