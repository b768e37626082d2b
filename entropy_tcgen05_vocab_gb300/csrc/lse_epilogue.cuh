// lse_epilogue.cuh -- the forward's epilogue: folds FP32 logit tiles,
// straight out of tensor memory, into per-row online log-sum-exp/entropy
// state, and merges the per-split partial states of a row into log-prob and
// entropy (the last warp to finish a 32-row group merges it).  Shared by the
// bf16/fp16 forward (kernels_fwd.cu) and the block-scaled forward
// (kernels_fwdmx.cu).
//
// Arithmetic (miles PR #2764 summary, "Implementation breakdown" item 2:
// upcast first, temperature in FP32 after the upcast; entropy from the same
// values): base 2 on y = z * (log2 e / tau), one FP32 multiply per logit,
//   m = max y,  S = sum 2^(y-m),  B = sum 2^(y-m) (y-m),
// rescaled with a = 2^(m-m') when m grows to m':  S <- a S,  B <- a (B + (m-m') S);
// then LSE(z/tau) = ln 2 (m + log2 S) and entropy = ln 2 (log2 S - B/S).
#pragma once

#include <cfloat>
#include <cstdint>

#include "ptx.cuh"
#include "schedule.h"
#include "support.cuh"
#include "vocab_pipeline.cuh"

namespace flp {

constexpr float kLn2 = 0.693147180559945309f;

// KMAX = largest number of target tokens per row the instantiation handles
// (1 for log-prob + entropy; up to kMaxTargets for K-candidate scoring).
// SUP: restrict each row to its sampling support.
template <int KMAX, bool SUP = false>
struct LseEpi {
  struct Params {
    const int64_t *targets;  // [T, K], by h row
    int K;                   // targets per row, 1 <= K <= KMAX
    const int64_t *row_idx;  // [n] or null
    int64_t T;
    int n;
    int V;
    float sl;                // log2(e) / tau
    float zsent;             // SUP: logit given to columns off the support
    float *pm, *ps, *pb;     // [slots][n] partial m, S, B
    float *zt;               // [n, K] raw FP32 logits of the targets
    uint32_t *counters;      // [ceil(n/32)] items finished per 32-row group
    int splits;              // partial slots per row
    float inv_tau;
    float *out_logp;         // [n, K]
    float *out_ent, *out_lse, *out_ez;  // [n], any may be null
    uint32_t *status;
    const uint32_t *support;  // SUP: [T, ld_support] words by h row
    int64_t ld_support;
    int tile_cols;            // columns from one tile() call of a warp to its next
  };
  const Params p;
  float m, s0, s1, b0, b1;
  int tgt[KMAX];  // -1: no valid target (never matched)
  int row_;
  SupportRow sup;

  __device__ __forceinline__ explicit LseEpi(const Params &pp) : p(pp) {}

  __device__ __forceinline__ void begin(int /*mt*/, int row) {
    m = SUP ? 0.5f * (p.zsent * p.sl) : -FLT_MAX;
    s0 = s1 = b0 = b1 = 0.f;
    row_ = row;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) tgt[k] = -1;
    if (SUP) sup.reset(nullptr, p.V);
    if (row < p.n) {
      const int64_t r = p.row_idx ? p.row_idx[row] : row;
      if (r >= 0 && r < p.T) {
        if (SUP) sup.reset(p.support + r * p.ld_support, p.V);
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          if (k < p.K) {
            const int64_t t = p.targets[r * p.K + k];
            if (t >= 0 && t < p.V) tgt[k] = static_cast<int>(t);
          }
        }
      }
    }
  }

  __device__ __forceinline__ void rescale(float cmax) {
    const float mn = fmaxf(m, cmax * p.sl);
    if (mn > m) {
      const float d = m - mn;
      const float a = ex2(d);
      b0 = a * fmaf(d, s0, b0);
      b1 = a * fmaf(d, s1, b1);
      s0 *= a;
      s1 *= a;
      m = mn;
    }
  }

  __device__ __forceinline__ void fold_full(const float (&x)[32]) {
    float cmax = x[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, x[j]);
    rescale(cmax);
    const float nm = -m;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float d0 = fmaf(x[j], p.sl, nm);
      const float d1 = fmaf(x[j + 1], p.sl, nm);
      const float e0 = ex2(d0);
      const float e1 = ex2(d1);
      s0 += e0;
      s1 += e1;
      b0 = fmaf(e0, d0, b0);
      b1 = fmaf(e1, d1, b1);
    }
  }

  __device__ __forceinline__ void fold_masked(const float (&x)[32], int nv) {
    float cmax = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) cmax = fmaxf(cmax, x[j]);
    rescale(cmax);
    const float nm = -m;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < nv) {
        const float d = fmaf(x[j], p.sl, nm);
        const float e = ex2(d);
        s0 += e;
        b0 = fmaf(e, d, b0);
      }
    }
  }

  __device__ __forceinline__ void tile(uint32_t taddr, int col0, int nchunks) {
    if (SUP) sup.start(col0);
    // With several targets, bit c marks the chunks that hold one, so a chunk
    // without any costs one test instead of KMAX.
    uint32_t hit = 0xffffffffu;
    if (KMAX > 1) {
      hit = 0u;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int rel = tgt[k] - col0;
        if (static_cast<unsigned>(rel) < static_cast<unsigned>(nchunks * 32)) hit |= 1u << (rel >> 5);
      }
    }
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int cb = col0 + c * 32;
      if (cb >= p.V) break;  // same for the whole warp
      const uint32_t w = SUP ? sup.next(col0, c) : 0u;
      float x[32];
      tmem_ld32(taddr + c * 32, x);
      if (SUP) {
        const uint32_t wc = sup.clip(w, cb);
        float xs[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) xs[j] = ((wc >> j) & 1u) ? x[j] : p.zsent;
        fold_full(xs);
      } else if (cb + 32 <= p.V) {
        fold_full(x);
      } else {
        fold_masked(x, p.V - cb);
      }
      // each target column lies in exactly one chunk: store its raw logit there
      if (!((hit >> c) & 1u)) continue;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int rel = tgt[k] - cb;
        if (static_cast<unsigned>(rel) < 32u) {
          float t = x[0];
#pragma unroll
          for (int j = 1; j < 32; ++j) t = (rel == j) ? x[j] : t;
          p.zt[static_cast<size_t>(row_) * p.K + k] = t;
        }
      }
    }
    if (SUP) sup.prefetch(col0 + p.tile_cols);
  }

  __device__ __forceinline__ void end(int split, int row) {
    if (row < p.n) {
      const size_t o = static_cast<size_t>(split) * p.n + row;
      p.pm[o] = m;
      p.ps[o] = s0 + s1;
      p.pb[o] = b0 + b1;
    }
    // The last warp to finish these 32 rows merges them.
    if (last_arrival(p.counters + (row >> 5), static_cast<uint32_t>(p.splits)) && row < p.n)
      merge_row(row);
  }

  // Merge the split partials (m_i, S_i, B_i) of one row:
  //   M = max m_i,  S = sum S_i 2^(m_i - M),  B = sum 2^(m_i - M) (B_i + (m_i - M) S_i),
  // then logp = z_tgt / tau - LSE and entropy = ln 2 (log2 S - B / S).
  __device__ __forceinline__ void merge_row(int i) const {
    const int n = p.n;
    float M = -FLT_MAX;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, __ldcg(p.pm + static_cast<size_t>(s) * n + i));
    float S = 0.f, B = 0.f;
    for (int s = 0; s < p.splits; ++s) {
      const size_t o = static_cast<size_t>(s) * n + i;
      const float d = __ldcg(p.pm + o) - M;
      const float a = exp2f(d);
      const float si = __ldcg(p.ps + o);
      S = fmaf(si, a, S);
      B = fmaf(a, fmaf(d, si, __ldcg(p.pb + o)), B);
    }
    const float l2s = log2f(S);
    float lse = kLn2 * (M + l2s);
    float ent = kLn2 * (l2s - B / S);
    const float qnan = __int_as_float(0x7fc00000);
    const int64_t r = p.row_idx ? p.row_idx[i] : i;
    const bool row_ok = r >= 0 && r < p.T;
    bool empty = false;
    if (!row_ok) {
      atomicAdd(p.status + kStatBadRow, 1u);
      lse = ent = qnan;
    } else if (SUP && !(S > 0.f)) {  // no token of the row is in its support
      atomicAdd(p.status + kStatEmptySupport, 1u);
      lse = ent = qnan;
      empty = true;
    }
    for (int k = 0; k < p.K; ++k) {
      const size_t o = static_cast<size_t>(i) * p.K + k;
      float logp = qnan;
      if (row_ok) {
        const int64_t t = p.targets[r * p.K + k];
        if (t < 0 || t >= p.V)
          atomicAdd(p.status + kStatBadTarget, 1u);
        else if (SUP && !empty && !((__ldg(p.support + r * p.ld_support + (t >> 5)) >> (t & 31)) & 1u))
          logp = -INFINITY;  // target outside the support
        else
          logp = __ldcg(p.zt + o) * p.inv_tau - lse;
      }
      if (p.out_logp) p.out_logp[o] = logp;
    }
    if (p.out_ent) p.out_ent[i] = ent;
    if (p.out_lse) p.out_lse[i] = lse;
    if (p.out_ez) p.out_ez[i] = lse - ent;
  }
};

}  // namespace flp
