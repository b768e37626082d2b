// kernels_bwd.cu -- backward of L = sum_i g1_i logp_i + g2_i ent_i by tile
// recompute (miles PR #4645, "How it works": Op -- the backward replays each
// tile instead of keeping the [tokens x vocab] logits or their gradient).
//
// For a chunk of R scored rows:
//   1. grad pass: the vocabulary pipeline recomputes z = h W^T tile by tile
//      and its epilogue turns each FP32 logit straight into the gradient of
//      the loss w.r.t. that logit,
//        G_v = (g1 (1[v = tgt] - p_v) - g2 p_v (z'_v - E_p[z'])) / tau,
//        p_v = exp(z'_v - LSE),  z' = z / tau,
//      with LSE and E_p[z'] from the forward statistics, written in the
//      model dtype into the bounded chunk buffer G [R, V];
//   2. dh[rows] = G W           (tcgen05 GEMM, K = V, W read MN-major);
//   3. dW (+)= G^T h[rows]      (tcgen05 GEMM, K = R, both operands MN-major).
// With a sampling support, LSE and E_p[z'] are taken over the support (the
// statistics pass restricts them the same way) and G is 0 off the support.
#include <algorithm>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gemm_pipeline.cuh"
#include "launch.h"
#include "launch_util.cuh"
#include "support.cuh"
#include "vocab_pipeline.cuh"

namespace flp {

namespace {
constexpr float kLog2eF = 1.442695040888963407f;

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
  if (bf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
  }
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ uint16_t pack1(float a, bool bf16) {
  if (bf16) {
    const __nv_bfloat16 v = __float2bfloat16_rn(a);
    return *reinterpret_cast<const uint16_t *>(&v);
  }
  const __half v = __float2half_rn(a);
  return *reinterpret_cast<const uint16_t *>(&v);
}

// 32 FP32 values -> 32 16-bit values at dst (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store32_16(void *dst, const float (&v)[32], bool bf16) {
  uint4 *d = static_cast<uint4 *>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack2(v[8 * q + 0], v[8 * q + 1], bf16);
    u.y = pack2(v[8 * q + 2], v[8 * q + 3], bf16);
    u.z = pack2(v[8 * q + 4], v[8 * q + 5], bf16);
    u.w = pack2(v[8 * q + 6], v[8 * q + 7], bf16);
    d[q] = u;
  }
}
// One 256-bit global store (8 words; dst 32-byte aligned).  A warp whose
// lanes each write a different row touches one line per lane per store, so
// storing a row's 64 or 128 bytes in 32-byte pieces halves the store
// instructions (and the lines the L1 processes) against 16-byte pieces.
__device__ __forceinline__ void st_global_v8(void *dst, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t a4, uint32_t a5, uint32_t a6,
                                             uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// One 256-bit global load (8 words; src 32-byte aligned).
__device__ __forceinline__ void ld_global_v8(const void *src, uint32_t (&a)[8]) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]),
                 "=r"(a[6]), "=r"(a[7])
               : "l"(src));
}

// store32_16 with 32-byte stores (dst 32-byte aligned).
__device__ __forceinline__ void store32_16_v8(void *dst, const float (&v)[32], bool bf16) {
  uint8_t *d = static_cast<uint8_t *>(dst);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float *w = v + 16 * q;
    st_global_v8(d + 32 * q, pack2(w[0], w[1], bf16), pack2(w[2], w[3], bf16),
                 pack2(w[4], w[5], bf16), pack2(w[6], w[7], bf16), pack2(w[8], w[9], bf16),
                 pack2(w[10], w[11], bf16), pack2(w[12], w[13], bf16), pack2(w[14], w[15], bf16));
  }
}

// Scored rows per h row (row_idx may name a row more than once).
__global__ void count_rows_kernel(const int64_t *__restrict__ row_idx, int64_t n, int64_t T,
                                  uint32_t *__restrict__ cnt) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t r = row_idx[i];
    if (r >= 0 && r < T) atomicAdd(cnt + r, 1u);
  }
}
}  // namespace

// ---------------------------------------------------------------- grad pass
template <bool SUP>
struct GradEpi {
  struct Params {
    int n;       // rows in the chunk
    int V;
    int r0;      // first scored position of the chunk
    int64_t T;
    const int64_t *targets;
    const int64_t *row_idx;
    const float *lse, *ez, *g1, *g2;
    float sl, inv_tau;
    uint16_t *G;  // [n, ldg]
    int64_t ldg;
    bool bf16;
    bool v8;      // G and its rows 32-byte aligned: 32-byte stores
    const uint32_t *support;  // SUP: [T, ld_support] words by h row
    int64_t ld_support;
    int tile_cols;            // columns from one tile() call of a warp to its next
  };
  const Params p;
  // G_v = a1 1[v = tgt] - p_v (a1 + a2 (z_v / tau - E z')), a1 = g1 / tau,
  // a2 = g2 / tau, folded per row into -p_v (c1 z_v + c0) with
  // c1 = a2 / tau and c0 = a1 - a2 E z' (z_v the raw FP32 logit).
  float lse2, a1, c1, c0;
  int tgt;
  bool valid;
  uint16_t *grow;
  SupportRow sup;

  __device__ __forceinline__ explicit GradEpi(const Params &pp) : p(pp) {}

  __device__ __forceinline__ void begin(int /*mt*/, int row) {
    valid = row < p.n;
    tgt = -1;
    lse2 = a1 = c1 = c0 = 0.f;
    grow = p.G + static_cast<int64_t>(valid ? row : 0) * p.ldg;
    if (SUP) sup.reset(nullptr, p.V);
    if (!valid) return;
    const int i = p.r0 + row;
    lse2 = p.lse[i] * kLog2eF;
    a1 = p.g1[i] * p.inv_tau;
    const float a2 = p.g2[i] * p.inv_tau;
    c1 = a2 * p.inv_tau;
    c0 = fmaf(-a2, p.ez[i], a1);
    const int64_t r = p.row_idx ? p.row_idx[i] : i;
    if (r >= 0 && r < p.T) {
      const int64_t t = p.targets[r];
      if (t >= 0 && t < p.V) tgt = static_cast<int>(t);
      if (SUP) sup.reset(p.support + r * p.ld_support, p.V);
    }
  }

  __device__ __forceinline__ void tile(uint32_t taddr, int col0, int nchunks) {
    if (SUP) sup.start(col0);
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int cb = col0 + c * 32;
      if (cb >= p.V) break;  // same for the whole warp
      const uint32_t w = SUP ? sup.next(col0, c) : 0u;
      float x[32];
      tmem_ld32(taddr + c * 32, x);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float pr = ex2(fmaf(x[j], p.sl, -lse2));
        x[j] = -pr * fmaf(x[j], c1, c0);
      }
      const int rel = tgt - cb;
      if (static_cast<unsigned>(rel) < 32u) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] += (rel == j) ? a1 : 0.f;
      }
      if (SUP) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = ((w >> j) & 1u) ? x[j] : 0.f;
      }
      if (!valid) continue;
      if (cb + 32 <= p.V) {
        if (p.v8)
          store32_16_v8(grow + cb, x, p.bf16);
        else
          store32_16(grow + cb, x, p.bf16);
      } else {
        const int nv = p.V - cb;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nv) grow[cb + j] = pack1(x[j], p.bf16);
      }
    }
    if (SUP) sup.prefetch(col0 + p.tile_cols);
  }

  __device__ __forceinline__ void end(int, int) {}
};

// ---------------------------------------------------------------- dh = G W
struct DhEpi {
  struct Params {
    int R, H, r0;
    int64_t T;
    const int64_t *row_idx;
    const uint32_t *rowcnt;  // scored rows per h row, or null (row_idx null: all distinct)
    uint16_t *dh;
    int64_t ld;
    bool bf16;
  };
  const Params p;
  __device__ __forceinline__ explicit DhEpi(const Params &pp) : p(pp) {}

  // Destination of product row `row` (chunk-local): the dh row, whether it
  // is valid, and whether that h row is scored more than once.
  struct Dest {
    uint16_t *drow;
    bool valid, repeated;
  };
  __device__ __forceinline__ static Dest dest(const Params &p, int row) {
    bool valid = row < p.R;
    int64_t orig = 0;
    if (valid) {
      orig = p.row_idx ? p.row_idx[p.r0 + row] : p.r0 + row;
      valid = orig >= 0 && orig < p.T;
    }
    const bool repeated = valid && p.rowcnt && p.rowcnt[orig] > 1u;
    return Dest{p.dh + (valid ? orig : 0) * p.ld, valid, repeated};
  }

  // Store 32 columns [col, col + 32) of one product row (those below H).
  // A row scored more than once gets the sum of its contributions: added
  // with packed 16-bit atomics onto the zeroed dh row (in any chunk order).
  __device__ __forceinline__ static void store(const Params &p, const Dest &d, int col,
                                               const float (&x)[32]) {
    if (d.repeated) {
      // H is a multiple of 8, so the valid columns of a chunk come in pairs
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        if (col + j >= p.H) break;
        if (p.bf16)
          atomicAdd(reinterpret_cast<__nv_bfloat162 *>(d.drow + col + j),
                    __floats2bfloat162_rn(x[j], x[j + 1]));
        else
          atomicAdd(reinterpret_cast<__half2 *>(d.drow + col + j), __floats2half2_rn(x[j], x[j + 1]));
      }
    } else if (col + 32 <= p.H) {
      store32_16(d.drow + col, x, p.bf16);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col + j < p.H) d.drow[col + j] = pack1(x[j], p.bf16);
    }
  }

  __device__ __forceinline__ void tile(uint32_t taddr, int row, int col0, int ncols) {
    const Dest d = dest(p, row);
#pragma unroll 1
    for (int c = 0; c < ncols / 32; ++c) {
      const int col = col0 + c * 32;
      if (col >= p.H) break;
      float x[32];
      tmem_ld32(taddr + c * 32, x);
      if (d.valid) store(p, d, col, x);
    }
  }
};

// The tail tiles of the dh GEMM were split into K segments whose FP32
// partial tiles sit in `part` (slot j * split + s for segment s of tail tile
// j, tile_m x tile_n row-major).  One thread per (row, 32-column chunk) of
// a tail tile adds the segments in order (so the result does not depend on
// which CTA finished first) and stores the sum as DhEpi does.
__global__ void __launch_bounds__(256) dh_tail_sum_kernel(const float *__restrict__ part,
                                                           int tail_tiles, int split,
                                                           int full_tiles, int n_tiles,
                                                           int tile_m, int tile_n,
                                                           DhEpi::Params p) {
  const int chunks = tile_n / 32;
  const int64_t total = static_cast<int64_t>(tail_tiles) * tile_m * chunks;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % chunks);
    const int r = static_cast<int>((i / chunks) % tile_m);
    const int j = static_cast<int>(i / (static_cast<int64_t>(chunks) * tile_m));
    const int t = full_tiles + j;
    const int mt = t / n_tiles, nt = t - (t / n_tiles) * n_tiles;
    const int row = mt * tile_m + r;
    const int col = nt * tile_n + c * 32;
    if (row >= p.R || col >= p.H) continue;
    const DhEpi::Dest d = DhEpi::dest(p, row);
    if (!d.valid) continue;
    float x[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) x[q] = 0.f;
    for (int sgm = 0; sgm < split; ++sgm) {
      const float4 *src = reinterpret_cast<const float4 *>(
          part + (static_cast<size_t>(j) * split + sgm) * tile_m * tile_n +
          static_cast<size_t>(r) * tile_n + c * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 v = __ldcg(src + q);
        x[4 * q] += v.x;
        x[4 * q + 1] += v.y;
        x[4 * q + 2] += v.z;
        x[4 * q + 3] += v.w;
      }
    }
    DhEpi::store(p, d, col, x);
  }
}

// ---------------------------------------------------------------- dW = G^T h
struct DwEpi {
  struct Params {
    int V, H;
    float *dW;
    int64_t ld;
    int accumulate;
    bool v8;  // dW 32-byte aligned (its rows are, ld being a multiple of 8): 32-byte stores
  };
  const Params p;
  __device__ __forceinline__ explicit DwEpi(const Params &pp) : p(pp) {}

  __device__ __forceinline__ void tile(uint32_t taddr, int v, int col0, int ncols) {
    const bool valid = v < p.V;
    float *drow = p.dW + static_cast<int64_t>(valid ? v : 0) * p.ld;
#pragma unroll 1
    for (int c = 0; c < ncols / 32; ++c) {
      const int col = col0 + c * 32;
      if (col >= p.H) break;
      float x[32];
      tmem_ld32(taddr + c * 32, x);
      if (!valid) continue;
      if (col + 32 <= p.H && p.v8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = x[8 * q + e];
          if (p.accumulate) {  // a later row chunk adds onto dW
            uint32_t prev[8];
            ld_global_v8(drow + col + 8 * q, prev);
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] += __uint_as_float(prev[e]);
          }
          st_global_v8(drow + col + 8 * q, __float_as_uint(w[0]), __float_as_uint(w[1]),
                       __float_as_uint(w[2]), __float_as_uint(w[3]), __float_as_uint(w[4]),
                       __float_as_uint(w[5]), __float_as_uint(w[6]), __float_as_uint(w[7]));
        }
      } else if (col + 32 <= p.H) {
        float4 *d = reinterpret_cast<float4 *>(drow + col);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 o = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
          if (p.accumulate) {
            const float4 prev = d[q];
            o.x += prev.x;
            o.y += prev.y;
            o.z += prev.z;
            o.w += prev.w;
          }
          d[q] = o;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col + j < p.H) drow[col + j] = p.accumulate ? drow[col + j] + x[j] : x[j];
      }
    }
  }
};

// ---------------------------------------------------------------- launchers
static_assert(kGradTileCols == 2 * kGradBN, "two MMAs per tile");
using GradLayout = PipeLayout<kGradBN, kGradStages, 2, kGradCG, 1, true>;
#define GRAD_KERNEL(SUP) \
  vocab_pipeline_kernel<kGradBN, kGradStages, 2, GradEpi<SUP>, kGradCG, 1, kGradEpiWarps, true>
constexpr int kGradThreads = pipe_threads(kGradEpiWarps);

template <bool SUP>
static cudaError_t launch_grad_t(const GradArgs &a, cudaStream_t stream) {
  typename GradEpi<SUP>::Params p;
  p.n = a.sch.n;
  p.V = a.sch.V;
  p.r0 = a.r0;
  p.T = a.T;
  p.targets = a.targets;
  p.row_idx = a.row_idx;
  p.lse = a.lse;
  p.ez = a.ez;
  p.g1 = a.g1;
  p.g2 = a.g2;
  p.sl = a.scale_log2;
  p.inv_tau = a.inv_tau;
  p.G = static_cast<uint16_t *>(a.G);
  p.ldg = a.ldg;
  p.bf16 = a.bf16;
  p.v8 = (reinterpret_cast<uintptr_t>(a.G) & 31u) == 0 && (a.ldg * 2) % 32 == 0;
  p.support = a.support;
  p.ld_support = a.ld_support;
  p.tile_cols = kGradTileCols;
  const uint32_t idesc = idesc_f16(a.bf16, kBM * kGradCG, kGradBN, false, false);
  return launch_persistent(GRAD_KERNEL(SUP), a.grid, kGradThreads, GradLayout::kSmemBytes, kGradCG,
                           stream, a.tmA, a.tmB, a.tmA, a.tmB, a.sch, idesc, p, a.status);
}

cudaError_t launch_grad(const GradArgs &a, cudaStream_t stream) {
  return a.support ? launch_grad_t<true>(a, stream) : launch_grad_t<false>(a, stream);
}

int grad_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const auto kern = GRAD_KERNEL(false);
  if (dev < 0 || dev >= 64) return resident_units(kern, kGradThreads, GradLayout::kSmemBytes, kGradCG, num_sms);
  if (!cached[dev]) cached[dev] = resident_units(kern, kGradThreads, GradLayout::kSmemBytes, kGradCG, num_sms);
  return cached[dev];
}

constexpr int kGemmCG = 2;
// Both backward GEMMs use 512-column output tiles (measured: +4 % each over
// 256-column tiles, although dh has few tiles to spread over the CTA pairs).
constexpr bool kDhWide = true;
constexpr bool kDwWide = true;
using DhCfg = GemmCfg<kGemmCG, kDhWide>;
using DwCfg = GemmCfg<kGemmCG, kDwWide>;
#define DH_KERNEL gemm_kernel<false, true, DhEpi, kGemmCG, kDhWide>
#define DW_KERNEL gemm_kernel<true, true, DwEpi, kGemmCG, kDwWide>

static GemmShape gemm_shape(int M, int N, int K, int tile_n) {
  GemmShape g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.m_tiles = (M + kBM * kGemmCG - 1) / (kBM * kGemmCG);
  g.n_tiles = (N + tile_n - 1) / tile_n;
  g.tiles = g.m_tiles * g.n_tiles;
  g.k_blocks = (K + kBK - 1) / kBK;
  g.items = g.tiles;
  g.full_tiles = g.tiles;
  g.split = 1;
  g.kb_per_seg = g.k_blocks;
  g.part = nullptr;
  g.wait_ns = 0;
  return g;
}

DhSplit dh_split_plan(int M, int N, int K, int units, int max_slots) {
  const GemmShape g = gemm_shape(M, N, K, DhCfg::kTileN);
  DhSplit d{g.tiles, g.tiles, 0, 1, g.k_blocks, g.tiles};
  if (g.tiles <= 0 || units <= 0) return d;
  const int rem = g.tiles % units;
  // split only a last wave that leaves at least half of the pairs idle
  if (rem == 0 || 2 * rem > units) return d;
  int s = units / rem;
  s = std::min(s, g.k_blocks / kDhSplitMinKb);
  s = std::min(s, max_slots / rem);
  if (s < 2) return d;
  const int per = (g.k_blocks + s - 1) / s;
  s = (g.k_blocks + per - 1) / per;  // every segment non-empty
  if (s < 2) return d;
  d.full_tiles = g.tiles - rem;
  d.tail = rem;
  d.split = s;
  d.kb_per_seg = per;
  d.items = d.full_tiles + rem * s;
  return d;
}

int dh_gemm_tiles(int M, int N) { return gemm_shape(M, N, 1, DhCfg::kTileN).tiles; }
int dw_gemm_tiles(int M, int N) { return gemm_shape(M, N, 1, DwCfg::kTileN).tiles; }
int gemm_cta_group() { return kGemmCG; }

int gemm_units(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const int t = pipe_threads(DwCfg::kEpiw);
  if (dev < 0 || dev >= 64) return resident_units(DW_KERNEL, t, DwCfg::L::kSmemBytes, kGemmCG, num_sms);
  if (!cached[dev]) cached[dev] = resident_units(DW_KERNEL, t, DwCfg::L::kSmemBytes, kGemmCG, num_sms);
  return cached[dev];
}

cudaError_t launch_dh_gemm(const GemmArgs &a, cudaStream_t stream) {
  DhEpi::Params p;
  p.R = a.M;
  p.H = a.N;
  p.r0 = a.r0;
  p.T = a.T;
  p.row_idx = a.row_idx;
  p.rowcnt = a.rowcnt;
  p.dh = static_cast<uint16_t *>(a.dh);
  p.ld = a.ld_dh;
  p.bf16 = a.bf16;
  GemmShape g = gemm_shape(a.M, a.N, a.K, DhCfg::kTileN);
  const DhSplit &d = a.dh_split;
  const bool split = d.split > 1;
  if (split) {
    if (!a.part || d.tiles != g.tiles || d.full_tiles + d.tail != g.tiles) return cudaErrorInvalidValue;
    g.full_tiles = d.full_tiles;
    g.split = d.split;
    g.kb_per_seg = d.kb_per_seg;
    g.items = d.items;
    g.part = a.part;
  }
  g.wait_ns = a.wait_ns;
  const uint32_t idesc = idesc_f16(a.bf16, kBM * kGemmCG, kGemmBN, false, true);
  cudaError_t e = launch_persistent(DH_KERNEL, a.grid, pipe_threads(DhCfg::kEpiw),
                                    DhCfg::L::kSmemBytes, kGemmCG, stream, a.tmA, a.tmB, g, idesc,
                                    p, a.status);
  if (e != cudaSuccess || !split) return e;
  // add up the tail tiles' K segments and store them
  const int tile_m = kBM * kGemmCG;
  const int64_t threads = static_cast<int64_t>(d.tail) * tile_m * (DhCfg::kTileN / 32);
  const int blocks = static_cast<int>(std::min<int64_t>((threads + 255) / 256, 4096));
  dh_tail_sum_kernel<<<blocks, 256, 0, stream>>>(a.part, d.tail, d.split, d.full_tiles, g.n_tiles,
                                                 tile_m, DhCfg::kTileN, p);
  return cudaGetLastError();
}

cudaError_t launch_count_rows(const int64_t *row_idx, int64_t n, int64_t T, uint32_t *cnt,
                              int num_sms, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 4;
  if (blocks > cap) blocks = cap;
  count_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(row_idx, n, T, cnt);
  return cudaGetLastError();
}

cudaError_t launch_dw_gemm(const GemmArgs &a, cudaStream_t stream) {
  DwEpi::Params p;
  p.V = a.M;
  p.H = a.N;
  p.dW = a.dW;
  p.ld = a.ld_dw;
  p.accumulate = a.accumulate;
  p.v8 = (reinterpret_cast<uintptr_t>(a.dW) & 31u) == 0 && (a.ld_dw * 4) % 32 == 0;
  const uint32_t idesc = idesc_f16(a.bf16, kBM * kGemmCG, kGemmBN, true, true);
  GemmShape g = gemm_shape(a.M, a.N, a.K, DwCfg::kTileN);
  g.wait_ns = a.wait_ns;
  return launch_persistent(DW_KERNEL, a.grid, pipe_threads(DwCfg::kEpiw), DwCfg::L::kSmemBytes,
                           kGemmCG, stream, a.tmA, a.tmB, g, idesc, p, a.status);
}

}  // namespace flp
