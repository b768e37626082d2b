// api.cu -- host side of libfusedlogp: argument validation, workspace
// layout, the tiling planner, tensor-map construction and the C entry
// points declared in include/fusedlogp.h.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fusedlogp.h"
#include "launch.h"

namespace flp {
namespace {

thread_local char g_err[512] = "";
thread_local cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;
// Limit of the kernels' barrier waits for calls from this thread (0: the
// kernels' default); set by flp_set_wait_limit.
thread_local uint64_t g_wait_ns = 0;

// Records the measurement-hook events (if set) around the tensor-core work.
struct KernelEvents {
  cudaEvent_t before, after;
  KernelEvents() : before(g_ev_before), after(g_ev_after) { g_ev_before = g_ev_after = nullptr; }
  cudaError_t start(cudaStream_t s) const { return before ? cudaEventRecord(before, s) : cudaSuccess; }
  cudaError_t stop(cudaStream_t s) const { return after ? cudaEventRecord(after, s) : cudaSuccess; }
};

flp_status fail(flp_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

flp_status cuda_fail(cudaError_t e, const char *what) {
  return fail(FLP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Vocabulary splits per row tile: at most 64, or as many as give about
// kSplitItems work items when there are few row tiles (with one row tile,
// 64 splits would leave 12 of 76 CTA pairs idle in the HBM-bound regime).
constexpr int64_t kMaxSplits = 64;
constexpr int64_t kSplitItems = 320;
constexpr size_t kAlign = 1024;
constexpr size_t kStatusBytes = 256;
// Upper bound of the backward's logit-gradient chunk.
constexpr int64_t kGradChunkBytes = int64_t(4) << 30;
// L2 budget of one band's hidden rows.
constexpr int64_t kBandBytes = int64_t(48) << 20;
// Range of flp_set_wait_limit.
constexpr uint64_t kMinWaitNs = 100;
constexpr uint64_t kMaxWaitNs = 60000000000ull;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool shape_ok(const flp_shape *s, const char **why) {
  if (!s) return *why = "shape is NULL", false;
  if (s->T < 0 || s->H <= 0 || s->V <= 0 || s->n_rows < 0) return *why = "negative or zero size", false;
  if (s->dtype != FLP_BF16 && s->dtype != FLP_FP16) return *why = "dtype must be FLP_BF16 or FLP_FP16", false;
  if (s->H % 8 || s->ld_h % 8 || s->ld_w % 8) return *why = "H, ld_h and ld_w must be multiples of 8", false;
  if (s->ld_h < s->H || s->ld_w < s->H) return *why = "ld_h and ld_w must be >= H", false;
  // Tile coordinates and row indices inside the kernels are 32-bit.
  if (s->n_rows > (int64_t(1) << 30) || s->V > (int64_t(1) << 30) || s->H > (int64_t(1) << 24))
    return *why = "size beyond the 32-bit tiling range", false;
  return true;
}

int vocab_tiles(int64_t V, int bn) { return static_cast<int>(cdiv(V, bn)); }

int max_splits(int64_t V, int bn, int64_t n_rows, int bm) {
  const int64_t row_tiles = std::max<int64_t>(1, cdiv(n_rows, bm));
  const int64_t cap = std::max<int64_t>(kMaxSplits, cdiv(kSplitItems, row_tiles));
  return static_cast<int>(std::min<int64_t>(vocab_tiles(V, bn), cap));
}

// Rows of the backward's logit-gradient chunk: as many as fit in 4 GiB, or
// fewer if FLP_GRAD_CHUNK_ROWS asks for it (a memory/tuning knob).
int64_t grad_chunk_rows(const flp_shape *s) {
  const int64_t ldg = cdiv(s->V, 16) * 16;
  int64_t r = kGradChunkBytes / (ldg * 2);
  r = std::max<int64_t>(128, r / 128 * 128);
  if (const char *env = std::getenv("FLP_GRAD_CHUNK_ROWS")) {
    const long long want = std::atoll(env);
    if (want > 0) r = std::min<int64_t>(r, want);
  }
  return std::min<int64_t>(r, std::max<int64_t>(s->n_rows, 1));
}

struct Layout {
  size_t status = 0, cnt = 0, cnt_bytes = 0, zt = 0, pm = 0, ps = 0, pb = 0, pc = 0, pm2 = 0,
         ps2 = 0;
  size_t hs = 0, hs2 = 0, lse = 0, ez = 0, g = 0, rowcnt = 0, part = 0, total = 0;
  size_t q8 = 0, sfa = 0;  // block-scaled KL: teacher rows in MXFP8 and their scale atoms
  int64_t grad_rows = 0;
  int part_slots = 0;  // backward: 512 KB FP32 partial tiles of the dh GEMM's split tail
};

// Partial-tile slots the backward's workspace holds for the dh GEMM's split
// tail: none if V is too short to split (fewer than two segments of
// kDhSplitMinKb k-blocks), else as many as the chunk's tiles could use,
// at most kDhSplitSlots.
int dh_part_slots(const flp_shape *s, int64_t grad_rows) {
  const int64_t kb = cdiv(s->V, 64);
  if (kb < 2 * kDhSplitMinKb) return 0;
  const int64_t tiles = dh_gemm_tiles(static_cast<int>(grad_rows), static_cast<int>(s->H));
  return static_cast<int>(std::min<int64_t>(kDhSplitSlots, tiles * (kb / kDhSplitMinKb)));
}

// The dh GEMM's tail split is on unless FLP_DH_SPLIT=0 (a tuning knob, read
// at each call).
bool dh_split_enabled() {
  const char *env = std::getenv("FLP_DH_SPLIT");
  return !(env && env[0] == '0' && env[1] == '\0');
}

// gather = false: the scoring or KL call scores rows 0..T-1 in place
// (row_idx NULL) and needs no gathered rows; they are the layout's last
// blocks for those ops, so the other offsets do not move.
Layout layout_for(const flp_shape *s, flp_op op, bool gather = true) {
  Layout L;
  if (op == FLP_OP_BACKWARD) gather = true;
  const size_t n = static_cast<size_t>(s->n_rows);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  L.status = take(kStatusBytes);
  // one arrival counter per 32-row group (the fused merge), cleared per call;
  // groups are counted over whole 256-row tiles
  L.cnt_bytes = static_cast<size_t>(cdiv(s->n_rows, 256) * 8 + 8) * 4;
  L.cnt = take(L.cnt_bytes);
  // the backward's statistics pass is the forward kernel
  const bool kl = op == FLP_OP_KL || op == FLP_OP_KL_MX;
  const bool mx = op == FLP_OP_KL_MX || op == FLP_OP_LOGPROB_ENTROPY_MX;
  const int bn = op == FLP_OP_KL ? kKlBN
                 : op == FLP_OP_KL_MX ? kMxBN
                 : op == FLP_OP_LOGPROB_ENTROPY_MX ? kMxFwdTileCols
                 : kFwdTileCols;
  const int epiw = op == FLP_OP_KL ? kKlEpiWarps
                   : op == FLP_OP_KL_MX ? kMxEpiWarps
                   : op == FLP_OP_LOGPROB_ENTROPY_MX ? kMxFEpiWarps
                   : kFwdEpiWarps;
  const size_t sm = static_cast<size_t>(max_splits(s->V, bn, s->n_rows, 128 * kFwdCG)) * (epiw / 4);  // partial slots
  L.pm = take(sm * n * 4);
  L.ps = take(sm * n * 4);
  L.pb = take(sm * n * 4);
  if (kl) {
    L.pm2 = take(sm * n * 4);
    L.ps2 = take(sm * n * 4);
  } else {
    L.zt = take(n * kMaxTargets * 4);  // raw target logits, up to kMaxTargets per row
  }
  if (mx) {
    // the teacher's (KL) or the scored (forward) rows quantised per call:
    // E4M3 codes and 512-byte scale atoms per 128 rows and 128-wide k-chunk
    L.q8 = take(n * static_cast<size_t>(s->H));
    L.sfa = take(static_cast<size_t>(cdiv(s->n_rows, 128) * cdiv(s->H, kMxChunk)) * 512);
  }
  // the block-scaled forward has no bf16/fp16 operand: its quantiser gathers
  if (gather && op != FLP_OP_LOGPROB_ENTROPY_MX) {
    L.hs = take(n * static_cast<size_t>(s->H) * 2);
    if (op == FLP_OP_KL) L.hs2 = take(n * static_cast<size_t>(s->H) * 2);
  }
  if (op == FLP_OP_BACKWARD) {
    L.lse = take(n * 4);
    L.ez = take(n * 4);
    L.grad_rows = grad_chunk_rows(s);
    L.g = take(static_cast<size_t>(L.grad_rows) * static_cast<size_t>(cdiv(s->V, 16) * 16) * 2);
    L.rowcnt = take(static_cast<size_t>(s->T) * 4);  // scored rows per h row
    L.part_slots = dh_part_slots(s, L.grad_rows);
    L.part = take(static_cast<size_t>(L.part_slots) * kDhSlotBytes);
  }
  L.total = off;
  return L;
}

// ------------------------------------------------------------------ planner
struct PlanKey {
  int64_t n, V, H, band_bytes;
  int bn, units, bm, a_ops;
  bool operator<(const PlanKey &o) const {
    return std::tie(n, V, H, band_bytes, bn, units, bm, a_ops) <
           std::tie(o.n, o.V, o.H, o.band_bytes, o.bn, o.units, o.bm, o.a_ops);
  }
};

// L2 budget of one band's hidden rows (FLP_BAND_MB overrides it).
int64_t band_budget() {
  if (const char *env = std::getenv("FLP_BAND_MB")) {
    const long long mb = std::atoll(env);
    if (mb > 0) return static_cast<int64_t>(mb) << 20;
  }
  return kBandBytes;
}

// `units` = CTAs (or CTA pairs) resident at once; `grid` is in the same
// units (the kernel launch multiplies by the CTA-group size).
struct Plan {
  Schedule sch;
  int grid;
  int64_t max_load;
};

std::mutex g_plan_mu;
std::map<PlanKey, Plan> g_plans;

// a_ops = hidden-state operands per row tile (2 for the KL: student and teacher).
Plan make_plan(int64_t n, int64_t V, int64_t H, int bn, int num_sms, int bm, int64_t band_bytes,
               int a_ops) {
  Plan best{};
  Schedule s{};
  s.n = static_cast<int>(n);
  s.V = static_cast<int>(V);
  s.row_tiles = static_cast<int>(cdiv(n, bm));
  s.vocab_tiles = vocab_tiles(V, bn);
  s.k_blocks = static_cast<int>(cdiv(H, 64));
  const int64_t a_tile_bytes = static_cast<int64_t>(bm) * H * 2 * a_ops;
  s.band = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(s.row_tiles, band_bytes / a_tile_bytes)));
  const int smax = max_splits(V, bn, n, bm);
  std::vector<int64_t> loads;
  int64_t best_load = -1;
  for (int S = 1; S <= smax; ++S) {
    const int tps = static_cast<int>(cdiv(s.vocab_tiles, S));
    if (cdiv(s.vocab_tiles, tps) != S) continue;  // an equivalent, smaller S exists
    Schedule c = s;
    c.splits = S;
    c.tiles_per_split = tps;
    c.items = s.row_tiles * S;
    if (c.items > (1 << 22)) break;
    const int grid = std::min(c.items, num_sms);
    loads.assign(grid, 0);
    for (int it = 0; it < c.items; ++it) {
      int mt, sp, v0, v1;
      c.item(it, mt, sp, v0, v1);
      loads[it % grid] += v1 - v0;
    }
    const int64_t mk = *std::max_element(loads.begin(), loads.end());
    // Keep the smallest S whose makespan is within 0.5% of the best.
    if (best_load < 0 || mk * 1000 < best_load * 995) {
      best_load = mk;
      best.sch = c;
      best.grid = grid;
      best.max_load = mk;
    }
  }
  return best;
}

Plan plan_cached(int64_t n, int64_t V, int64_t H, int bn, int units, int bm, int a_ops = 1) {
  const int64_t band_bytes = band_budget();
  const PlanKey k{n, V, H, band_bytes, bn, units, bm, a_ops};
  std::lock_guard<std::mutex> g(g_plan_mu);
  auto it = g_plans.find(k);
  if (it != g_plans.end()) return it->second;
  if (g_plans.size() > 256) g_plans.clear();
  Plan p = make_plan(n, V, H, bn, units, bm, band_bytes, a_ops);
  g_plans.emplace(k, p);
  return p;
}

// ------------------------------------------------------------------ device
struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_devs;

flp_status device_info(DeviceInfo *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> g(g_dev_mu);
  auto it = g_devs.find(dev);
  if (it == g_devs.end()) {
    DeviceInfo d;
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.ok = (major == 10 && minor == 3);
    it = g_devs.emplace(dev, d).first;
  }
  if (!it->second.ok)
    return fail(FLP_ERR_UNSUPPORTED, "device %d is not compute capability 10.3 (sm_103a)", dev);
  *out = it->second;
  return FLP_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

flp_status get_encoder(EncodeTiledFn *out) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) return fail(FLP_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *out = fn;
  return FLP_OK;
}

// 2-D map over a row-major [outer, ld] matrix of 16-bit elements using
// `inner` columns; boxes of box_inner x box_outer, 128-byte swizzle.
flp_status make_map(CUtensorMap *m, flp_dtype dt, const void *base, int64_t inner, int64_t outer,
                    int64_t ld, int box_inner, int box_outer) {
  EncodeTiledFn enc;
  flp_status st = get_encoder(&enc);
  if (st != FLP_OK) return st;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, dt == FLP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FLP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return FLP_OK;
}

// 2-D map of any element type over `outer` rows of `inner` elements,
// `stride` bytes apart.
flp_status make_map_typed(CUtensorMap *m, CUtensorMapDataType type, const void *base, int64_t inner,
                          int64_t outer, int64_t stride, int box_inner, int box_outer,
                          CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc;
  flp_status st = get_encoder(&enc);
  if (st != FLP_OK) return st;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, type, 2, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FLP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d, type %d)", static_cast<int>(r),
                static_cast<int>(type));
  return FLP_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Block-scaled teacher head: the E2M1 codes [V, H/2], then (1 KiB aligned)
// the scale atoms, two of 512 B per 224-row vocabulary tile and 128-wide
// k-chunk.
size_t mx_head_code_bytes(int64_t V, int64_t H) {
  return align_up(static_cast<size_t>(V) * static_cast<size_t>(H / 2));
}
size_t mx_head_atom_bytes(int64_t V, int64_t H) {
  return static_cast<size_t>(cdiv(V, kMxBN)) * static_cast<size_t>(H / kMxChunk) * 1024;
}

flp_status check_common(const flp_shape *s, flp_op op, const void *ws, size_t ws_bytes,
                        bool gather = true) {
  const char *why = nullptr;
  if (!shape_ok(s, &why)) return fail(FLP_ERR_INVALID_ARG, "%s", why);
  if (!ws) return fail(FLP_ERR_WORKSPACE, "workspace is NULL");
  const size_t need = layout_for(s, op, gather).total;
  if (ws_bytes < need)
    return fail(FLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  if (reinterpret_cast<uintptr_t>(ws) % 256)
    return fail(FLP_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return FLP_OK;
}

template <class T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

// ---------------------------------------------------------------- static scratch
// Scratch of flp_logprob_entropy_noalloc: one array per device, sized at
// build time, so that entry point never allocates device memory.
static_assert(FLP_NOALLOC_SCRATCH_BYTES % kAlign == 0, "scratch size");
static __device__ __align__(256) unsigned char g_noalloc_scratch[FLP_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
std::map<unsigned long long, void *> g_scratch_addr;  // by CUDA context id

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Id of the CUDA context current on this thread (unique for the life of the
// process, so a context made after a reset gets a new one); false if there
// is none yet or the driver does not provide the query.
bool current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array in the current device's context.  It is
// looked up (cudaGetSymbolAddress, with that device current) once per
// context: normally once per device, and again after the device's context
// was reset, when the library's module is loaded anew and the array may sit
// elsewhere.
flp_status noalloc_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned long long ctx = 0;
  const bool keyed = current_context_id(&ctx);
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (keyed) {
    auto it = g_scratch_addr.find(ctx);
    if (it != g_scratch_addr.end()) {
      *out = it->second;
      return FLP_OK;
    }
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
  // the look-up makes the device's context current if it was not yet
  if (keyed || current_context_id(&ctx)) g_scratch_addr[ctx] = p;
  *out = p;
  return FLP_OK;
}

// Checks of a sampling-support argument (null = no support restriction).
flp_status check_support(const flp_shape *s, const uint32_t *support, int64_t ld_support) {
  if (!support) return FLP_OK;
  if (reinterpret_cast<uintptr_t>(support) % 4 != 0)
    return fail(FLP_ERR_INVALID_ARG, "support must be 4-byte aligned");
  if (ld_support < cdiv(s->V, 32))
    return fail(FLP_ERR_INVALID_ARG, "ld_support (%lld) < ceil(V / 32) (%lld)",
                static_cast<long long>(ld_support), static_cast<long long>(cdiv(s->V, 32)));
  return FLP_OK;
}

flp_status logprob_impl(const flp_shape *s, const void *h, const void *W, const int64_t *targets,
                        int K, const int64_t *row_idx, const uint32_t *support,
                        int64_t ld_support, float temperature, float *out_logp,
                        float *out_ent, float *out_lse, float *out_ez, void *ws, size_t ws_bytes,
                        flp_stream_t stream) {
  g_err[0] = 0;
  const KernelEvents ev;
  flp_status st = check_common(s, FLP_OP_LOGPROB_ENTROPY, ws, ws_bytes, row_idx != nullptr);
  if (st != FLP_OK) return st;
  if (!(std::isfinite(temperature) && temperature > 0.f))
    return fail(FLP_ERR_INVALID_ARG, "temperature must be finite and > 0");
  if (K < 1 || K > kMaxTargets)
    return fail(FLP_ERR_INVALID_ARG, "K must be within 1 .. %d", kMaxTargets);
  if (s->n_rows == 0) return FLP_OK;
  if (!row_idx && s->n_rows != s->T)
    return fail(FLP_ERR_INVALID_ARG, "row_idx is NULL but n_rows != T");
  if (!h || !W || !targets || !out_logp || !out_ent)
    return fail(FLP_ERR_INVALID_ARG, "h, W, targets, out_logp and out_ent are required");
  if (!aligned16(h) || !aligned16(W)) return fail(FLP_ERR_INVALID_ARG, "h and W must be 16-byte aligned");
  if ((st = check_support(s, support, ld_support)) != FLP_OK) return st;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FLP_OK) return st;

  const Layout L = layout_for(s, FLP_OP_LOGPROB_ENTROPY, row_idx != nullptr);
  // few rows: single CTAs on 128-row tiles (the workspace's partial slots
  // cover this plan too: twice the columns' worth of splits per row)
  const bool few = s->n_rows <= kSmallRows;
  const int cg = few ? 1 : kFwdCG;
  const Plan p = few ? plan_cached(s->n_rows, s->V, s->H, kFwdBN, fwd1_units(dev.sms), 128)
                     : plan_cached(s->n_rows, s->V, s->H, kFwdTileCols, fwd_units(dev.sms), 128 * kFwdCG);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  FwdArgs a{};
  const void *A = h;
  int64_t lda = s->ld_h;
  if (row_idx) {
    A = at<void>(ws, L.hs);
    lda = s->H;
  }
  if ((st = make_map(&a.tmA, s->dtype, A, s->H, s->n_rows, lda, 64, 128)) != FLP_OK) return st;
  if ((st = make_map(&a.tmB, s->dtype, W, s->H, s->V, s->ld_w, 64, kFwdBN / cg)) != FLP_OK)
    return st;
  a.sch = p.sch;
  a.sch.wait_ns = g_wait_ns;
  a.grid = p.grid * cg;
  a.bf16 = s->dtype == FLP_BF16;
  a.targets = targets;
  a.K = K;
  a.row_idx = row_idx;
  a.T = s->T;
  a.inv_tau = 1.0f / temperature;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  a.pm = at<float>(ws, L.pm);
  a.ps = at<float>(ws, L.ps);
  a.pb = at<float>(ws, L.pb);
  a.zt = at<float>(ws, L.zt);
  a.counters = at<uint32_t>(ws, L.cnt);
  a.out_logp = out_logp;
  a.out_ent = out_ent;
  a.out_lse = out_lse;
  a.out_ez = out_ez;
  a.status = at<uint32_t>(ws, L.status);
  a.support = support;
  a.ld_support = ld_support;

  // status words and row-group counters are adjacent: one clear
  cudaError_t e = cudaMemsetAsync(a.status, 0, L.cnt + L.cnt_bytes - L.status, cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  if (row_idx) {
    e = launch_gather(h, s->ld_h, row_idx, s->n_rows, s->T, s->H, at<void>(ws, L.hs), dev.sms, cs);
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  }
  if ((e = ev.start(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  e = few ? launch_fwd_scoring_1cta(a, cs) : launch_fwd_scoring(a, cs);
  if (e != cudaSuccess) return cuda_fail(e, "scoring launch");
  if ((e = ev.stop(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  return FLP_OK;
}

// KL(teacher || student); the teacher head is W_t, or (mx.packed != null)
// the blocked MXFP4 operand mx.
flp_status kl_impl(const flp_shape *s, const void *h_s, const void *W_s, const void *h_t,
                   const void *W_t, const MxOperand &mx, const int64_t *row_idx, float *out_kl,
                   void *ws, size_t ws_bytes, flp_stream_t stream) {
  const KernelEvents ev;
  flp_status st = check_common(s, FLP_OP_KL, ws, ws_bytes, row_idx != nullptr);
  if (st != FLP_OK) return st;
  if (s->n_rows == 0) return FLP_OK;
  if (!row_idx && s->n_rows != s->T)
    return fail(FLP_ERR_INVALID_ARG, "row_idx is NULL but n_rows != T");
  if (!h_s || !W_s || !h_t || !(W_t || mx.packed) || !out_kl)
    return fail(FLP_ERR_INVALID_ARG, "h_s, W_s, h_t, the teacher head and out_kl are required");
  if (!aligned16(h_s) || !aligned16(W_s) || !aligned16(h_t) || (W_t && !aligned16(W_t)))
    return fail(FLP_ERR_INVALID_ARG, "h_s, W_s, h_t and W_t must be 16-byte aligned");
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FLP_OK) return st;

  const Layout L = layout_for(s, FLP_OP_KL, row_idx != nullptr);
  const int units = mx.packed ? kl_mx_units(dev.sms) : kl_units(dev.sms);
  const Plan p = plan_cached(s->n_rows, s->V, s->H, kKlBN, units, 128 * kKlCG, 2);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  KlArgs a{};
  const void *As = h_s, *At = h_t;
  int64_t lda = s->ld_h;
  if (row_idx) {
    As = at<void>(ws, L.hs);
    At = at<void>(ws, L.hs2);
    lda = s->H;
  }
  if ((st = make_map(&a.tmAs, s->dtype, As, s->H, s->n_rows, lda, 64, 128)) != FLP_OK) return st;
  if ((st = make_map(&a.tmAt, s->dtype, At, s->H, s->n_rows, lda, 64, 128)) != FLP_OK) return st;
  if ((st = make_map(&a.tmBs, s->dtype, W_s, s->H, s->V, s->ld_w, 64, kKlBN / kKlCG)) != FLP_OK)
    return st;
  if (W_t && (st = make_map(&a.tmBt, s->dtype, W_t, s->H, s->V, s->ld_w, 64, kKlBN / kKlCG)) !=
                 FLP_OK)
    return st;
  a.mx = mx;
  a.sch = p.sch;
  a.sch.wait_ns = g_wait_ns;
  a.grid = p.grid * kKlCG;
  a.bf16 = s->dtype == FLP_BF16;
  a.row_idx = row_idx;
  a.T = s->T;
  a.pmt = at<float>(ws, L.pm);
  a.pst = at<float>(ws, L.ps);
  a.pct = at<float>(ws, L.pb);
  a.pms = at<float>(ws, L.pm2);
  a.pss = at<float>(ws, L.ps2);
  a.counters = at<uint32_t>(ws, L.cnt);
  a.out_kl = out_kl;
  a.status = at<uint32_t>(ws, L.status);

  cudaError_t e = cudaMemsetAsync(a.status, 0, L.cnt + L.cnt_bytes - L.status, cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  if (row_idx) {
    e = launch_gather(h_s, s->ld_h, row_idx, s->n_rows, s->T, s->H, at<void>(ws, L.hs), dev.sms, cs);
    if (e == cudaSuccess)
      e = launch_gather(h_t, s->ld_h, row_idx, s->n_rows, s->T, s->H, at<void>(ws, L.hs2), dev.sms, cs);
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  }
  if ((e = ev.start(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  if ((e = launch_kl(a, cs)) != cudaSuccess) return cuda_fail(e, "KL launch");
  if ((e = ev.stop(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  return FLP_OK;
}

// KL(teacher || student) with the teacher on the block-scaled tensor cores:
// the scored teacher rows are quantised to MXFP8 in the workspace, then one
// persistent launch forms both heads' logit tiles and folds them.
flp_status kl_bs_impl(const flp_shape *s, const void *h_s, const void *W_s, const void *h_t,
                      const void *head, const int64_t *row_idx, float *out_kl, void *ws,
                      size_t ws_bytes, flp_stream_t stream) {
  const KernelEvents ev;
  flp_status st = check_common(s, FLP_OP_KL_MX, ws, ws_bytes, row_idx != nullptr);
  if (st != FLP_OK) return st;
  if (s->H % kMxChunk != 0)
    return fail(FLP_ERR_INVALID_ARG, "H must be a multiple of 128 for the block-scaled teacher");
  // the scale atoms are addressed by 32-bit tensor-map row coordinates
  if (cdiv(s->V, kMxBN) * (s->H / kMxChunk) * 64 > (int64_t(1) << 31) - 64 ||
      cdiv(s->n_rows, 128) * (s->H / kMxChunk) * 32 > (int64_t(1) << 31) - 32)
    return fail(FLP_ERR_INVALID_ARG, "size beyond the block-scaled tiling range");
  if (s->n_rows == 0) return FLP_OK;
  if (!row_idx && s->n_rows != s->T)
    return fail(FLP_ERR_INVALID_ARG, "row_idx is NULL but n_rows != T");
  if (!h_s || !W_s || !h_t || !head || !out_kl)
    return fail(FLP_ERR_INVALID_ARG, "h_s, W_s, h_t, the teacher head and out_kl are required");
  if (!aligned16(h_s) || !aligned16(W_s) || !aligned16(h_t))
    return fail(FLP_ERR_INVALID_ARG, "h_s, W_s and h_t must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(head) % 256 != 0)
    return fail(FLP_ERR_INVALID_ARG, "the teacher head must be 256-byte aligned");
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FLP_OK) return st;

  const Layout L = layout_for(s, FLP_OP_KL_MX, row_idx != nullptr);
  const Plan p = plan_cached(s->n_rows, s->V, s->H, kMxBN, kl_bs_units(dev.sms), 256, 2);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int64_t kc = s->H / kMxChunk;
  KlBsArgs a{};
  const void *As = h_s;
  int64_t lda = s->ld_h;
  if (row_idx) {
    As = at<void>(ws, L.hs);
    lda = s->H;
  }
  uint8_t *q8 = at<uint8_t>(ws, L.q8), *sfa = at<uint8_t>(ws, L.sfa);
  const uint8_t *codes = static_cast<const uint8_t *>(head);
  const uint8_t *atoms = codes + mx_head_code_bytes(s->V, s->H);
  if ((st = make_map(&a.tmAs, s->dtype, As, s->H, s->n_rows, lda, 64, 128)) != FLP_OK) return st;
  if ((st = make_map(&a.tmBs, s->dtype, W_s, s->H, s->V, s->ld_w, 64, kMxBN / 2)) != FLP_OK)
    return st;
  if ((st = make_map_typed(&a.tmAt, CU_TENSOR_MAP_DATA_TYPE_UINT8, q8, s->H, s->n_rows, s->H,
                           kMxChunk, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != FLP_OK)
    return st;
  if ((st = make_map_typed(&a.tmBt, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, codes, s->H, s->V,
                           s->H / 2, kMxChunk, kMxBN / 2, CU_TENSOR_MAP_SWIZZLE_128B)) != FLP_OK)
    return st;
  if ((st = make_map_typed(&a.tmSfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, sfa, 16,
                           cdiv(s->n_rows, 128) * kc * 32, 16, 16, 32,
                           CU_TENSOR_MAP_SWIZZLE_NONE)) != FLP_OK)
    return st;
  if ((st = make_map_typed(&a.tmSfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, atoms, 16,
                           cdiv(s->V, kMxBN) * kc * 64, 16, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      FLP_OK)
    return st;
  a.sch = p.sch;
  a.sch.k_blocks = static_cast<int>(kc);
  a.sch.wait_ns = g_wait_ns;
  a.grid = p.grid * 2;
  a.bf16 = s->dtype == FLP_BF16;
  a.row_idx = row_idx;
  a.T = s->T;
  a.pmt = at<float>(ws, L.pm);
  a.pst = at<float>(ws, L.ps);
  a.pct = at<float>(ws, L.pb);
  a.pms = at<float>(ws, L.pm2);
  a.pss = at<float>(ws, L.ps2);
  a.counters = at<uint32_t>(ws, L.cnt);
  a.out_kl = out_kl;
  a.status = at<uint32_t>(ws, L.status);

  cudaError_t e = cudaMemsetAsync(a.status, 0, L.cnt + L.cnt_bytes - L.status, cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  if (row_idx &&
      (e = launch_gather(h_s, s->ld_h, row_idx, s->n_rows, s->T, s->H, at<void>(ws, L.hs), dev.sms,
                         cs)) != cudaSuccess)
    return cuda_fail(e, "gather launch");
  if ((e = launch_mxfp8_quantize(h_t, a.bf16, s->n_rows, s->H, s->ld_h, row_idx, s->T, q8, sfa,
                                 true, dev.sms, cs)) != cudaSuccess)
    return cuda_fail(e, "MXFP8 quantize launch");
  if ((e = ev.start(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  if ((e = launch_kl_blockscaled(a, cs)) != cudaSuccess) return cuda_fail(e, "block-scaled KL launch");
  if ((e = ev.stop(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  return FLP_OK;
}

// Log-prob and entropy with the logits on the block-scaled tensor cores: the
// scored rows are quantised to MXFP8 in the workspace (gathered on the way),
// then one persistent launch forms the logit tiles against the MXFP4 head
// and folds them.
flp_status fwd_bs_impl(const flp_shape *s, const void *h, const void *head,
                       const int64_t *targets, const int64_t *row_idx, float temperature,
                       float *out_logp, float *out_ent, float *out_lse, float *out_ez, void *ws,
                       size_t ws_bytes, flp_stream_t stream) {
  const KernelEvents ev;
  flp_status st = check_common(s, FLP_OP_LOGPROB_ENTROPY_MX, ws, ws_bytes, false);
  if (st != FLP_OK) return st;
  if (s->H % kMxChunk != 0)
    return fail(FLP_ERR_INVALID_ARG, "H must be a multiple of 128 for the block-scaled forward");
  if (!(std::isfinite(temperature) && temperature > 0.f))
    return fail(FLP_ERR_INVALID_ARG, "temperature must be finite and > 0");
  // the scale atoms are addressed by 32-bit tensor-map row coordinates (the
  // last tile may name one head tile past the end)
  if ((cdiv(s->V, kMxBN) + 1) * (s->H / kMxChunk) * 64 > (int64_t(1) << 31) - 64 ||
      cdiv(s->n_rows, 128) * (s->H / kMxChunk) * 32 > (int64_t(1) << 31) - 32)
    return fail(FLP_ERR_INVALID_ARG, "size beyond the block-scaled tiling range");
  if (s->n_rows == 0) return FLP_OK;
  if (!row_idx && s->n_rows != s->T)
    return fail(FLP_ERR_INVALID_ARG, "row_idx is NULL but n_rows != T");
  if (!h || !head || !targets || !out_logp || !out_ent)
    return fail(FLP_ERR_INVALID_ARG, "h, head, targets, out_logp and out_ent are required");
  if (!aligned16(h)) return fail(FLP_ERR_INVALID_ARG, "h must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(head) % 256 != 0)
    return fail(FLP_ERR_INVALID_ARG, "the head must be 256-byte aligned");
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FLP_OK) return st;

  const Layout L = layout_for(s, FLP_OP_LOGPROB_ENTROPY_MX, false);
  const Plan p = plan_cached(s->n_rows, s->V, s->H, kMxFwdTileCols, fwd_bs_units(dev.sms), 256);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int64_t kc = s->H / kMxChunk;
  FwdBsArgs a{};
  uint8_t *q8 = at<uint8_t>(ws, L.q8), *sfa = at<uint8_t>(ws, L.sfa);
  const uint8_t *codes = static_cast<const uint8_t *>(head);
  const uint8_t *atoms = codes + mx_head_code_bytes(s->V, s->H);
  if ((st = make_map_typed(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, q8, s->H, s->n_rows, s->H,
                           kMxChunk, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != FLP_OK)
    return st;
  if ((st = make_map_typed(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, codes, s->H, s->V,
                           s->H / 2, kMxChunk, kMxBN / 2, CU_TENSOR_MAP_SWIZZLE_128B)) != FLP_OK)
    return st;
  if ((st = make_map_typed(&a.tmSfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, sfa, 16,
                           cdiv(s->n_rows, 128) * kc * 32, 16, 16, 32,
                           CU_TENSOR_MAP_SWIZZLE_NONE)) != FLP_OK)
    return st;
  if ((st = make_map_typed(&a.tmSfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, atoms, 16,
                           cdiv(s->V, kMxBN) * kc * 64, 16, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      FLP_OK)
    return st;
  a.sch = p.sch;
  a.sch.k_blocks = static_cast<int>(kc);
  a.sch.wait_ns = g_wait_ns;
  a.grid = p.grid * 2;
  a.targets = targets;
  a.row_idx = row_idx;
  a.T = s->T;
  a.inv_tau = 1.0f / temperature;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  a.pm = at<float>(ws, L.pm);
  a.ps = at<float>(ws, L.ps);
  a.pb = at<float>(ws, L.pb);
  a.zt = at<float>(ws, L.zt);
  a.counters = at<uint32_t>(ws, L.cnt);
  a.out_logp = out_logp;
  a.out_ent = out_ent;
  a.out_lse = out_lse;
  a.out_ez = out_ez;
  a.status = at<uint32_t>(ws, L.status);

  cudaError_t e = cudaMemsetAsync(a.status, 0, L.cnt + L.cnt_bytes - L.status, cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  if ((e = launch_mxfp8_quantize(h, s->dtype == FLP_BF16, s->n_rows, s->H, s->ld_h, row_idx, s->T,
                                 q8, sfa, true, dev.sms, cs)) != cudaSuccess)
    return cuda_fail(e, "MXFP8 quantize launch");
  if ((e = ev.start(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  if ((e = launch_fwd_blockscaled(a, cs)) != cudaSuccess)
    return cuda_fail(e, "block-scaled scoring launch");
  if ((e = ev.stop(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  return FLP_OK;
}

flp_status backward_impl(const flp_shape *s, const void *h, const void *W, const int64_t *targets,
                         const int64_t *row_idx, const uint32_t *support, int64_t ld_support,
                         float temperature, const float *g1, const float *g2, const float *lse,
                         const float *ez, void *dh, float *dW, void *ws, size_t ws_bytes,
                         flp_stream_t stream) {
  g_err[0] = 0;
  const KernelEvents ev;
  flp_status st = check_common(s, FLP_OP_BACKWARD, ws, ws_bytes);
  if (st != FLP_OK) return st;
  if (!(std::isfinite(temperature) && temperature > 0.f))
    return fail(FLP_ERR_INVALID_ARG, "temperature must be finite and > 0");
  if (!dh && !dW) return fail(FLP_ERR_INVALID_ARG, "dh and dW are both NULL: nothing to compute");
  if ((dh && !aligned16(dh)) || (dW && !aligned16(dW)))
    return fail(FLP_ERR_INVALID_ARG, "dh and dW must be 16-byte aligned");
  if ((lse == nullptr) != (ez == nullptr))
    return fail(FLP_ERR_INVALID_ARG, "lse and ez must both be given or both be NULL");
  if (s->n_rows > 0) {
    if (!h || !W || !targets || !g1 || !g2)
      return fail(FLP_ERR_INVALID_ARG, "h, W, targets, g1 and g2 are required");
    if (!aligned16(h) || !aligned16(W)) return fail(FLP_ERR_INVALID_ARG, "h and W must be 16-byte aligned");
    if (!row_idx && s->n_rows != s->T)
      return fail(FLP_ERR_INVALID_ARG, "row_idx is NULL but n_rows != T");
    if ((st = check_support(s, support, ld_support)) != FLP_OK) return st;
  }
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FLP_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const Layout L = layout_for(s, FLP_OP_BACKWARD);
  uint32_t *status = at<uint32_t>(ws, L.status);
  const size_t esz = 2;
  cudaError_t e = cudaMemsetAsync(status, 0, L.cnt + L.cnt_bytes - L.status, cs);
  // rows that are not scored get a zero gradient
  if (e == cudaSuccess && dh && s->T > 0)
    e = cudaMemset2DAsync(dh, s->ld_h * esz, 0, s->H * esz, s->T, cs);
  if (e == cudaSuccess && dW && s->n_rows == 0)
    e = cudaMemset2DAsync(dW, s->ld_w * 4, 0, s->H * 4, s->V, cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  if (s->n_rows == 0) return FLP_OK;

  const void *A = h;
  int64_t lda = s->ld_h;
  uint32_t *rowcnt = nullptr;
  if (row_idx) {
    A = at<void>(ws, L.hs);
    lda = s->H;
    e = launch_gather(h, s->ld_h, row_idx, s->n_rows, s->T, s->H, at<void>(ws, L.hs), dev.sms, cs);
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
    if (dh) {
        // rows named more than once have their dh contributions summed
        rowcnt = at<uint32_t>(ws, L.rowcnt);
        e = cudaMemsetAsync(rowcnt, 0, static_cast<size_t>(s->T) * 4, cs);
        if (e == cudaSuccess) e = launch_count_rows(row_idx, s->n_rows, s->T, rowcnt, dev.sms, cs);
        if (e != cudaSuccess) return cuda_fail(e, "row count");
    }
  }
  const float inv_tau = 1.0f / temperature;
  const float sl = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  if ((e = ev.start(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");

  // Per-row statistics (LSE, E[z']) unless the caller kept them from the forward.
  if (!lse) {
    FwdArgs a{};
    const Plan p = plan_cached(s->n_rows, s->V, s->H, kFwdTileCols, fwd_units(dev.sms), 128 * kFwdCG);
    if ((st = make_map(&a.tmA, s->dtype, A, s->H, s->n_rows, lda, 64, 128)) != FLP_OK) return st;
    if ((st = make_map(&a.tmB, s->dtype, W, s->H, s->V, s->ld_w, 64, kFwdBN / kFwdCG)) != FLP_OK)
      return st;
    a.sch = p.sch;
    a.sch.wait_ns = g_wait_ns;
    a.grid = p.grid * kFwdCG;
    a.bf16 = s->dtype == FLP_BF16;
    a.targets = targets;
    a.K = 1;
    a.row_idx = row_idx;
    a.T = s->T;
    a.inv_tau = inv_tau;
    a.scale_log2 = sl;
    a.pm = at<float>(ws, L.pm);
    a.ps = at<float>(ws, L.ps);
    a.pb = at<float>(ws, L.pb);
    a.zt = at<float>(ws, L.zt);
    a.counters = at<uint32_t>(ws, L.cnt);
    a.out_lse = at<float>(ws, L.lse);
    a.out_ez = at<float>(ws, L.ez);
    a.status = status;
    a.support = support;
    a.ld_support = ld_support;
    if ((e = launch_fwd_scoring(a, cs)) != cudaSuccess) return cuda_fail(e, "stats launch");
    lse = a.out_lse;
    ez = a.out_ez;
  }

  const int64_t ldg = cdiv(s->V, 16) * 16;
  void *G = at<void>(ws, L.g);
  const int64_t n = s->n_rows;
  const int64_t num = (n - 1) / L.grad_rows + 1;
  const int64_t each = cdiv(n, num);
  const char *eb = static_cast<const char *>(A);
  for (int64_t r0 = 0; r0 < n; r0 += each) {
    const int rc = static_cast<int>(std::min(each, n - r0));
    const void *Ar = eb + static_cast<size_t>(r0) * lda * esz;
    // 1. G = d loss / d z for the chunk's rows
    GradArgs ga{};
    const Plan p = plan_cached(rc, s->V, s->H, kGradTileCols, grad_units(dev.sms), 128 * kGradCG);
    if ((st = make_map(&ga.tmA, s->dtype, Ar, s->H, rc, lda, 64, 128)) != FLP_OK) return st;
    if ((st = make_map(&ga.tmB, s->dtype, W, s->H, s->V, s->ld_w, 64, kGradBN / kGradCG)) != FLP_OK)
      return st;
    ga.sch = p.sch;
    ga.sch.wait_ns = g_wait_ns;
    ga.grid = p.grid * kGradCG;
    ga.bf16 = s->dtype == FLP_BF16;
    ga.r0 = static_cast<int>(r0);
    ga.T = s->T;
    ga.targets = targets;
    ga.row_idx = row_idx;
    ga.lse = lse;
    ga.ez = ez;
    ga.g1 = g1;
    ga.g2 = g2;
    ga.scale_log2 = sl;
    ga.inv_tau = inv_tau;
    ga.G = G;
    ga.ldg = ldg;
    ga.status = status;
    ga.support = support;
    ga.ld_support = ld_support;
    if ((e = launch_grad(ga, cs)) != cudaSuccess) return cuda_fail(e, "grad launch");
    // 2. dh[rows] = G W   (M = rc, N = H, K = V; W is MN-major for this product)
    if (dh) {
      GemmArgs da{};
      if ((st = make_map(&da.tmA, s->dtype, G, s->V, rc, ldg, 64, 128)) != FLP_OK) return st;
      if ((st = make_map(&da.tmB, s->dtype, W, s->H, s->V, s->ld_w, 64, 64)) != FLP_OK) return st;
      da.M = rc;
      da.N = static_cast<int>(s->H);
      da.K = static_cast<int>(s->V);
      const int units = gemm_units(dev.sms);
      da.dh_split = dh_split_plan(da.M, da.N, da.K, units, dh_split_enabled() ? L.part_slots : 0);
      da.part = at<float>(ws, L.part);
      da.grid = gemm_cta_group() * std::min(da.dh_split.items, units);
      da.bf16 = ga.bf16;
      da.status = status;
      da.r0 = static_cast<int>(r0);
      da.T = s->T;
      da.row_idx = row_idx;
      da.rowcnt = rowcnt;
      da.dh = dh;
      da.ld_dh = s->ld_h;
      da.wait_ns = g_wait_ns;
      if ((e = launch_dh_gemm(da, cs)) != cudaSuccess) return cuda_fail(e, "dh launch");
    }
    // 3. dW (+)= G^T h[rows]   (M = V, N = H, K = rc; both operands MN-major)
    if (dW) {
      GemmArgs wa{};
      if ((st = make_map(&wa.tmA, s->dtype, G, s->V, rc, ldg, 64, 64)) != FLP_OK) return st;
      if ((st = make_map(&wa.tmB, s->dtype, Ar, s->H, rc, lda, 64, 64)) != FLP_OK) return st;
      wa.M = static_cast<int>(s->V);
      wa.N = static_cast<int>(s->H);
      wa.K = rc;
      wa.grid = gemm_cta_group() * std::min(dw_gemm_tiles(wa.M, wa.N), gemm_units(dev.sms));
      wa.bf16 = ga.bf16;
      wa.status = status;
      wa.dW = dW;
      wa.ld_dw = s->ld_w;
      wa.accumulate = r0 > 0;
      wa.wait_ns = g_wait_ns;
      if ((e = launch_dw_gemm(wa, cs)) != cudaSuccess) return cuda_fail(e, "dW launch");
    }
  }
  if ((e = ev.stop(cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  return FLP_OK;
}

}  // namespace
}  // namespace flp

using namespace flp;

extern "C" {

size_t flp_workspace_size(const flp_shape *shape, flp_op op) {
  const char *why = nullptr;
  if (!shape_ok(shape, &why)) return 0;
  if (op != FLP_OP_LOGPROB_ENTROPY && op != FLP_OP_KL && op != FLP_OP_BACKWARD &&
      op != FLP_OP_KL_MX && op != FLP_OP_LOGPROB_ENTROPY_MX)
    return 0;
  if ((op == FLP_OP_KL_MX || op == FLP_OP_LOGPROB_ENTROPY_MX) && shape->H % kMxChunk != 0) return 0;
  return layout_for(shape, op).total;
}

const char *flp_status_string(flp_status s) {
  switch (s) {
    case FLP_OK: return "ok";
    case FLP_ERR_INVALID_ARG: return "invalid argument";
    case FLP_ERR_UNSUPPORTED: return "unsupported device or input combination";
    case FLP_ERR_WORKSPACE: return "workspace missing or too small";
    case FLP_ERR_CUDA: return "CUDA error";
    case FLP_ERR_DEVICE_STATUS: return "the device recorded a problem";
  }
  return "unknown status";
}

const char *flp_last_error(void) { return g_err; }

flp_status flp_set_wait_limit(uint64_t limit_ns) {
  g_err[0] = 0;
  if (limit_ns != 0 && (limit_ns < kMinWaitNs || limit_ns > kMaxWaitNs))
    return fail(FLP_ERR_INVALID_ARG, "limit_ns must be 0 or within %llu .. %llu",
                static_cast<unsigned long long>(kMinWaitNs),
                static_cast<unsigned long long>(kMaxWaitNs));
  g_wait_ns = limit_ns;
  return FLP_OK;
}

flp_status flp_set_kernel_events(void *before, void *after) {
  g_ev_before = static_cast<cudaEvent_t>(before);
  g_ev_after = static_cast<cudaEvent_t>(after);
  return FLP_OK;
}

flp_status flp_plan_scoring(const flp_shape *shape, flp_op op, int32_t num_sms, flp_plan *out) {
  const char *why = nullptr;
  if (!shape_ok(shape, &why)) return fail(FLP_ERR_INVALID_ARG, "%s", why);
  if (!out || num_sms <= 0) return fail(FLP_ERR_INVALID_ARG, "out is NULL or num_sms <= 0");
  if (op != FLP_OP_LOGPROB_ENTROPY && op != FLP_OP_KL && op != FLP_OP_BACKWARD &&
      op != FLP_OP_KL_MX && op != FLP_OP_LOGPROB_ENTROPY_MX)
    return fail(FLP_ERR_INVALID_ARG, "unknown op");
  std::memset(out, 0, sizeof *out);
  if (shape->n_rows == 0) return FLP_OK;
  // the forward's few-rows path runs single CTAs
  const bool few = op == FLP_OP_LOGPROB_ENTROPY && shape->n_rows <= kSmallRows;
  const bool kl = op == FLP_OP_KL || op == FLP_OP_KL_MX;
  const int bn = op == FLP_OP_KL                    ? kKlBN
                 : op == FLP_OP_KL_MX               ? kMxBN
                 : op == FLP_OP_LOGPROB_ENTROPY_MX  ? kMxFwdTileCols
                 : few                              ? kFwdBN
                                                    : kFwdTileCols;
  const int cg = kl || op == FLP_OP_LOGPROB_ENTROPY_MX ? 2 : (few ? 1 : kFwdCG);
  const int units = std::max(1, num_sms / cg);
  const Plan p = plan_cached(shape->n_rows, shape->V, shape->H, bn, units, 128 * cg, kl ? 2 : 1);
  out->row_tiles = p.sch.row_tiles;
  out->vocab_tiles = p.sch.vocab_tiles;
  out->block_m = 128 * cg;
  out->block_n = bn;
  out->cta_group = cg;
  out->splits = p.sch.splits;
  out->tiles_per_split = p.sch.tiles_per_split;
  out->band = p.sch.band;
  out->items = p.sch.items;
  out->grid = p.grid * cg;
  out->max_tiles_per_cta = p.max_load;
  out->dh_split = 1;
  if (op == FLP_OP_BACKWARD) {
    out->chunk_rows = grad_chunk_rows(shape);
    // rows of the first chunk (the chunk rule of flp_row_chunks)
    const int64_t first = cdiv(shape->n_rows, (shape->n_rows - 1) / out->chunk_rows + 1);
    const DhSplit d = dh_split_plan(static_cast<int>(first), static_cast<int>(shape->H),
                                    static_cast<int>(shape->V), std::max(1, num_sms / gemm_cta_group()),
                                    dh_split_enabled() ? dh_part_slots(shape, out->chunk_rows) : 0);
    out->dh_split = d.split;
    out->dh_tail_tiles = d.split > 1 ? d.tail : 0;
  }
  return FLP_OK;
}

int64_t flp_row_chunks(int64_t n_rows, int64_t chunk_rows, int64_t *out_lengths, int64_t max_out) {
  if (n_rows <= 0 || chunk_rows <= 0) return 0;
  const int64_t num = (n_rows - 1) / chunk_rows + 1;
  const int64_t each = cdiv(n_rows, num);
  int64_t k = 0;
  for (int64_t start = 0; start < n_rows; start += each, ++k)
    if (out_lengths && k < max_out) out_lengths[k] = std::min(each, n_rows - start);
  return k;
}

flp_status flp_logprob_entropy(const flp_shape *s, const void *h, const void *W,
                               const int64_t *targets, const int64_t *row_idx, float temperature,
                               float *out_logp, float *out_ent, float *out_lse, float *out_ez,
                               void *ws, size_t ws_bytes, flp_stream_t stream) {
  return logprob_impl(s, h, W, targets, 1, row_idx, nullptr, 0, temperature, out_logp, out_ent,
                      out_lse, out_ez, ws, ws_bytes, stream);
}

flp_status flp_logprob_entropy_support(const flp_shape *s, const void *h, const void *W,
                                       const int64_t *targets, const int64_t *row_idx,
                                       const uint32_t *support, int64_t ld_support,
                                       float temperature, float *out_logp, float *out_ent,
                                       float *out_lse, float *out_ez, void *ws, size_t ws_bytes,
                                       flp_stream_t stream) {
  g_err[0] = 0;
  if (!support) return fail(FLP_ERR_INVALID_ARG, "support is required");
  return logprob_impl(s, h, W, targets, 1, row_idx, support, ld_support, temperature, out_logp,
                      out_ent, out_lse, out_ez, ws, ws_bytes, stream);
}

flp_status flp_logprob_entropy_k(const flp_shape *s, const void *h, const void *W,
                                 const int64_t *targets, int32_t K, const int64_t *row_idx,
                                 float temperature, float *out_logp, float *out_ent,
                                 float *out_lse, float *out_ez, void *ws, size_t ws_bytes,
                                 flp_stream_t stream) {
  return logprob_impl(s, h, W, targets, K, row_idx, nullptr, 0, temperature, out_logp, out_ent,
                      out_lse, out_ez, ws, ws_bytes, stream);
}


flp_status flp_kl(const flp_shape *s, const void *h_s, const void *W_s, const void *h_t,
                  const void *W_t, const int64_t *row_idx, float *out_kl, void *ws,
                  size_t ws_bytes, flp_stream_t stream) {
  g_err[0] = 0;
  if (!W_t && s && s->n_rows > 0) return fail(FLP_ERR_INVALID_ARG, "W_t is required");
  return kl_impl(s, h_s, W_s, h_t, W_t, MxOperand{nullptr, nullptr, 0}, row_idx, out_kl, ws,
                 ws_bytes, stream);
}

int64_t flp_mxfp4_rows(int64_t V) { return V <= 0 ? 0 : cdiv(V, 256) * 256; }

size_t flp_mxfp4_bytes(int64_t V, int64_t H, size_t *packed_bytes, size_t *scale_bytes) {
  if (V <= 0 || H <= 0 || H % 64 != 0) return 0;
  const size_t rows = static_cast<size_t>(flp_mxfp4_rows(V));
  const size_t blocks = static_cast<size_t>(H / 64);
  if (packed_bytes) *packed_bytes = blocks * rows * 32;
  if (scale_bytes) *scale_bytes = blocks * rows * 2;
  return blocks * rows * 34;
}

flp_status flp_mxfp4_quantize(const void *W, flp_dtype dtype, int64_t V, int64_t H,
                              int64_t ld_w, uint8_t *packed, uint8_t *scales,
                              flp_stream_t stream) {
  g_err[0] = 0;
  if (V <= 0 || H <= 0 || H % 64 != 0)
    return fail(FLP_ERR_INVALID_ARG, "V must be > 0 and H a positive multiple of 64");
  if (dtype != FLP_BF16 && dtype != FLP_FP16) return fail(FLP_ERR_INVALID_ARG, "bad dtype");
  if (ld_w < H) return fail(FLP_ERR_INVALID_ARG, "ld_w < H");
  if (!W || !packed || !scales) return fail(FLP_ERR_INVALID_ARG, "W, packed and scales are required");
  if (reinterpret_cast<uintptr_t>(W) % 2 != 0 || !aligned16(packed))
    return fail(FLP_ERR_INVALID_ARG, "W must be 2-byte and packed 16-byte aligned");
  DeviceInfo dev;
  const flp_status st = device_info(&dev);
  if (st != FLP_OK) return st;
  const cudaError_t e =
      launch_mxfp4_quantize(W, dtype == FLP_BF16, V, H, ld_w, flp_mxfp4_rows(V), packed, scales,
                            dev.sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return FLP_OK;
}

flp_status flp_kl_mxfp4(const flp_shape *s, const void *h_s, const void *W_s, const void *h_t,
                        const uint8_t *Wt_packed, const uint8_t *Wt_scales,
                        const int64_t *row_idx, float *out_kl, void *ws, size_t ws_bytes,
                        flp_stream_t stream) {
  g_err[0] = 0;
  const char *why = nullptr;
  if (!shape_ok(s, &why)) return fail(FLP_ERR_INVALID_ARG, "%s", why);
  if (s->dtype != FLP_BF16)
    return fail(FLP_ERR_UNSUPPORTED, "the MXFP4 teacher head needs bf16 student and teacher rows");
  if (s->H % 64 != 0) return fail(FLP_ERR_INVALID_ARG, "H must be a multiple of 64");
  if (s->n_rows > 0 && (!Wt_packed || !Wt_scales))
    return fail(FLP_ERR_INVALID_ARG, "Wt_packed and Wt_scales are required");
  if ((Wt_packed && !aligned16(Wt_packed)) || (Wt_scales && !aligned16(Wt_scales)))
    return fail(FLP_ERR_INVALID_ARG, "Wt_packed and Wt_scales must be 16-byte aligned");
  const MxOperand mx{Wt_packed, Wt_scales, static_cast<long long>(flp_mxfp4_rows(s->V))};
  return kl_impl(s, h_s, W_s, h_t, nullptr, mx, row_idx, out_kl, ws, ws_bytes, stream);
}


size_t flp_mx_head_bytes(int64_t V, int64_t H) {
  if (V <= 0 || H <= 0 || H % kMxChunk != 0 || V > (int64_t(1) << 30) || H > (int64_t(1) << 24))
    return 0;
  return mx_head_code_bytes(V, H) + mx_head_atom_bytes(V, H);
}

flp_status flp_mx_head_quantize(const void *W, flp_dtype dtype, int64_t V, int64_t H, int64_t ld_w,
                                void *head, flp_stream_t stream) {
  g_err[0] = 0;
  if (flp_mx_head_bytes(V, H) == 0)
    return fail(FLP_ERR_INVALID_ARG, "V must be > 0 and H a positive multiple of 128");
  if (dtype != FLP_BF16 && dtype != FLP_FP16) return fail(FLP_ERR_INVALID_ARG, "bad dtype");
  if (ld_w < H) return fail(FLP_ERR_INVALID_ARG, "ld_w < H");
  if (!W || !head) return fail(FLP_ERR_INVALID_ARG, "W and head are required");
  if (reinterpret_cast<uintptr_t>(W) % 2 != 0 || reinterpret_cast<uintptr_t>(head) % 256 != 0)
    return fail(FLP_ERR_INVALID_ARG, "W must be 2-byte and head 256-byte aligned");
  DeviceInfo dev;
  const flp_status st = device_info(&dev);
  if (st != FLP_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *codes = static_cast<uint8_t *>(head);
  const size_t used = static_cast<size_t>(V) * static_cast<size_t>(H / 2);
  uint8_t *atoms = codes + mx_head_code_bytes(V, H);
  // the kernel writes neither the padding after the codes nor the atom bytes
  // of the rows past each tile's 224
  cudaError_t e = cudaMemsetAsync(codes + used, 0, flp_mx_head_bytes(V, H) - used, cs);
  if (e == cudaSuccess)
    e = launch_mx_head_quantize(W, dtype == FLP_BF16, V, H, ld_w, codes, atoms, dev.sms, cs);
  if (e != cudaSuccess) return cuda_fail(e, "head quantize launch");
  return FLP_OK;
}

flp_status flp_mxfp8_quantize(const void *X, flp_dtype dtype, int64_t R, int64_t H, int64_t ld,
                              uint8_t *codes, uint8_t *scales, flp_stream_t stream) {
  g_err[0] = 0;
  if (R < 0 || H <= 0 || H % 32 != 0 || ld < H || ld % 8 != 0)
    return fail(FLP_ERR_INVALID_ARG, "need R >= 0, H a positive multiple of 32, ld >= H and a multiple of 8");
  if (dtype != FLP_BF16 && dtype != FLP_FP16) return fail(FLP_ERR_INVALID_ARG, "bad dtype");
  if (R == 0) return FLP_OK;
  if (!X || !codes || !scales) return fail(FLP_ERR_INVALID_ARG, "X, codes and scales are required");
  if (!aligned16(X) || !aligned16(codes))
    return fail(FLP_ERR_INVALID_ARG, "X and codes must be 16-byte aligned");
  DeviceInfo dev;
  const flp_status st = device_info(&dev);
  if (st != FLP_OK) return st;
  const cudaError_t e = launch_mxfp8_quantize(X, dtype == FLP_BF16, R, H, ld, nullptr, R, codes,
                                              scales, false, dev.sms,
                                              reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "MXFP8 quantize launch");
  return FLP_OK;
}

flp_status flp_kl_mx(const flp_shape *s, const void *h_s, const void *W_s, const void *h_t,
                     const void *Wt_head, const int64_t *row_idx, float *out_kl, void *ws,
                     size_t ws_bytes, flp_stream_t stream) {
  g_err[0] = 0;
  return kl_bs_impl(s, h_s, W_s, h_t, Wt_head, row_idx, out_kl, ws, ws_bytes, stream);
}

flp_status flp_logprob_entropy_mx(const flp_shape *s, const void *h, const void *head,
                                  const int64_t *targets, const int64_t *row_idx,
                                  float temperature, float *out_logp, float *out_ent,
                                  float *out_lse, float *out_ez, void *ws, size_t ws_bytes,
                                  flp_stream_t stream) {
  g_err[0] = 0;
  return fwd_bs_impl(s, h, head, targets, row_idx, temperature, out_logp, out_ent, out_lse, out_ez,
                     ws, ws_bytes, stream);
}

flp_status flp_backward(const flp_shape *s, const void *h, const void *W, const int64_t *targets,
                        const int64_t *row_idx, float temperature, const float *g1,
                        const float *g2, const float *lse, const float *ez, void *dh, float *dW,
                        void *ws, size_t ws_bytes, flp_stream_t stream) {
  return backward_impl(s, h, W, targets, row_idx, nullptr, 0, temperature, g1, g2, lse, ez, dh, dW,
                       ws, ws_bytes, stream);
}

flp_status flp_backward_support(const flp_shape *s, const void *h, const void *W,
                                const int64_t *targets, const int64_t *row_idx,
                                const uint32_t *support, int64_t ld_support, float temperature,
                                const float *g1, const float *g2, const float *lse,
                                const float *ez, void *dh, float *dW, void *ws, size_t ws_bytes,
                                flp_stream_t stream) {
  g_err[0] = 0;
  if (!support) return fail(FLP_ERR_INVALID_ARG, "support is required");
  return backward_impl(s, h, W, targets, row_idx, support, ld_support, temperature, g1, g2, lse,
                       ez, dh, dW, ws, ws_bytes, stream);
}

flp_status flp_pack_support(const uint8_t *mask, int64_t T, int64_t V, int64_t ld_mask,
                            uint32_t *support, int64_t ld_support, flp_stream_t stream) {
  g_err[0] = 0;
  if (T < 0 || V <= 0) return fail(FLP_ERR_INVALID_ARG, "T must be >= 0 and V > 0");
  if (ld_mask < V) return fail(FLP_ERR_INVALID_ARG, "ld_mask < V");
  if (ld_support < cdiv(V, 32)) return fail(FLP_ERR_INVALID_ARG, "ld_support < ceil(V / 32)");
  if (T == 0) return FLP_OK;
  if (!mask || !support) return fail(FLP_ERR_INVALID_ARG, "mask and support are required");
  if (reinterpret_cast<uintptr_t>(support) % 4 != 0)
    return fail(FLP_ERR_INVALID_ARG, "support must be 4-byte aligned");
  DeviceInfo dev;
  const flp_status st = device_info(&dev);
  if (st != FLP_OK) return st;
  const cudaError_t e = launch_pack_support(mask, T, V, ld_mask, support, ld_support, dev.sms,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pack launch");
  return FLP_OK;
}

flp_status flp_logprob_entropy_noalloc(const flp_shape *s, const void *h, const void *W,
                                       const int64_t *targets, const int64_t *row_idx,
                                       float temperature, float *out_logp, float *out_ent,
                                       float *out_lse, float *out_ez, flp_stream_t stream) {
  g_err[0] = 0;
  const char *why = nullptr;
  if (!shape_ok(s, &why)) return fail(FLP_ERR_INVALID_ARG, "%s", why);
  // without row_idx no rows are gathered, so no room is needed for them
  const size_t need = layout_for(s, FLP_OP_LOGPROB_ENTROPY, row_idx != nullptr).total;
  if (need > FLP_NOALLOC_SCRATCH_BYTES)
    return fail(FLP_ERR_WORKSPACE,
                "problem needs %zu bytes of scratch; the static scratch holds %zu "
                "(use flp_logprob_entropy with a workspace)",
                need, static_cast<size_t>(FLP_NOALLOC_SCRATCH_BYTES));
  if (s->n_rows == 0) return FLP_OK;
  void *scratch = nullptr;
  const flp_status st = noalloc_scratch(&scratch);
  if (st != FLP_OK) return st;
  return flp_logprob_entropy(s, h, W, targets, row_idx, temperature, out_logp, out_ent, out_lse,
                             out_ez, scratch, FLP_NOALLOC_SCRATCH_BYTES, stream);
}

flp_status flp_selftest_wait_timeout(uint64_t limit_ns, void *ws, flp_stream_t stream) {
  g_err[0] = 0;
  if (!ws) return fail(FLP_ERR_WORKSPACE, "workspace is NULL");
  if (limit_ns < 1000000ull || limit_ns > 1000000000ull)
    return fail(FLP_ERR_INVALID_ARG, "limit_ns must be within 1 ms .. 1 s");
  DeviceInfo dev;
  const flp_status st = device_info(&dev);
  if (st != FLP_OK) return st;
  const cudaError_t e =
      launch_wait_timeout(limit_ns, static_cast<uint32_t *>(ws), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return FLP_OK;
}

flp_status flp_read_device_status(const void *ws, flp_device_status *out, flp_stream_t stream) {
  g_err[0] = 0;
  if (!ws || !out) return fail(FLP_ERR_INVALID_ARG, "workspace and out are required");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t w[4];
  e = cudaMemcpy(w, ws, sizeof w, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  out->bad_targets = w[kStatBadTarget];
  out->bad_rows = w[kStatBadRow];
  out->timeouts = w[kStatTimeout];
  out->empty_supports = w[kStatEmptySupport];
  if (out->bad_targets || out->bad_rows || out->timeouts || out->empty_supports)
    return fail(FLP_ERR_DEVICE_STATUS,
                "device status: %u bad targets, %u bad rows, %u timeouts, %u empty supports",
                out->bad_targets, out->bad_rows, out->timeouts, out->empty_supports);
  return FLP_OK;
}

}  // extern "C"
