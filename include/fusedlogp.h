/*
 * fusedlogp.h -- C ABI of libfusedlogp: fused LM-head token scoring on one
 * GB300 GPU (sm_103a).
 *
 * For each scored row r of the hidden states h[T,H] the library forms the
 * logits z = h[r] W^T one vocabulary tile at a time on the tensor cores
 * (FP32 accumulation), divides by the temperature in FP32 after that
 * upcast, and folds each tile into a per-row online log-sum-exp.  The
 * [T,V] logits are never written to memory.
 *
 * Pages this follows:
 *   - miles PR #2764 summary (prhub), "Implementation breakdown" items 2-4:
 *     upcast each chunk of logits to FP32, then apply the temperature in
 *     FP32; log-prob and entropy come from the same upcast values; FP16
 *     and BF16 inputs are both accepted; sums accumulate in FP32.
 *   - miles PR #4645 ("--log-probs-backend fused_lm_head"), "How it works":
 *     the output layer runs only on the rows that are scored (response
 *     rows), tile by tile, and the [tokens x vocab] logits and their
 *     gradient are never materialised; the backward replays each tile.
 *   - DeepSeek-V4 book ch. 19, "Never materialize logits" and "TileLang KL
 *     kernel": teacher logits are rebuilt from cached hidden states through
 *     the teacher head and an exact full-vocabulary KL is computed without
 *     either logit tensor existing in memory, in a fixed (static) memory
 *     layout.
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller.  The
 *     library allocates no device memory during a call: scratch space is the
 *     caller's workspace, sized by flp_workspace_size().
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and is asynchronous.  No call synchronises, except
 *     flp_read_device_status().
 *   - Arguments are validated on the host before anything is enqueued; a
 *     call that returns an error has enqueued nothing, except FLP_ERR_CUDA
 *     from a failed launch.  flp_last_error() gives a one-line reason.
 *   - Data-dependent problems do not fail the call: a target outside [0,V)
 *     or a row_idx entry outside [0,T) yields NaN in that row's outputs and
 *     is counted in the workspace's device status (flp_read_device_status).
 *   - Matrices are row-major.  h is [T, ld_h] with H <= ld_h used columns;
 *     W is [V, ld_w].  H, ld_h and ld_w must be multiples of 8 and h, W
 *     16-byte aligned (tensor-memory-access copies move 16-byte units).
 *   - n_rows == 0 is valid (the "no scored rows" case): the scoring and KL
 *     calls enqueue nothing, the backward only zeroes dh and dW.
 */
#ifndef FUSEDLOGP_H
#define FUSEDLOGP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st *flp_stream_t;

typedef enum {
    FLP_OK = 0,
    FLP_ERR_INVALID_ARG = 1,   /* null pointer, bad size (also one beyond the 32-bit tiling
                                  range), stride, alignment or temperature */
    FLP_ERR_UNSUPPORTED = 2,   /* no usable sm_103a device, or an unsupported combination
                                  (the MXFP4 teacher with fp16 rows) */
    FLP_ERR_WORKSPACE = 3,     /* workspace null or smaller than flp_workspace_size() */
    FLP_ERR_CUDA = 4,          /* a CUDA runtime/driver call or a launch failed */
    FLP_ERR_DEVICE_STATUS = 5  /* flp_read_device_status(): the device recorded a problem */
} flp_status;

typedef enum { FLP_BF16 = 0, FLP_FP16 = 1 } flp_dtype;

typedef enum {
    FLP_OP_LOGPROB_ENTROPY = 0,
    FLP_OP_KL = 1,
    FLP_OP_BACKWARD = 2,
    FLP_OP_KL_MX = 3,  /* flp_kl_mx: the teacher on the block-scaled tensor cores */
    FLP_OP_LOGPROB_ENTROPY_MX = 4  /* flp_logprob_entropy_mx: scoring on the block-scaled
                                      tensor cores */
} flp_op;

/*
 * Problem shape.  n_rows is the number of scored rows: the length of
 * row_idx, or T when row_idx is NULL.  dtype is the element type of h and W
 * (and of dh in the backward).
 */
typedef struct {
    int64_t T;       /* rows of h; entries of targets */
    int64_t H;       /* hidden size: the contraction length */
    int64_t V;       /* vocabulary size: rows of W */
    int64_t n_rows;  /* scored rows */
    flp_dtype dtype; /* FLP_BF16 or FLP_FP16 */
    int64_t ld_h;    /* row stride of h (and dh) in elements, >= H */
    int64_t ld_w;    /* row stride of W (and dW) in elements, >= H */
} flp_shape;

/* Problems the device counted during the last call on a workspace. */
typedef struct {
    uint32_t bad_targets; /* scored rows whose target was outside [0, V) */
    uint32_t bad_rows;    /* row_idx entries outside [0, T) */
    uint32_t timeouts;    /* pipeline waits that gave up; outputs of that call are invalid */
    uint32_t empty_supports; /* scored rows whose sampling support held no token */
} flp_device_status;

/*
 * Bytes of workspace `op` needs for `shape` (0 if the shape is invalid).
 * The size is a function of the shape alone (not of the device or of
 * whether row_idx is given); it is about n_rows*H*2 bytes for the gathered
 * rows (twice that for the KL's two heads), plus O(n_rows * 64) bytes of
 * per-row partial state, plus, for the backward, one bounded chunk of the
 * bf16/fp16 logit gradient (at most 4 GiB; never a [T,V] buffer for the
 * forward or KL), 4*T bytes of per-row counts and at most 40 MiB of FP32
 * partial tiles for the dh GEMM (when the last wave of its output tiles
 * would leave most CTA pairs idle, those tiles are split along V and their
 * partial sums added in a fixed order).
 * The size returned is always enough.  The scoring and KL calls made with
 * row_idx == NULL gather no rows and accept a workspace smaller by the
 * gathered rows' bytes (n_rows*H*2 per head, rounded up to 1 KiB).
 */
size_t flp_workspace_size(const flp_shape *shape, flp_op op);

/*
 * Target log-probability and entropy of softmax(z / temperature) per
 * scored row, z = h[row] W^T (miles PR #2764 summary, "Implementation
 * breakdown" items 2-3: each chunk of logits is upcast to FP32, divided by
 * the temperature in FP32, and the log-prob and entropy are both taken from
 * those values; miles PR #4645, "How it works": the output layer runs on the
 * scored rows only, a tile at a time).
 *
 *   h            [T, ld_h] bf16/fp16 hidden states
 *   W            [V, ld_w] bf16/fp16 output-layer (LM head) weight
 *   targets      [T] int64 target token of each h row (indexed by h row,
 *                not by scored position)
 *   row_idx      [n_rows] int64 rows of h to score, any order, duplicates
 *                allowed; NULL scores rows 0..T-1 (then n_rows must be T)
 *   temperature  finite and > 0; applied in FP32 after the FP32 upcast
 *                (1 is an exact no-op)
 *   out_logp     [n_rows] float: z'_tgt - logsumexp(z'),  z' = z / temperature
 *   out_ent      [n_rows] float: entropy (nats) of softmax(z')
 *   out_lse      [n_rows] float or NULL: logsumexp(z')
 *   out_ez       [n_rows] float or NULL: E_p[z'] = out_lse - out_ent
 * Outputs are compact, in row_idx order.
 */
flp_status flp_logprob_entropy(const flp_shape *shape, const void *h, const void *W,
                               const int64_t *targets, const int64_t *row_idx,
                               float temperature, float *out_logp, float *out_ent,
                               float *out_lse, float *out_ez,
                               void *workspace, size_t workspace_bytes, flp_stream_t stream);

/*
 * K target tokens per scored row (score centering's K-candidate scoring,
 * miles PR #4645, "Scope": a fused log-prob op with K targets per row):
 * the same pass as flp_logprob_entropy, capturing K target logits per row.
 *   targets      [T, K] int64, row-major, indexed by h row
 *   K            1 .. FLP_MAX_TARGETS
 *   out_logp     [n_rows, K] float: z'_{targets[row, k]} - logsumexp(z')
 *   out_ent, out_lse, out_ez as in flp_logprob_entropy.
 * A candidate outside [0, V) gives NaN in its slot and is counted in
 * bad_targets.  Uses the workspace of FLP_OP_LOGPROB_ENTROPY.
 */
#define FLP_MAX_TARGETS 8

flp_status flp_logprob_entropy_k(const flp_shape *shape, const void *h, const void *W,
                                 const int64_t *targets, int32_t K, const int64_t *row_idx,
                                 float temperature, float *out_logp, float *out_ent,
                                 float *out_lse, float *out_ez,
                                 void *workspace, size_t workspace_bytes, flp_stream_t stream);

/*
 * Log-prob and entropy under each row's sampling support (miles PR #2764
 * summary, math_utils.py snippet: the sampling_mask argument of
 * calculate_log_probs_and_entropy, cut into row chunks with the logits and
 * tokens).  The distribution of row r is softmax(z') restricted to the
 * tokens of its support S_r and renormalised; tokens off S_r have
 * probability 0:
 *   out_logp   z'_tgt - log sum_{v in S} exp(z'_v); -INFINITY if tgt is not in S
 *   out_ent    entropy (nats) of the restricted distribution
 *   out_lse    log sum_{v in S} exp(z'_v);   out_ez = sum_{v in S} p_v z'_v
 *   support    [T, ld_support] uint32 words, DEVICE, indexed by h row (like
 *              targets): token v is in row r's support iff bit (v % 32) of
 *              support[r * ld_support + v / 32] is set.  Bits at v >= V are
 *              ignored.  4-byte aligned; ld_support >= ceil(V / 32).
 *              flp_pack_support builds it from a byte-per-token mask.
 * Other arguments as in flp_logprob_entropy; same workspace.  A row whose
 * support holds no token gets NaN outputs and is counted in empty_supports.
 */
flp_status flp_logprob_entropy_support(const flp_shape *shape, const void *h, const void *W,
                                       const int64_t *targets, const int64_t *row_idx,
                                       const uint32_t *support, int64_t ld_support,
                                       float temperature, float *out_logp, float *out_ent,
                                       float *out_lse, float *out_ez,
                                       void *workspace, size_t workspace_bytes,
                                       flp_stream_t stream);

/*
 * Packs a byte-per-token support mask into the bit words the *_support entry
 * points read: support[r * ld_support + w] gets bit j set iff
 * mask[r * ld_mask + 32 w + j] != 0 (and 32 w + j < V).  Bits past V and
 * words past ceil(V / 32) are written as 0.
 *   mask      [T, ld_mask] uint8 (e.g. a torch.bool tensor), DEVICE, ld_mask >= V
 *   support   [T, ld_support] uint32, DEVICE, 4-byte aligned, ld_support >= ceil(V / 32)
 */
flp_status flp_pack_support(const uint8_t *mask, int64_t T, int64_t V, int64_t ld_mask,
                            uint32_t *support, int64_t ld_support, flp_stream_t stream);

/*
 * Full-vocabulary KL(teacher || student) per scored row (DeepSeek-V4 book
 * ch. 19, "TileLang KL kernel": the exact KL over the whole vocabulary from
 * the two heads' logits, rebuilt from the cached hidden states, in a static
 * memory layout, with neither logit tensor in memory):
 *   KL = sum_v p_t,v (log p_t,v - log p_s,v),
 *   p_s = softmax(h_s[row] W_s^T),  p_t = softmax(h_t[row] W_t^T),
 * temperature 1, neither logit tensor materialised.  Student and teacher
 * share shape (T, H, V, dtype, ld_h, ld_w).
 *   h_s, h_t     [T, ld_h];  W_s, W_t [V, ld_w]
 *   row_idx      [n_rows] int64 or NULL (all rows)
 *   out_kl       [n_rows] float
 */
flp_status flp_kl(const flp_shape *shape, const void *h_s, const void *W_s,
                  const void *h_t, const void *W_t, const int64_t *row_idx,
                  float *out_kl, void *workspace, size_t workspace_bytes,
                  flp_stream_t stream);

/*
 * Teacher head in MXFP4 (DeepSeek-V4 book ch. 19, "1. FP4 in OPD": the
 * inference-only teacher forwards run on 4-bit MXFP4 weights, which cuts the
 * teacher head's memory and read traffic about 4x against bf16).
 *
 * Format (OCP Microscaling FP4): E2M1 elements (1 sign, 2 exponent bits with
 * bias 1, 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) with one
 * E8M0 scale code s (value 2^(s - 127)) per 32 consecutive elements of a row.
 * Layout (blocked, so that a tile of rows is contiguous): with
 * V_pad = flp_mxfp4_rows(V) and for each 64-wide column block kb < H/64 and
 * row v < V_pad,
 *   packed[(kb * V_pad + v) * 32 + b]  elements kb*64 + 2b (low nibble) and
 *                                      kb*64 + 2b + 1 (high nibble) of row v
 *   scales[(kb * V_pad + v) * 2 + j]   scale code of elements kb*64 + 32j ..
 *                                      kb*64 + 32j + 31
 * Rows v >= V are zero.  Sizes: flp_mxfp4_bytes.  H must be a multiple of 64.
 */
int64_t flp_mxfp4_rows(int64_t V);  /* V rounded up to a multiple of 256 (0 if V <= 0) */

/* Bytes of the packed codes and the scales; returns their sum (0 if V <= 0 or
 * H is not a positive multiple of 64).  Either out pointer may be NULL. */
size_t flp_mxfp4_bytes(int64_t V, int64_t H, size_t *packed_bytes, size_t *scale_bytes);

/*
 * Quantises W [V, ld_w] (bf16/fp16, DEVICE, finite values) to MXFP4:
 *   s = floor(log2 max |x|) - 2 + 127 over each 32-element block, clamped to
 *       [0, 254] (0 for an all-zero block);
 *   each element = the E2M1 value nearest to x / 2^(s - 127), ties to the
 *       even code, magnitudes above 6 saturated to 6; zero is stored as +0.
 * packed and scales are DEVICE buffers of flp_mxfp4_bytes' sizes; packed
 * 16-byte aligned.  Enqueued on `stream`.
 */
flp_status flp_mxfp4_quantize(const void *W, flp_dtype dtype, int64_t V, int64_t H,
                              int64_t ld_w, uint8_t *packed, uint8_t *scales,
                              flp_stream_t stream);

/*
 * flp_kl with the teacher head given in MXFP4 (Wt_packed, Wt_scales as
 * produced by flp_mxfp4_quantize for V rows of H columns): the teacher logits
 * are h_t[row] times the decoded weights, exactly (every MXFP4 value is a
 * bf16 value, decoded in shared memory next to the tensor cores; decoded
 * values below bf16's normal range, 2^-126, which only scale codes 0 and 1
 * can give, flush to zero).  bf16 only (FLP_ERR_UNSUPPORTED for fp16); H a
 * multiple of 64; both buffers 16-byte aligned.  Same workspace as FLP_OP_KL.
 */
flp_status flp_kl_mxfp4(const flp_shape *shape, const void *h_s, const void *W_s,
                        const void *h_t, const uint8_t *Wt_packed, const uint8_t *Wt_scales,
                        const int64_t *row_idx, float *out_kl,
                        void *workspace, size_t workspace_bytes, flp_stream_t stream);

/*
 * The teacher forward on the block-scaled tensor cores (DeepSeek-V4 book
 * ch. 19, "1. FP4 in OPD": the inference-only teacher forwards run in native
 * FP4, which cuts the teacher head's memory and read traffic; the MMA that
 * takes FP4 weights natively takes the other operand in a microscaling
 * format too).  The teacher head is MXFP4 as for flp_mxfp4_quantize (same
 * rounding), in the layout the block-scaled MMA reads; the teacher's hidden
 * rows are quantised to MXFP8 per call (flp_mxfp8_quantize's rule); the
 * teacher logits are the exact products of the two quantised operands,
 * accumulated in FP32 by tcgen05.mma kind::mxf8f6f4 at twice the bf16 rate.
 * The student is computed as in flp_kl.
 *
 * Head layout (`head`, flp_mx_head_bytes bytes, 256-byte aligned DEVICE
 * buffer):
 *   codes   [V, H/2] bytes at head: byte b of row v holds elements 2b (low
 *           nibble) and 2b + 1 (high nibble), E2M1 codes
 *   atoms   at head + (V * H/2 rounded up to 1024): for vocabulary tile
 *           t = v / 224, row i = v % 224, 128-wide k-chunk c = k / 128 and
 *           step j = (k % 128) / 32, the E8M0 scale of elements
 *           c*128 + 32j .. + 31 of row v sits in the 512-byte atom
 *           (t * (H/128) + c) * 2 + i / 128, at byte
 *           (i % 128 % 32) * 16 + (i % 128 / 32) * 4 + j.  The padding after
 *           the codes and the atom bytes of rows past V (and past each
 *           tile's 224 rows) are 0.
 */
/* Bytes of a block-scaled teacher head (0 if V <= 0 or H is not a positive
 * multiple of 128). */
size_t flp_mx_head_bytes(int64_t V, int64_t H);

/*
 * Quantises W [V, ld_w] (bf16/fp16, DEVICE, finite) to MXFP4 in the head
 * layout above: per 32-element block s = floor(log2 max|x|) - 2 + 127
 * clamped to [0, 254] (0 for an all-zero block), elements the E2M1 value
 * nearest to x / 2^(s - 127), ties to the even code, saturated at 6, zero as
 * +0 (the rule of flp_mxfp4_quantize).  H a multiple of 128.
 */
flp_status flp_mx_head_quantize(const void *W, flp_dtype dtype, int64_t V, int64_t H,
                                int64_t ld_w, void *head, flp_stream_t stream);

/*
 * OCP MXFP8 (E4M3 elements: 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, largest finite 448; one E8M0 scale per 32 elements) of X [R, ld]
 * (bf16/fp16, DEVICE, finite, 16-byte aligned, ld a multiple of 8):
 *   s = floor(log2 max|x|) - 8 + 127 over each 32-element block, clamped to
 *       [0, 254] (0 for an all-zero block);
 *   each element = the E4M3 value nearest to x / 2^(s - 127), ties to the
 *       even code, magnitudes above 448 saturated to 448, zero as +0.
 *   codes   [R, H] uint8 row-major (16-byte aligned); scales [R, H/32] uint8.
 * This is the quantisation flp_kl_mx applies to the teacher's hidden rows.
 */
flp_status flp_mxfp8_quantize(const void *X, flp_dtype dtype, int64_t R, int64_t H, int64_t ld,
                              uint8_t *codes, uint8_t *scales, flp_stream_t stream);

/*
 * KL(teacher || student) per scored row as flp_kl, with the teacher's logits
 * h_t[row]^MXFP8 times the MXFP4 head `Wt_head` (from flp_mx_head_quantize,
 * V rows of H columns) on the block-scaled tensor cores.  bf16 or fp16 rows
 * and student head; H a multiple of 128.  Workspace: flp_workspace_size(shape,
 * FLP_OP_KL_MX) (it holds the quantised teacher rows: n_rows * H bytes plus
 * their scales).
 */
flp_status flp_kl_mx(const flp_shape *shape, const void *h_s, const void *W_s,
                     const void *h_t, const void *Wt_head, const int64_t *row_idx,
                     float *out_kl, void *workspace, size_t workspace_bytes,
                     flp_stream_t stream);

/*
 * flp_logprob_entropy with the logits on the block-scaled tensor cores, for
 * scoring that needs no backward (DeepSeek-V4 book ch. 19, "1. FP4 in OPD":
 * rollout, the teachers and the reference model that gives the KL baseline
 * run their forwards in native 4-bit precision): each scored row h[row] is
 * quantised to MXFP8 (flp_mxfp8_quantize's rule) inside the call and the
 * logits are h[row]^MXFP8 times the MXFP4 head `head` (from
 * flp_mx_head_quantize, V rows of H columns), FP32-accumulated with the
 * scales applied inside the MMA; then, as in flp_logprob_entropy (temperature
 * in FP32 after the upcast), per scored position i:
 *   out_logp[i] = z'[tgt] - LSE,  out_ent[i] = entropy,  out_lse / out_ez
 *   optional (NULL to skip).
 * h bf16 or fp16 [T, ld_h], 16-byte aligned; H a multiple of 128; head
 * 256-byte aligned.  targets [T] by h row; row_idx [n_rows] or NULL (then
 * n_rows == T).  Bad rows and targets are handled as in flp_logprob_entropy.
 * Workspace: flp_workspace_size(shape, FLP_OP_LOGPROB_ENTROPY_MX) (it holds
 * the quantised rows: n_rows * H bytes plus their scales).  shape->ld_w is
 * not used but must pass the shape checks (set it to H).  The head buffer
 * must hold flp_mx_head_bytes(V, H) bytes (the library cannot check its
 * size).  Errors: FLP_ERR_INVALID_ARG for H not a multiple of 128, a
 * non-finite or non-positive temperature, a missing or misaligned pointer,
 * or sizes beyond the 32-bit coordinates of the scale atoms;
 * FLP_ERR_WORKSPACE for a missing or short workspace.
 */
flp_status flp_logprob_entropy_mx(const flp_shape *shape, const void *h, const void *head,
                                  const int64_t *targets, const int64_t *row_idx,
                                  float temperature, float *out_logp, float *out_ent,
                                  float *out_lse, float *out_ez, void *workspace,
                                  size_t workspace_bytes, flp_stream_t stream);

/*
 * Gradients of L = sum_i g1[i] logp_i + g2[i] ent_i (logp, ent as in
 * flp_logprob_entropy) by tile recompute (miles PR #4645, "How it works": the
 * backward replays each logit tile instead of keeping the [tokens x vocab]
 * logits or their gradient from the forward):
 *   G_iv = (g1[i] (1[v = tgt_i] - p_iv) - g2[i] p_iv (z'_iv - E_p[z'_i])) / temperature
 *   dh[row_idx[i], :] = sum_v G_iv W[v, :]      (dtype of h; rows not scored are 0)
 *   dW[v, :]          = sum_i G_iv h[row_idx[i], :]   (float32, overwritten)
 *   g1, g2       [n_rows] float upstream gradients of logp and ent
 *   lse, ez      [n_rows] float from a previous flp_logprob_entropy with
 *                the same inputs (out_lse, out_ez), or both NULL: the
 *                statistics are then recomputed (one extra forward pass)
 *   dh           [T, ld_h] dtype; dW [V, ld_w] float32.  Either may be NULL
 *                (not both) to skip that gradient, e.g. for a frozen output
 *                layer: a NULL dW skips the dW GEMM, a third of the work.
 * row_idx may name a row more than once: that row's dh is the sum of its
 * contributions, added onto the zeroed row with packed 16-bit atomics (so
 * for a row named three or more times the low bits depend on the order of
 * the additions; every other row is written once and is bitwise
 * reproducible).
 * n_rows == 0 writes zeros to dh and dW (those given).  The scored rows are processed in
 * chunks of at most flp's chunk size (as many rows as keep the chunk's
 * logit gradient within 4 GiB; the environment variable FLP_GRAD_CHUNK_ROWS,
 * read at each call, can lower it); chunk lengths follow flp_row_chunks.
 * FLP_DH_SPLIT=0 (read at each call) turns off the split of the dh GEMM's
 * last wave (flp_plan's dh_split); the results agree to FP32 rounding.
 */
flp_status flp_backward(const flp_shape *shape, const void *h, const void *W,
                        const int64_t *targets, const int64_t *row_idx,
                        float temperature, const float *g1, const float *g2,
                        const float *lse, const float *ez, void *dh, float *dW,
                        void *workspace, size_t workspace_bytes, flp_stream_t stream);

/*
 * flp_backward under each row's sampling support (as in
 * flp_logprob_entropy_support): p, lse and E_p[z'] are taken over the row's
 * support, and
 *   G_iv = 1[v in S_i] (g1[i] (1[v = tgt_i] - p_iv) - g2[i] p_iv (z'_iv - E_p[z'_i])) / temperature
 * (a target outside S_i contributes no one-hot term).  lse and ez, if
 * given, must come from flp_logprob_entropy_support with the same support.
 * Every scored row's support must hold at least one token.
 */
flp_status flp_backward_support(const flp_shape *shape, const void *h, const void *W,
                                const int64_t *targets, const int64_t *row_idx,
                                const uint32_t *support, int64_t ld_support, float temperature,
                                const float *g1, const float *g2, const float *lse,
                                const float *ez, void *dh, float *dW,
                                void *workspace, size_t workspace_bytes, flp_stream_t stream);

/*
 * Synchronises `stream` and copies the device status of the last call that
 * used `workspace`.  Returns FLP_ERR_DEVICE_STATUS if any counter is
 * non-zero (the counters are still copied), FLP_OK otherwise.
 */
flp_status flp_read_device_status(const void *workspace, flp_device_status *out,
                                  flp_stream_t stream);

/*
 * Log-prob and entropy without a caller workspace (no counterpart in the
 * pages: this entry point exists for callers that cannot hand the library
 * device memory).  Some callers have no way to allocate device memory at the
 * point where they score: a host program or plugin that owns no allocator, a
 * framework whose memory pool already holds the device's free memory, or a
 * latency-critical loop where cudaMalloc, which may synchronise the device,
 * is not allowed.  This variant takes the same arguments as
 * flp_logprob_entropy minus the workspace and allocates nothing: its scratch
 * space is one statically sized device array inside the library,
 * FLP_NOALLOC_SCRATCH_BYTES (16 MiB), which every GPU that loads the library
 * holds until the process exits.
 *
 *   - The scratch a problem needs is flp_workspace_size(shape,
 *     FLP_OP_LOGPROB_ENTROPY) with row_idx given; with row_idx == NULL no
 *     rows are gathered and the n_rows * H * 2 bytes of gathered rows are
 *     not needed.  A problem that needs more than FLP_NOALLOC_SCRATCH_BYTES
 *     is rejected with FLP_ERR_WORKSPACE before anything is enqueued.  For
 *     example, 4,096 rows x H 4,096 x V 151,936 need 6.1 MiB without row_idx
 *     and fit; with row_idx the gathered rows add 32 MiB and the call is
 *     rejected (at that H and V, up to 1,718 gathered rows fit).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and so does the first
 *     call after the device's context was reset (the library's module, and
 *     the array with it, is then loaded anew).  That first call may also be
 *     the one that makes CUDA load the library's module, which places the
 *     array in device memory.  Make it before any stream capture.
 *   - All calls in the process share the one array, and it keeps the last
 *     call's contents (the status words are cleared at the start of every
 *     call).  Calls whose GPU work overlaps -- on two streams, or from two
 *     host threads -- race on it and give wrong results: serialise them.
 *   - The device status counters of these calls live inside the shared
 *     array and are not exposed.  A row_idx entry outside [0, T) gives NaN
 *     in every output of that row; a target outside [0, V) gives NaN in that
 *     row's out_logp only (its entropy, log-sum-exp and E[z'] stay finite),
 *     so check out_logp to catch bad targets.
 */
#define FLP_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

flp_status flp_logprob_entropy_noalloc(const flp_shape *shape, const void *h, const void *W,
                                       const int64_t *targets, const int64_t *row_idx,
                                       float temperature, float *out_logp, float *out_ent,
                                       float *out_lse, float *out_ez, flp_stream_t stream);

/*
 * Measurement hook.  Makes the NEXT scoring call on the calling host thread
 * record `before` (a cudaEvent_t) on its stream immediately before its
 * tensor-core kernels and `after` immediately after them, so a caller can
 * time the dominant kernel(s) apart from the small gather/merge kernels.
 * The events are used once and then forgotten; pass NULLs to cancel.
 */
flp_status flp_set_kernel_events(void *before, void *after);

/*
 * Self-test of the bounded waits the kernels use on the GPU: launches one
 * tiny kernel whose thread waits on an mbarrier that nothing arrives on.  The
 * wait gives up after limit_ns nanoseconds (1 ms .. 1 s), adds one to the
 * timeout counter of the 256-byte device status block at `workspace` (whose
 * other words are left alone; clear it first) and the kernel exits normally.
 * Read the counter with flp_read_device_status().  Used by the tests to show
 * that a stalled pipeline wait ends in a reported status, not a hung GPU.
 */
flp_status flp_selftest_wait_timeout(uint64_t limit_ns, void *workspace, flp_stream_t stream);

/*
 * Lowers (or restores) the wall-clock limit of the barrier waits inside the
 * kernels of later calls made from the calling host thread: 0 restores the
 * default of 4 s; otherwise limit_ns must lie within 100 ns .. 60 s.  The
 * setting stays until it is changed.  Every pipeline wait is bounded by
 * this limit; a wait that runs out sets the pipeline's abort flag, lets the
 * copies and tensor-core operations already in flight finish, frees its
 * tensor memory, adds one to the `timeouts` counter of the call's device
 * status and ends the kernel normally.  That call's outputs are then
 * invalid, and the context stays usable.  The tests use a limit shorter
 * than a pipeline stage to drive that path on purpose.
 */
flp_status flp_set_wait_limit(uint64_t limit_ns);

/* Static description of a status code. */
const char *flp_status_string(flp_status status);

/* One-line reason for the last failure on the calling host thread ("" if none). */
const char *flp_last_error(void);

/*
 * Tiling plan of the scoring kernels, for inspection and tests (pure host
 * function; no GPU needed).  num_sms is the number of SMs to plan for.
 * FLP_OP_LOGPROB_ENTROPY with n_rows <= 128 reports the few-rows plan that
 * the scoring calls (flp_logprob_entropy and its _k and _support forms) use:
 * single CTAs (cta_group 1) on 128-row x 256-column tiles.
 */
typedef struct {
    int32_t row_tiles;      /* ceil(n_rows / block_m) */
    int32_t vocab_tiles;    /* ceil(V / block_n) */
    int32_t block_m;        /* scored rows per tensor-core tile (128 x cta_group) */
    int32_t block_n;        /* vocabulary columns per tensor-core tile */
    int32_t cta_group;      /* CTAs that share one tile (2: tcgen05 CTA pairs) */
    int32_t splits;         /* vocabulary splits per row tile (partial states per row) */
    int32_t tiles_per_split;
    int32_t band;           /* row tiles that share the weight stream in one band */
    int32_t items;          /* work items = row_tiles * splits */
    int32_t grid;           /* persistent CTAs launched (a multiple of cta_group) */
    int64_t max_tiles_per_cta; /* load of the busiest CTA (pair), in block_m x block_n tiles */
    int64_t chunk_rows;     /* FLP_OP_BACKWARD: rows per logit-gradient chunk (else 0) */
    int32_t dh_split;       /* FLP_OP_BACKWARD, first chunk: K segments into which each tile
                               of the dh GEMM's last, partial wave is split (1: none) */
    int32_t dh_tail_tiles;  /* FLP_OP_BACKWARD, first chunk: the tiles so split */
} flp_plan;

flp_status flp_plan_scoring(const flp_shape *shape, flp_op op, int32_t num_sms, flp_plan *out);

/*
 * Row chunks of the backward: the scored rows are processed in
 * num_chunks = (n_rows - 1) / chunk_rows + 1 chunks of at most
 * ceil(n_rows / num_chunks) rows each (the last one shorter), the chunking
 * rule of the pages' calculate_log_probs_and_entropy.  Writes up to
 * `max_out` chunk lengths; returns the number of chunks (0 for n_rows = 0).
 */
int64_t flp_row_chunks(int64_t n_rows, int64_t chunk_rows, int64_t *out_lengths,
                       int64_t max_out);

#ifdef __cplusplus
}
#endif

#endif /* FUSEDLOGP_H */
