/*
 * oracle.c -- float64 CPU oracle for fused LM-head token scoring.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library; it is the plain definition of what that library computes,
 * written out so a reader can check it against the pages by eye.
 *
 * What it follows (pages and sections):
 *   - miles PR #2764 summary (prhub), "Implementation breakdown" item 2 and
 *     the math_utils.py snippet: logits are upcast (here: exact float64),
 *     then divided by the temperature after the upcast; log-prob and
 *     entropy are taken from the same upcast values.
 *   - miles PR #4645, "How it works" (Op, Selection): logits z = h W^T for
 *     the scored (response) rows only; log-prob of the target and entropy
 *     per row; backward = gradient of sum(g1*logp + g2*ent) w.r.t. h and W.
 *   - DeepSeek-V4 book ch. 19, "Never materialize logits" / "TileLang KL
 *     kernel": exact full-vocabulary KL between teacher and student heads,
 *     read here as KL(teacher || student) = sum_v p_t (log p_t - log p_s).
 *
 * Definitions (per scored row r, all in float64 from the exact values of
 * the bf16/fp16 inputs):
 *   z_v   = sum_k h[r,k] W[v,k]          z'_v = z_v / tau
 *   LSE   = m + log(sum_v exp(z'_v - m)),  m = max_v z'_v   (two passes)
 *   p_v   = exp(z'_v - LSE)
 *   logp  = z'_tgt - LSE
 *   ent   = LSE - sum_v p_v z'_v          Ez = sum_v p_v z'_v
 *   KL    = sum_v p_t,v ((z_t,v - LSE_t) - (z_s,v - LSE_s))
 *   G_v   = (g1 (1[v=tgt] - p_v) - g2 p_v (z'_v - Ez)) / tau
 *   dh[r] = sum_v G_v W[v,:]              dW[v,:] += G_v h[r,:]
 *
 * The z rows are held whole (no blocking of the vocabulary, no online
 * rescaling): this is the definition, not the fast method.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element types of the matrices handed to the oracle. */
enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_F64 = 2, ORC_MXFP4 = 3 };

/*
 * A matrix [V, H] stored in MXFP4 (OCP Microscaling: E2M1 elements, one
 * E8M0 power-of-two scale per 32 consecutive elements of a row), in the
 * blocked layout the library uses: for each 64-wide column block kb and each
 * row v < V_pad, 32 bytes of elements (byte b: element 2b in the low nibble,
 * 2b+1 in the high nibble) at packed[(kb * V_pad + v) * 32] and two scale
 * codes at scales[(kb * V_pad + v) * 2] (elements 0..31 and 32..63 of the
 * block).  Handed to orc_decode as a pointer to this struct.
 */
typedef struct {
    const uint8_t *packed;
    const uint8_t *scales;
    int64_t V_pad;
    int64_t H;
} orc_mx_matrix;

/* E2M1 magnitudes by code (sign in bit 3): 1 sign, 2 exponent (bias 1), 1 mantissa bit. */
static const double orc_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static double orc_mx_element(const orc_mx_matrix *m, int64_t v, int64_t k)
{
    int64_t blk = (k / 64) * m->V_pad + v;
    uint8_t byte = m->packed[blk * 32 + (k % 64) / 2];
    int code = (k % 2) ? (byte >> 4) : (byte & 15);
    int sc = m->scales[blk * 2 + (k % 64) / 32];
    double mag = ldexp(orc_e2m1_mag[code & 7], sc - 127);
    return (code & 8) ? -mag : mag;
}

/* Rows of h whose logits are held at once. */
#define ORC_ROW_BLOCK 32

static double orc_bf16(uint16_t b)
{
    /* bf16 is the top half of an IEEE binary32: exact widening. */
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double orc_fp16(uint16_t b)
{
    /* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
    int sign = (b >> 15) & 1;
    int e = (b >> 10) & 0x1f;
    int f = b & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);             /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Decode n consecutive elements starting at element offset off. */
static void orc_decode(const void *p, int type, int64_t off, int64_t n, double *out)
{
    int64_t i;
    if (type == ORC_BF16) {
        const uint16_t *q = (const uint16_t *)p + off;
        for (i = 0; i < n; ++i) out[i] = orc_bf16(q[i]);
    } else if (type == ORC_FP16) {
        const uint16_t *q = (const uint16_t *)p + off;
        for (i = 0; i < n; ++i) out[i] = orc_fp16(q[i]);
    } else if (type == ORC_MXFP4) {
        const orc_mx_matrix *m = (const orc_mx_matrix *)p;
        for (i = 0; i < n; ++i) out[i] = orc_mx_element(m, (off + i) / m->H, (off + i) % m->H);
    } else {
        const double *q = (const double *)p + off;
        for (i = 0; i < n; ++i) out[i] = q[i];
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_decode_array(const void *p, int type, int64_t n, double *out)
{
    orc_decode(p, type, 0, n, out);
}

/*
 * z[b][v] = sum_k h[rows[b],k] * W[v,k] for b < nb, all v < V.
 * hd holds the nb decoded h rows (nb x H).  W is decoded one vocab row at a
 * time.
 */
static void orc_logits_block(const double *hd, int64_t nb, int64_t H, int64_t V,
                             const void *W, int wtype, int64_t ld_w, double *z)
{
    int64_t v;
#pragma omp parallel
    {
        double *wd = (double *)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(static)
        for (v = 0; v < V; ++v) {
            int64_t b, k;
            orc_decode(W, wtype, v * ld_w, H, wd);
            for (b = 0; b < nb; ++b) {
                const double *hr = hd + b * H;
                double acc = 0.0;
                for (k = 0; k < H; ++k) acc += hr[k] * wd[k];
                z[b * V + v] = acc;
            }
        }
        free(wd);
    }
}

/* Decode the h rows rows[i0 .. i0+nb) into hd (nb x H). */
static void orc_gather_h(const void *h, int htype, int64_t ld_h, const int64_t *rows,
                         int64_t i0, int64_t nb, int64_t H, double *hd)
{
    int64_t b;
    for (b = 0; b < nb; ++b) orc_decode(h, htype, rows[i0 + b] * ld_h, H, hd + b * H);
}

/* Two-pass log-sum-exp of x[0..V) (max shift, then sum of exponentials). */
static double orc_lse(const double *x, int64_t V)
{
    double m = -INFINITY, s = 0.0;
    int64_t v;
    for (v = 0; v < V; ++v)
        if (x[v] > m) m = x[v];
    for (v = 0; v < V; ++v) s += exp(x[v] - m);
    return m + log(s);
}

/*
 * Log-prob of the target and entropy of softmax(z/tau) for the rows
 * rows[0..n) of h (indices into h; duplicates allowed).  targets is indexed
 * by the original h row.  Any of the four outputs may be NULL.
 * Returns 0, or -1 on an out-of-range row or target (outputs for that row
 * are NaN and the scan continues).
 */
int orc_logprob_entropy(int64_t H, int64_t V,
                        const void *h, int htype, int64_t ld_h,
                        const void *W, int wtype, int64_t ld_w,
                        const int64_t *rows, int64_t n, int64_t T,
                        const int64_t *targets, double tau,
                        double *logp, double *ent, double *lse_out, double *ez_out)
{
    int rc = 0;
    int64_t i0;
    double *hd = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *z = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    if (!hd || !z) { free(hd); free(z); return -2; }
    for (i0 = 0; i0 < n; i0 += ORC_ROW_BLOCK) {
        int64_t nb = n - i0 < ORC_ROW_BLOCK ? n - i0 : ORC_ROW_BLOCK;
        int64_t b;
        int bad_row = 0;
        for (b = 0; b < nb; ++b)
            if (rows[i0 + b] < 0 || rows[i0 + b] >= T) bad_row = 1;
        if (bad_row) {
            /* Keep the plain path simple: score valid rows one at a time. */
            for (b = 0; b < nb; ++b) {
                int64_t i = i0 + b;
                if (rows[i] < 0 || rows[i] >= T) {
                    if (logp) logp[i] = NAN;
                    if (ent) ent[i] = NAN;
                    if (lse_out) lse_out[i] = NAN;
                    if (ez_out) ez_out[i] = NAN;
                    rc = -1;
                } else {
                    int r = orc_logprob_entropy(H, V, h, htype, ld_h, W, wtype, ld_w,
                                                rows + i, 1, T, targets, tau,
                                                logp ? logp + i : NULL, ent ? ent + i : NULL,
                                                lse_out ? lse_out + i : NULL,
                                                ez_out ? ez_out + i : NULL);
                    if (r) rc = r;
                }
            }
            continue;
        }
        orc_gather_h(h, htype, ld_h, rows, i0, nb, H, hd);
        orc_logits_block(hd, nb, H, V, W, wtype, ld_w, z);
        for (b = 0; b < nb; ++b) {
            int64_t i = i0 + b, v;
            double *zr = z + b * V;
            double L, ez = 0.0;
            int64_t tgt = targets ? targets[rows[i]] : -1;
            /* upcast first (already float64), then temperature. */
            for (v = 0; v < V; ++v) zr[v] = zr[v] / tau;
            L = orc_lse(zr, V);
            for (v = 0; v < V; ++v) ez += exp(zr[v] - L) * zr[v];
            if (logp) {
                if (tgt >= 0 && tgt < V) logp[i] = zr[tgt] - L;
                else { logp[i] = NAN; rc = -1; }
            }
            if (ent) ent[i] = L - ez;
            if (lse_out) lse_out[i] = L;
            if (ez_out) ez_out[i] = ez;
        }
    }
    free(hd);
    free(z);
    return rc;
}

/*
 * Full-vocabulary KL(teacher || student) per scored row.  Both heads share
 * H and V; the temperature is 1.
 */
int orc_kl(int64_t H, int64_t V,
           const void *h_s, const void *W_s, const void *h_t, const void *W_t,
           int type, int64_t ld_h, int64_t ld_w,
           const int64_t *rows, int64_t n, double *kl)
{
    int64_t i0;
    double *hds = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *hdt = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *zs = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    double *zt = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    if (!hds || !hdt || !zs || !zt) { free(hds); free(hdt); free(zs); free(zt); return -2; }
    for (i0 = 0; i0 < n; i0 += ORC_ROW_BLOCK) {
        int64_t nb = n - i0 < ORC_ROW_BLOCK ? n - i0 : ORC_ROW_BLOCK;
        int64_t b;
        orc_gather_h(h_s, type, ld_h, rows, i0, nb, H, hds);
        orc_gather_h(h_t, type, ld_h, rows, i0, nb, H, hdt);
        orc_logits_block(hds, nb, H, V, W_s, type, ld_w, zs);
        orc_logits_block(hdt, nb, H, V, W_t, type, ld_w, zt);
        for (b = 0; b < nb; ++b) {
            const double *s = zs + b * V, *t = zt + b * V;
            double Ls = orc_lse(s, V), Lt = orc_lse(t, V), acc = 0.0;
            int64_t v;
            for (v = 0; v < V; ++v) {
                double lpt = t[v] - Lt, lps = s[v] - Ls;
                acc += exp(lpt) * (lpt - lps);
            }
            kl[i0 + b] = acc;
        }
    }
    free(hds); free(hdt); free(zs); free(zt);
    return 0;
}

/*
 * Backward of L = sum_i g1[i] logp[i] + g2[i] ent[i] over the scored rows
 * rows[0..n).
 *   dh_rows (n x H, float64) receives sum_v G_iv W[v,:] for scored position
 *     i; the caller scatters it to h row rows[i] (adding duplicates).
 *   dW_sel (nv x H, float64) receives dW[vsel[j],:] = sum_i G_i,vsel[j] h[rows[i],:]
 *     for the nv selected vocab rows (vsel may be NULL with nv = V for all).
 * Either output may be NULL.  Caller zero-fills dW_sel.
 */
int orc_backward(int64_t H, int64_t V,
                 const void *h, int htype, int64_t ld_h,
                 const void *W, int wtype, int64_t ld_w,
                 const int64_t *rows, int64_t n, int64_t T,
                 const int64_t *targets, double tau,
                 const double *g1, const double *g2,
                 double *dh_rows, const int64_t *vsel, int64_t nv, double *dW_sel)
{
    int64_t i0;
    double *hd = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *z = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    if (!hd || !z) { free(hd); free(z); return -2; }
    for (i0 = 0; i0 < n; i0 += ORC_ROW_BLOCK) {
        int64_t nb = n - i0 < ORC_ROW_BLOCK ? n - i0 : ORC_ROW_BLOCK;
        int64_t b;
        for (b = 0; b < nb; ++b)
            if (rows[i0 + b] < 0 || rows[i0 + b] >= T) { free(hd); free(z); return -1; }
        orc_gather_h(h, htype, ld_h, rows, i0, nb, H, hd);
        orc_logits_block(hd, nb, H, V, W, wtype, ld_w, z);
        /* z row b becomes the gradient row G_b in place. */
        for (b = 0; b < nb; ++b) {
            int64_t i = i0 + b, v;
            double *zr = z + b * V;
            double L, ez = 0.0;
            int64_t tgt = targets[rows[i]];
            if (tgt < 0 || tgt >= V) { free(hd); free(z); return -1; }
            for (v = 0; v < V; ++v) zr[v] = zr[v] / tau;
            L = orc_lse(zr, V);
            for (v = 0; v < V; ++v) ez += exp(zr[v] - L) * zr[v];
            for (v = 0; v < V; ++v) {
                double p = exp(zr[v] - L);
                double onehot = (v == tgt) ? 1.0 : 0.0;
                zr[v] = (g1[i] * (onehot - p) - g2[i] * p * (zr[v] - ez)) / tau;
            }
        }
        if (dh_rows) {
            /* dh_rows[i] = sum_v G_iv W[v,:]; threads own slices of the
             * hidden dimension so each W element is decoded once. */
            int64_t k0, k;
            double *acc = (double *)calloc((size_t)nb * H, sizeof(double));
#pragma omp parallel for schedule(static)
            for (k0 = 0; k0 < H; k0 += 64) {
                int64_t kn = H - k0 < 64 ? H - k0 : 64, v, bb, kk;
                double wseg[64];
                for (v = 0; v < V; ++v) {
                    orc_decode(W, wtype, v * ld_w + k0, kn, wseg);
                    for (bb = 0; bb < nb; ++bb) {
                        double g = z[bb * V + v];
                        double *a = acc + bb * H + k0;
                        for (kk = 0; kk < kn; ++kk) a[kk] += g * wseg[kk];
                    }
                }
            }
            for (b = 0; b < nb; ++b)
                for (k = 0; k < H; ++k) dh_rows[(i0 + b) * H + k] = acc[b * H + k];
            free(acc);
        }
        if (dW_sel) {
            int64_t j;
#pragma omp parallel for schedule(static)
            for (j = 0; j < nv; ++j) {
                int64_t v = vsel ? vsel[j] : j, bb, k;
                for (bb = 0; bb < nb; ++bb) {
                    double g = z[bb * V + v];
                    const double *hr = hd + bb * H;
                    for (k = 0; k < H; ++k) dW_sel[j * H + k] += g * hr[k];
                }
            }
        }
    }
    free(hd); free(z);
    return 0;
}

/*
 * K target tokens per scored row (score centering's K-candidate scoring,
 * miles PR #4645, "Scope": "K targets per row"): logp[i*K + k] =
 * z'_{targets[rows[i]*K + k]} - LSE for k < K, with the entropy, LSE and E[z']
 * of the row as in orc_logprob_entropy.  targets is [T, K] row-major.
 * Returns 0, or -1 if any row or target is out of range (NaN written there).
 */
int orc_logprob_k(int64_t H, int64_t V,
                  const void *h, int htype, int64_t ld_h,
                  const void *W, int wtype, int64_t ld_w,
                  const int64_t *rows, int64_t n, int64_t T,
                  const int64_t *targets, int64_t K, double tau,
                  double *logp, double *ent, double *lse_out)
{
    int rc = 0;
    int64_t i0;
    double *hd = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *z = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    if (!hd || !z) { free(hd); free(z); return -2; }
    for (i0 = 0; i0 < n; i0 += ORC_ROW_BLOCK) {
        int64_t nb = n - i0 < ORC_ROW_BLOCK ? n - i0 : ORC_ROW_BLOCK;
        int64_t b, k;
        for (b = 0; b < nb; ++b)
            if (rows[i0 + b] < 0 || rows[i0 + b] >= T) { free(hd); free(z); return -1; }
        orc_gather_h(h, htype, ld_h, rows, i0, nb, H, hd);
        orc_logits_block(hd, nb, H, V, W, wtype, ld_w, z);
        for (b = 0; b < nb; ++b) {
            int64_t i = i0 + b, v;
            double *zr = z + b * V;
            double L, ez = 0.0;
            for (v = 0; v < V; ++v) zr[v] = zr[v] / tau;
            L = orc_lse(zr, V);
            for (v = 0; v < V; ++v) ez += exp(zr[v] - L) * zr[v];
            for (k = 0; k < K; ++k) {
                int64_t t = targets[rows[i] * K + k];
                if (t >= 0 && t < V) logp[i * K + k] = zr[t] - L;
                else { logp[i * K + k] = NAN; rc = -1; }
            }
            if (ent) ent[i] = L - ez;
            if (lse_out) lse_out[i] = L;
        }
    }
    free(hd);
    free(z);
    return rc;
}

/*
 * Sampling-support restriction (miles PR #2764 summary, math_utils.py
 * snippet: calculate_log_probs_and_entropy's sampling_mask, cut into row
 * chunks together with the logits and the tokens).  Read as: the log-prob
 * and entropy are those of the sampling distribution, softmax(z') restricted
 * to the row's support S and renormalised; off S, p_v = 0.
 *
 * support is a bitmask of uint32 words, [T, ld_s], indexed by the original h
 * row like the targets: token v is in row r's support iff bit (v % 32) of
 * word support[r * ld_s + v / 32] is set.
 */
static int orc_in_support(const uint32_t *srow, int64_t v)
{
    return (int)((srow[v / 32] >> (v % 32)) & 1u);
}

/* log sum_{v in S} exp(x_v), two passes; -inf for an empty S. */
static double orc_lse_support(const double *x, int64_t V, const uint32_t *srow)
{
    double m = -INFINITY, s = 0.0;
    int64_t v;
    for (v = 0; v < V; ++v)
        if (orc_in_support(srow, v) && x[v] > m) m = x[v];
    if (m == -INFINITY) return -INFINITY;
    for (v = 0; v < V; ++v)
        if (orc_in_support(srow, v)) s += exp(x[v] - m);
    return m + log(s);
}

/*
 * Per scored row, over the support S:
 *   LSE_S = log sum_{v in S} exp(z'_v),   p_v = exp(z'_v - LSE_S) on S
 *   logp  = z'_tgt - LSE_S if tgt is in S, -inf if it is not
 *   ent   = LSE_S - sum_{v in S} p_v z'_v,  ez = sum_{v in S} p_v z'_v
 * A row with an empty support, an out-of-range row or an out-of-range target
 * gives NaN (the target: logp only) and rc -1.
 */
int orc_logprob_entropy_support(int64_t H, int64_t V,
                                const void *h, int htype, int64_t ld_h,
                                const void *W, int wtype, int64_t ld_w,
                                const int64_t *rows, int64_t n, int64_t T,
                                const int64_t *targets, const uint32_t *support,
                                int64_t ld_s, double tau,
                                double *logp, double *ent, double *lse_out, double *ez_out)
{
    int rc = 0;
    int64_t i;
    double *hd = (double *)malloc((size_t)H * sizeof(double));
    double *z = (double *)malloc((size_t)V * sizeof(double));
    if (!hd || !z) { free(hd); free(z); return -2; }
    for (i = 0; i < n; ++i) {
        int64_t r = rows[i], v, tgt;
        const uint32_t *srow;
        double L, ez = 0.0;
        if (r < 0 || r >= T) {
            logp[i] = ent[i] = NAN;
            if (lse_out) lse_out[i] = NAN;
            if (ez_out) ez_out[i] = NAN;
            rc = -1;
            continue;
        }
        srow = support + r * ld_s;
        orc_decode(h, htype, r * ld_h, H, hd);
        orc_logits_block(hd, 1, H, V, W, wtype, ld_w, z);
        for (v = 0; v < V; ++v) z[v] = z[v] / tau;
        L = orc_lse_support(z, V, srow);
        if (L == -INFINITY) {
            logp[i] = ent[i] = NAN;
            if (lse_out) lse_out[i] = NAN;
            if (ez_out) ez_out[i] = NAN;
            rc = -1;
            continue;
        }
        for (v = 0; v < V; ++v)
            if (orc_in_support(srow, v)) ez += exp(z[v] - L) * z[v];
        tgt = targets[r];
        if (tgt < 0 || tgt >= V) { logp[i] = NAN; rc = -1; }
        else logp[i] = orc_in_support(srow, tgt) ? z[tgt] - L : -INFINITY;
        ent[i] = L - ez;
        if (lse_out) lse_out[i] = L;
        if (ez_out) ez_out[i] = ez;
    }
    free(hd);
    free(z);
    return rc;
}

/*
 * Backward of L = sum_i g1[i] logp[i] + g2[i] ent[i] with the support
 * restriction above.  On S the gradient with respect to z is the unrestricted
 * formula with p and E z' taken over S; off S it is 0:
 *   G_v = 1[v in S] (g1 (1[v=tgt] - p_v) - g2 p_v (z'_v - Ez')) / tau
 * (a target outside S contributes no one-hot term, since G vanishes off S).
 * Outputs as in orc_backward; rows must be valid with non-empty supports
 * (rc -1 otherwise).
 */
int orc_backward_support(int64_t H, int64_t V,
                         const void *h, int htype, int64_t ld_h,
                         const void *W, int wtype, int64_t ld_w,
                         const int64_t *rows, int64_t n, int64_t T,
                         const int64_t *targets, const uint32_t *support, int64_t ld_s,
                         double tau, const double *g1, const double *g2,
                         double *dh_rows, const int64_t *vsel, int64_t nv, double *dW_sel)
{
    int64_t i;
    double *hd = (double *)malloc((size_t)H * sizeof(double));
    double *z = (double *)malloc((size_t)V * sizeof(double));
    double *wd = (double *)malloc((size_t)H * sizeof(double));
    if (!hd || !z || !wd) { free(hd); free(z); free(wd); return -2; }
    for (i = 0; i < n; ++i) {
        int64_t r = rows[i], v, k, j, tgt;
        const uint32_t *srow;
        double L, ez = 0.0;
        if (r < 0 || r >= T) { free(hd); free(z); free(wd); return -1; }
        tgt = targets[r];
        if (tgt < 0 || tgt >= V) { free(hd); free(z); free(wd); return -1; }
        srow = support + r * ld_s;
        orc_decode(h, htype, r * ld_h, H, hd);
        orc_logits_block(hd, 1, H, V, W, wtype, ld_w, z);
        for (v = 0; v < V; ++v) z[v] = z[v] / tau;
        L = orc_lse_support(z, V, srow);
        if (L == -INFINITY) { free(hd); free(z); free(wd); return -1; }
        for (v = 0; v < V; ++v)
            if (orc_in_support(srow, v)) ez += exp(z[v] - L) * z[v];
        /* z becomes the gradient row G in place. */
        for (v = 0; v < V; ++v) {
            if (orc_in_support(srow, v)) {
                double p = exp(z[v] - L);
                double onehot = (v == tgt) ? 1.0 : 0.0;
                z[v] = (g1[i] * (onehot - p) - g2[i] * p * (z[v] - ez)) / tau;
            } else {
                z[v] = 0.0;
            }
        }
        if (dh_rows) {
            double *d = dh_rows + i * H;
            for (k = 0; k < H; ++k) d[k] = 0.0;
            for (v = 0; v < V; ++v) {
                if (z[v] == 0.0) continue;
                orc_decode(W, wtype, v * ld_w, H, wd);
                for (k = 0; k < H; ++k) d[k] += z[v] * wd[k];
            }
        }
        if (dW_sel) {
            for (j = 0; j < nv; ++j) {
                double g = z[vsel ? vsel[j] : j];
                for (k = 0; k < H; ++k) dW_sel[j * H + k] += g * hd[k];
            }
        }
    }
    free(hd); free(z); free(wd);
    return 0;
}

/*
 * MXFP4 quantisation of W [V, H] (bf16/fp16/f64), OCP Microscaling rule, per
 * 32 consecutive elements x_0..x_31 of a row:
 *   e = floor(log2(max |x_i|)) - 2   (2 = exponent of E2M1's largest value, 6)
 *   scale code = e + 127, clamped to [0, 254]; all-zero block: code 0
 *   element = the E2M1 value nearest to x_i / 2^(code - 127), ties to the
 *             even code (mantissa bit 0), magnitudes above 6 saturated to 6;
 *             a zero magnitude is stored as +0 (code 0).
 * Output in the blocked layout of orc_mx_matrix, V_pad >= V rows (rows past V
 * are zero).  H must be a multiple of 64.
 */
int orc_mxfp4_quantize(const void *W, int wtype, int64_t V, int64_t H, int64_t ld_w,
                       int64_t V_pad, uint8_t *packed, uint8_t *scales)
{
    int64_t v, k0, i;
    double x[32];
    if (H % 64 != 0 || V_pad < V) return -1;
    memset(packed, 0, (size_t)(H / 64) * V_pad * 32);
    memset(scales, 0, (size_t)(H / 64) * V_pad * 2);
    for (v = 0; v < V; ++v) {
        for (k0 = 0; k0 < H; k0 += 32) {
            double amax = 0.0, unit;
            int code = 0, fe;
            int64_t blk = (k0 / 64) * V_pad + v;
            orc_decode(W, wtype, v * ld_w + k0, 32, x);
            for (i = 0; i < 32; ++i)
                if (fabs(x[i]) > amax) amax = fabs(x[i]);
            if (amax > 0.0) {
                frexp(amax, &fe);          /* amax = f 2^fe, f in [0.5, 1) */
                code = (fe - 1) - 2 + 127;
                if (code < 0) code = 0;
                if (code > 254) code = 254;
            }
            scales[blk * 2 + (k0 % 64) / 32] = (uint8_t)code;
            unit = ldexp(1.0, code - 127);
            for (i = 0; i < 32; ++i) {
                double a = fabs(x[i]) / unit, best = 1e300;
                int c, q = 0;
                for (c = 0; c < 8; ++c) {   /* nearest magnitude, ties to the even code */
                    double d = fabs(a - orc_e2m1_mag[c]);
                    if (d < best || (d == best && (c % 2) == 0)) { best = d; q = c; }
                }
                if (a > 6.0) q = 7;
                if (q != 0 && x[i] < 0) q |= 8;
                {
                    int64_t byte = blk * 32 + ((k0 % 64) + i) / 2;
                    packed[byte] |= (uint8_t)(((k0 + i) % 2) ? (q << 4) : q);
                }
            }
        }
    }
    return 0;
}

/* Decoded values of an MXFP4 matrix: out [V, H] float64. */
void orc_mxfp4_dequantize(const uint8_t *packed, const uint8_t *scales, int64_t V, int64_t H,
                          int64_t V_pad, double *out)
{
    orc_mx_matrix m;
    int64_t v;
    m.packed = packed; m.scales = scales; m.V_pad = V_pad; m.H = H;
    for (v = 0; v < V; ++v) orc_decode(&m, ORC_MXFP4, v * H, H, out + v * H);
}

/*
 * KL(teacher || student) with the teacher head in MXFP4 (DeepSeek-V4 book
 * ch. 19, "1. FP4 in OPD": inference-only teacher forwards use 4-bit MXFP4
 * weights): exactly orc_kl with W_t replaced by its decoded values.
 * h_s, W_s, h_t share `type` and strides; W_t is the MXFP4 matrix.
 */
int orc_kl_mxfp4(int64_t H, int64_t V,
                 const void *h_s, const void *W_s, const void *h_t,
                 const uint8_t *Wt_packed, const uint8_t *Wt_scales, int64_t V_pad,
                 int type, int64_t ld_h, int64_t ld_w,
                 const int64_t *rows, int64_t n, double *kl)
{
    int64_t i0;
    orc_mx_matrix wt;
    double *hds = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *hdt = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *zs = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    double *zt = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    if (!hds || !hdt || !zs || !zt) { free(hds); free(hdt); free(zs); free(zt); return -2; }
    wt.packed = Wt_packed; wt.scales = Wt_scales; wt.V_pad = V_pad; wt.H = H;
    for (i0 = 0; i0 < n; i0 += ORC_ROW_BLOCK) {
        int64_t nb = n - i0 < ORC_ROW_BLOCK ? n - i0 : ORC_ROW_BLOCK;
        int64_t b;
        orc_gather_h(h_s, type, ld_h, rows, i0, nb, H, hds);
        orc_gather_h(h_t, type, ld_h, rows, i0, nb, H, hdt);
        orc_logits_block(hds, nb, H, V, W_s, type, ld_w, zs);
        orc_logits_block(hdt, nb, H, V, &wt, ORC_MXFP4, H, zt);
        for (b = 0; b < nb; ++b) {
            const double *s = zs + b * V, *t = zt + b * V;
            double Ls = orc_lse(s, V), Lt = orc_lse(t, V), acc = 0.0;
            int64_t v;
            for (v = 0; v < V; ++v) {
                double lpt = t[v] - Lt, lps = s[v] - Ls;
                acc += exp(lpt) * (lpt - lps);
            }
            kl[i0 + b] = acc;
        }
    }
    free(hds); free(hdt); free(zs); free(zt);
    return 0;
}


/*
 * OCP Microscaling MXFP8 with E4M3 elements: the format the teacher hidden
 * states take on the block-scaled tensor-core path, beside the MXFP4
 * teacher head (DeepSeek-V4 book ch. 19, "1. FP4 in OPD": the teacher's
 * inference-only forward runs in native low precision; the block-scaled
 * MMA needs both of its operands in a microscaling format).
 *   E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent field
 *   0 is subnormal: (m / 8) 2^-6.  Codes 0x7F and 0xFF are NaN, so the
 *   largest finite value is 0x7E = 1.75 * 2^8 = 448.
 * Per 32 consecutive elements x_0..x_31 of a row:
 *   scale code = floor(log2(max |x_i|)) - 8 + 127 (8 = exponent of 448),
 *                clamped to [0, 254]; all-zero block: code 0
 *   element    = the finite E4M3 value nearest to x_i / 2^(code - 127), ties
 *                to the even code (mantissa bit 0 clear), magnitudes above 448
 *                saturated to 448; a zero result is stored as +0 (code 0).
 */
static double orc_e4m3(int c)
{
    int e = (c >> 3) & 15, m = c & 7;
    double v = e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m / 8.0, -6);
    if ((c & 0x7F) == 0x7F) return NAN;
    return (c & 0x80) ? -v : v;
}

double orc_e4m3_value(int code) { return orc_e4m3(code & 0xFF); }

/* One block of 32 values -> 32 E4M3 codes and the scale code. */
static void orc_mxfp8_block(const double *x, uint8_t *codes, uint8_t *scale)
{
    double amax = 0.0, unit;
    int code = 0, fe, i;
    for (i = 0; i < 32; ++i)
        if (fabs(x[i]) > amax) amax = fabs(x[i]);
    if (amax > 0.0) {
        frexp(amax, &fe);                  /* amax = f 2^fe, f in [0.5, 1) */
        code = (fe - 1) - 8 + 127;
        if (code < 0) code = 0;
        if (code > 254) code = 254;
    }
    *scale = (uint8_t)code;
    unit = ldexp(1.0, code - 127);
    for (i = 0; i < 32; ++i) {
        double a = fabs(x[i]) / unit, best = 1e300;
        int c, q = 0;
        for (c = 0; c <= 0x7E; ++c) {     /* nearest finite magnitude, ties to the even code */
            double d = fabs(a - orc_e4m3(c));
            if (d < best || (d == best && (c % 2) == 0)) { best = d; q = c; }
        }
        if (a > 448.0) q = 0x7E;
        if (q != 0 && x[i] < 0) q |= 0x80;
        codes[i] = (uint8_t)q;
    }
}

/*
 * MXFP8 quantisation of X [R, H] (bf16/fp16/f64, row stride ld), H a
 * multiple of 32: codes [R, H] row-major, scales [R, H / 32].
 */
int orc_mxfp8_quantize(const void *X, int xtype, int64_t R, int64_t H, int64_t ld,
                       uint8_t *codes, uint8_t *scales)
{
    int64_t r, k0;
    double x[32];
    if (H % 32 != 0) return -1;
    for (r = 0; r < R; ++r)
        for (k0 = 0; k0 < H; k0 += 32) {
            orc_decode(X, xtype, r * ld + k0, 32, x);
            orc_mxfp8_block(x, codes + r * H + k0, scales + r * (H / 32) + k0 / 32);
        }
    return 0;
}

/* Decoded values of an MXFP8 matrix: out [R, H] float64. */
void orc_mxfp8_dequantize(const uint8_t *codes, const uint8_t *scales, int64_t R, int64_t H,
                          double *out)
{
    int64_t r, k;
    for (r = 0; r < R; ++r)
        for (k = 0; k < H; ++k)
            out[r * H + k] = ldexp(orc_e4m3(codes[r * H + k]), (int)scales[r * (H / 32) + k / 32] - 127);
}

/*
 * KL(teacher || student) on the block-scaled teacher path: as orc_kl_mxfp4
 * (teacher head W_t in MXFP4, blocked layout), with each teacher hidden row
 * h_t[r] first quantised to MXFP8 by the rule above; the teacher logits are
 * the float64 products of the two decoded operands.  The student is exact
 * (bf16 h_s and W_s).  H a multiple of 64.
 */
int orc_kl_mx(int64_t H, int64_t V,
              const void *h_s, const void *W_s, const void *h_t,
              const uint8_t *Wt_packed, const uint8_t *Wt_scales, int64_t V_pad,
              int type, int64_t ld_h, int64_t ld_w,
              const int64_t *rows, int64_t n, double *kl)
{
    int64_t i0;
    orc_mx_matrix wt;
    double *hds = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *hdt = (double *)malloc((size_t)ORC_ROW_BLOCK * H * sizeof(double));
    double *zs = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    double *zt = (double *)malloc((size_t)ORC_ROW_BLOCK * V * sizeof(double));
    if (!hds || !hdt || !zs || !zt) { free(hds); free(hdt); free(zs); free(zt); return -2; }
    wt.packed = Wt_packed; wt.scales = Wt_scales; wt.V_pad = V_pad; wt.H = H;
    for (i0 = 0; i0 < n; i0 += ORC_ROW_BLOCK) {
        int64_t nb = n - i0 < ORC_ROW_BLOCK ? n - i0 : ORC_ROW_BLOCK;
        int64_t b, k0;
        orc_gather_h(h_s, type, ld_h, rows, i0, nb, H, hds);
        orc_gather_h(h_t, type, ld_h, rows, i0, nb, H, hdt);
        for (b = 0; b < nb; ++b)            /* h_t rows -> their MXFP8 values */
            for (k0 = 0; k0 < H; k0 += 32) {
                uint8_t c[32], sc;
                int i;
                double *x = hdt + b * H + k0;
                orc_mxfp8_block(x, c, &sc);
                for (i = 0; i < 32; ++i) x[i] = ldexp(orc_e4m3(c[i]), (int)sc - 127);
            }
        orc_logits_block(hds, nb, H, V, W_s, type, ld_w, zs);
        orc_logits_block(hdt, nb, H, V, &wt, ORC_MXFP4, H, zt);
        for (b = 0; b < nb; ++b) {
            const double *s = zs + b * V, *t = zt + b * V;
            double Ls = orc_lse(s, V), Lt = orc_lse(t, V), acc = 0.0;
            int64_t v;
            for (v = 0; v < V; ++v) {
                double lpt = t[v] - Lt, lps = s[v] - Ls;
                acc += exp(lpt) * (lpt - lps);
            }
            kl[i0 + b] = acc;
        }
    }
    free(hds); free(hdt); free(zs); free(zt);
    return 0;
}

/*
 * Log-prob and entropy on the block-scaled path (DeepSeek-V4 book ch. 19,
 * "1. FP4 in OPD": every forward that needs no backward -- among them the
 * reference model's log-probs for the KL baseline -- runs in native 4-bit
 * precision).  The head W is MXFP4 in the blocked layout of orc_kl_mxfp4,
 * and each scored row h[rows[i]] is first quantised to MXFP8 by
 * orc_mxfp8_block; z is the float64 product of the two decoded operands,
 * and logp, entropy, LSE and E[z'] follow as in orc_logprob_entropy.
 * H a multiple of 64.  Bad rows and targets give NaN as there (return -1).
 */
int orc_logprob_entropy_mx(int64_t H, int64_t V,
                           const void *h, int htype, int64_t ld_h,
                           const uint8_t *W_packed, const uint8_t *W_scales, int64_t V_pad,
                           const int64_t *rows, int64_t n, int64_t T,
                           const int64_t *targets, double tau,
                           double *logp, double *ent, double *lse_out, double *ez_out)
{
    int64_t i, k0;
    int rc;
    orc_mx_matrix w;
    double *hq = (double *)malloc((size_t)(n > 0 ? n : 1) * H * sizeof(double));
    int64_t *r2 = (int64_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
    int64_t *tg = (int64_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
    if (!hq || !r2 || !tg) { free(hq); free(r2); free(tg); return -2; }
    /* the scored rows, quantised, become rows 0..n-1 of hq; a bad index stays bad */
    for (i = 0; i < n; ++i) {
        if (rows[i] < 0 || rows[i] >= T) { r2[i] = -1; tg[i] = 0; continue; }
        r2[i] = i;
        tg[i] = targets[rows[i]];
        orc_decode(h, htype, rows[i] * ld_h, H, hq + i * H);
        for (k0 = 0; k0 < H; k0 += 32) {
            uint8_t c[32], sc;
            int j;
            double *x = hq + i * H + k0;
            orc_mxfp8_block(x, c, &sc);
            for (j = 0; j < 32; ++j) x[j] = ldexp(orc_e4m3(c[j]), (int)sc - 127);
        }
    }
    w.packed = W_packed; w.scales = W_scales; w.V_pad = V_pad; w.H = H;
    rc = orc_logprob_entropy(H, V, hq, ORC_F64, H, &w, ORC_MXFP4, H, r2, n, n, tg, tau,
                             logp, ent, lse_out, ez_out);
    free(hq); free(r2); free(tg);
    return rc;
}
