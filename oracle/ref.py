"""NumPy float64 restatement of the oracle.

Test infrastructure only (see the package docstring).  Independent of
``oracle.c``: its own decoding of the storage formats, its own two-pass
log-sum-exp, with ``numpy.matmul`` (float64 BLAS) as the one library step
for the logits.  Used to cross-check the C oracle and for the large
full-vocabulary passes that the C loops are too slow for (the per-row
statistics every dW element depends on).

Definitions: miles PR #2764 summary (prhub), "Implementation breakdown"
item 2 and its math_utils.py snippet (upcast, then divide by the
temperature); miles PR #4645, "How it works" (scored rows only, log-prob
and entropy per row, backward through h and W); DeepSeek-V4 book ch. 19,
"TileLang KL kernel" (exact full-vocabulary KL, read as KL(t || s)).
"""
import numpy as np


def decode(x, dtype):
    """Exact float64 values of a bf16/fp16 bit-pattern array (or a float array)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype in (torch.bfloat16, torch.float16):
                x = x.contiguous().view(torch.int16).numpy().view(np.uint16)
            else:
                x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if dtype == "bf16":
        with np.errstate(invalid="ignore"):   # NaN payloads widen with a warning
            return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "fp16":
        return x.astype(np.uint16).view(np.float16).astype(np.float64)
    return x.astype(np.float64)


def _rows(rows, T):
    return np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)


def _lse(zp):
    """Row-wise log-sum-exp, max shift then sum (two passes)."""
    m = zp.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(zp - m).sum(axis=1, keepdims=True)))[:, 0]


def support_bits(support, rows, V):
    """Boolean [len(rows), V] membership from a uint32 support bitmask [T, ld]
    indexed by h row: token v is in row r's support iff bit v % 32 of word
    v // 32 of row r is set."""
    words = np.ascontiguousarray(np.asarray(support).view(np.uint32)[rows])
    bits = np.unpackbits(words.view(np.uint8), axis=1, bitorder="little")
    return bits[:, :V].astype(bool)


def _lse_on(zp, keep):
    """Row-wise log-sum-exp over the entries where keep is True (-inf if none)."""
    m = np.where(keep, zp, -np.inf).max(axis=1, keepdims=True)
    safe = np.where(np.isfinite(m), m, 0.0)
    s = np.where(keep, np.exp(np.where(keep, zp, safe) - safe), 0.0).sum(axis=1, keepdims=True)
    with np.errstate(divide="ignore"):
        return np.where(s[:, 0] > 0, safe[:, 0] + np.log(s[:, 0]), -np.inf)


def row_stats(hd, Wd, rows, tau, block=256, support=None):
    """lse and Ez' = sum_v p_v z'_v per scored row, from decoded float64 h, W.
    With a support bitmask, both are taken over each row's support (p = 0 off
    it); an empty support gives NaN."""
    rows = _rows(rows, hd.shape[0])
    lse = np.empty(rows.shape[0])
    ez = np.empty(rows.shape[0])
    for i0 in range(0, rows.shape[0], block):
        r = rows[i0:i0 + block]
        zp = (hd[r] @ Wd.T) / tau
        if support is None:
            L = _lse(zp)
            p = np.exp(zp - L[:, None])
        else:
            keep = support_bits(support, r, Wd.shape[0])
            L = _lse_on(zp, keep)
            with np.errstate(invalid="ignore"):
                p = np.where(keep, np.exp(np.where(keep, zp, 0.0) - L[:, None]), 0.0)
            L = np.where(np.isfinite(L), L, np.nan)
        lse[i0:i0 + block] = L
        ez[i0:i0 + block] = (p * zp).sum(axis=1) + 0.0 * L
    return lse, ez


def logprob_entropy(h, W, targets, rows, tau, dtype, block=256, support=None):
    """logp, ent, lse, ez per scored row.  With ``support`` (uint32 bitmask
    [T, ld] by h row) the distribution is softmax(z') restricted to the row's
    support and renormalised (math_utils.py's sampling_mask); a target off
    the support has logp = -inf."""
    hd, Wd = decode(h, dtype), decode(W, dtype)
    rows = _rows(rows, hd.shape[0])
    tg = np.asarray(targets, dtype=np.int64)[rows]
    lse, ez = row_stats(hd, Wd, rows, tau, block, support)
    zt = np.einsum("ik,ik->i", hd[rows], Wd[tg]) / tau
    logp = zt - lse
    if support is not None:
        on = support_bits(support, rows, Wd.shape[0])[np.arange(rows.shape[0]), tg]
        logp = np.where(on | np.isnan(lse), logp, -np.inf)
    return {"logp": logp, "ent": lse - ez, "lse": lse, "ez": ez}


def kl(h_s, W_s, h_t, W_t, rows, dtype, block=256):
    hs, Ws, ht, Wt = (decode(a, dtype) for a in (h_s, W_s, h_t, W_t))
    rows = _rows(rows, hs.shape[0])
    out = np.empty(rows.shape[0])
    for i0 in range(0, rows.shape[0], block):
        r = rows[i0:i0 + block]
        ls = hs[r] @ Ws.T
        lt = ht[r] @ Wt.T
        ls = ls - _lse(ls)[:, None]
        lt = lt - _lse(lt)[:, None]
        out[i0:i0 + block] = (np.exp(lt) * (lt - ls)).sum(axis=1)
    return out


def grad_logits(zp, tgt, lse, ez, g1, g2, tau, keep=None):
    """dL/dz for L = g1 logp + g2 ent, rows of z' = z/tau (float64).  With a
    support (keep: boolean [rows, V]) the gradient is the same formula on the
    support, with p, lse and ez taken over it, and 0 off it."""
    if keep is not None:
        zp = np.where(keep, zp, lse[:, None])
    p = np.exp(zp - lse[:, None])
    onehot = np.zeros_like(zp)
    onehot[np.arange(zp.shape[0]), tgt] = 1.0
    G = (g1[:, None] * (onehot - p) - g2[:, None] * p * (zp - ez[:, None])) / tau
    return G if keep is None else np.where(keep, G, 0.0)


def backward(h, W, targets, rows, tau, g1, g2, dtype, dh_rows_sel=None, vsel=None,
             block=256, stats=None, support=None):
    """Gradients of sum(g1 logp + g2 ent).

    dh_rows_sel: positions i (into rows) whose dh rows to return (default all).
    vsel: vocabulary rows of dW to return (default all).  dW needs every
    scored row's statistics, which this computes with a float64 matmul pass
    over the full vocabulary unless ``stats=(lse, ez)`` is supplied (each
    computed by :func:`row_stats`).  ``support``: as in :func:`logprob_entropy`.
    Returns (dh_rows [len(sel),H], dW_sel [len(vsel),H]).
    """
    hd, Wd = decode(h, dtype), decode(W, dtype)
    rows = _rows(rows, hd.shape[0])
    n = rows.shape[0]
    g1 = np.asarray(g1, dtype=np.float64)
    g2 = np.asarray(g2, dtype=np.float64)
    tg = np.asarray(targets, dtype=np.int64)[rows]
    sel = np.arange(n) if dh_rows_sel is None else np.asarray(dh_rows_sel, dtype=np.int64)
    vs = np.arange(Wd.shape[0]) if vsel is None else np.asarray(vsel, dtype=np.int64)

    # dh rows: only the selected positions' statistics are needed.
    dh = np.empty((sel.shape[0], hd.shape[1]))
    for i0 in range(0, sel.shape[0], block):
        s = sel[i0:i0 + block]
        zp = (hd[rows[s]] @ Wd.T) / tau
        keep = None if support is None else support_bits(support, rows[s], Wd.shape[0])
        if keep is None:
            L = _lse(zp)
            ez = (np.exp(zp - L[:, None]) * zp).sum(axis=1)
        else:
            L = _lse_on(zp, keep)
            ez = np.where(keep, np.exp(np.where(keep, zp, L[:, None]) - L[:, None]) * zp,
                          0.0).sum(axis=1)
        G = grad_logits(zp, tg[s], L, ez, g1[s], g2[s], tau, keep)
        dh[i0:i0 + block] = G @ Wd

    # dW rows: every scored row contributes to every vocabulary row.
    lse, ez = stats if stats is not None else row_stats(hd, Wd, rows, tau, block, support)
    zp = (hd[rows] @ Wd[vs].T) / tau                       # [n, len(vs)]
    p = np.exp(zp - lse[:, None])
    onehot = (tg[:, None] == vs[None, :]).astype(np.float64)
    G = (g1[:, None] * (onehot - p) - g2[:, None] * p * (zp - ez[:, None])) / tau
    if support is not None:
        G = np.where(support_bits(support, rows, Wd.shape[0])[:, vs], G, 0.0)
    dW = G.T @ hd[rows]
    return dh, dW


# ---------------------------------------------------------------- MXFP4
# OCP Microscaling FP4: E2M1 elements (1 sign, 2 exponent bits with bias 1, 1
# mantissa bit) with one E8M0 power-of-two scale per 32 consecutive elements
# of a row.  Blocked layout: for column block kb (64 wide) and row v < V_pad,
# packed[kb, v, b] holds elements 2b (low nibble) and 2b+1 (high nibble),
# scales[kb, v, j] the code of elements 32j .. 32j+31 of the block.

def mxfp4_vpad(V):
    return -(-V // 256) * 256


def mxfp4_quantize(W, dtype):
    """(packed uint8 [H/64, V_pad, 32], scales uint8 [H/64, V_pad, 2]).

    Restated independently of the C quantiser: the scale exponent from
    numpy.frexp, the rounding as numpy.rint (ties to even) in units of the
    grid spacing of the octave the value falls in (0.5 below 2, 1 in [2, 4),
    2 from 4), saturation at 6."""
    x = decode(W, dtype)
    V, H = x.shape
    assert H % 64 == 0
    Vp = mxfp4_vpad(V)
    blocks = x.reshape(V, H // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    _, fe = np.frexp(amax)
    code = np.where(amax > 0, np.clip(fe - 1 - 2 + 127, 0, 254), 0).astype(np.int64)
    a = np.abs(blocks) / np.ldexp(1.0, code - 127)[:, :, None]
    spacing = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    q = np.minimum(np.rint(a / spacing) * spacing, 6.0)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    idx = np.searchsorted(mags, q)
    assert np.all(mags[idx] == q)
    nib = np.where((blocks < 0) & (idx > 0), idx | 8, idx).reshape(V, H)
    packed = np.zeros((H // 64, Vp, 32), np.uint8)
    pairs = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8).reshape(V, H // 64, 32)
    packed[:, :V, :] = pairs.transpose(1, 0, 2)
    scales = np.zeros((H // 64, Vp, 2), np.uint8)
    scales[:, :V, :] = code.reshape(V, H // 64, 2).transpose(1, 0, 2)
    return packed, scales


def mxfp4_dequantize(packed, scales, V):
    """Decoded float64 [V, H] of a blocked MXFP4 matrix."""
    packed = np.asarray(packed, np.uint8)
    scales = np.asarray(scales, np.uint8)
    nkb = packed.shape[0]
    lo = (packed[:, :V, :] & 15).astype(np.int64)
    hi = (packed[:, :V, :] >> 4).astype(np.int64)
    nib = np.stack([lo, hi], axis=3).reshape(nkb, V, 64)       # element order within the block
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    val = np.where(nib & 8, -1.0, 1.0) * mags[nib & 7]
    sc = np.repeat(scales[:, :V, :].astype(np.int64), 32, axis=2)  # [nkb, V, 64]
    val = np.ldexp(val, sc - 127)
    return val.transpose(1, 0, 2).reshape(V, nkb * 64)


def kl_mxfp4(h_s, W_s, h_t, packed, scales, rows, dtype, block=256):
    """KL(teacher || student) with the teacher head given in MXFP4."""
    hs, Ws, ht = (decode(a, dtype) for a in (h_s, W_s, h_t))
    Wt = mxfp4_dequantize(packed, scales, Ws.shape[0])
    rows = _rows(rows, hs.shape[0])
    out = np.empty(rows.shape[0])
    for i0 in range(0, rows.shape[0], block):
        r = rows[i0:i0 + block]
        ls = hs[r] @ Ws.T
        lt = ht[r] @ Wt.T
        ls = ls - _lse(ls)[:, None]
        lt = lt - _lse(lt)[:, None]
        out[i0:i0 + block] = (np.exp(lt) * (lt - ls)).sum(axis=1)
    return out


# ---------------------------------------------------------------- MXFP8
# OCP Microscaling MXFP8 with E4M3 elements (1 sign, 4 exponent bits with
# bias 7, 3 mantissa bits; exponent field 0 subnormal; 0x7F NaN, largest
# finite 448) and one E8M0 scale per 32 consecutive elements of a row: the
# teacher hidden states' format on the block-scaled tensor-core path.

def e4m3_values():
    """Float64 values of the 256 E4M3 codes (NaN for 0x7F and 0xFF)."""
    c = np.arange(256)
    e, m = (c >> 3) & 15, c & 7
    v = np.where(e > 0, np.ldexp(1.0 + m / 8.0, e - 7), np.ldexp(m / 8.0, -6))
    v = np.where(c & 0x80, -v, v)
    v[[0x7F, 0xFF]] = np.nan
    return v


def mxfp8_quantize(X, dtype):
    """(codes uint8 [R, H], scales uint8 [R, H/32]).

    Restated independently of the C quantiser: the scale from numpy.frexp;
    the element rounding as numpy.rint (ties to even) in units of the grid
    spacing of the value's octave (2^(e - 3) for a value in [2^e, 2^(e+1)),
    e >= -6, and the subnormal spacing 2^-9 below 2^-6), saturated at 448."""
    x = decode(X, dtype)
    R, H = x.shape
    assert H % 32 == 0
    blocks = x.reshape(R, H // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    _, fe = np.frexp(amax)
    code = np.where(amax > 0, np.clip(fe - 1 - 8 + 127, 0, 254), 0).astype(np.int64)
    a = np.abs(blocks) / np.ldexp(1.0, code - 127)[:, :, None]
    with np.errstate(divide="ignore"):
        oct_e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    spacing = np.where(a >= 2.0 ** -6, np.ldexp(1.0, (np.maximum(oct_e, -6) - 3).astype(np.int64)),
                       2.0 ** -9)
    q = np.minimum(np.rint(a / spacing) * spacing, 448.0)
    vals = e4m3_values()[:0x7F]                       # the non-negative finite codes, ascending
    idx = np.searchsorted(vals, q)
    assert np.all(vals[idx] == q)
    codes = np.where((blocks < 0) & (idx > 0), idx | 0x80, idx).astype(np.uint8).reshape(R, H)
    return codes, code.astype(np.uint8)


def mxfp8_dequantize(codes, scales):
    codes = np.asarray(codes, np.uint8)
    R, H = codes.shape
    sc = np.repeat(np.asarray(scales, np.int64), 32, axis=1)
    return np.ldexp(e4m3_values()[codes], sc - 127)


def kl_mx(h_s, W_s, h_t, packed, scales, rows, dtype, block=256):
    """KL(teacher || student) on the block-scaled teacher path: the teacher
    hidden rows quantised to MXFP8 and the teacher head in MXFP4 (blocked
    layout); the student exact."""
    hs, Ws = decode(h_s, dtype), decode(W_s, dtype)
    Wt = mxfp4_dequantize(packed, scales, Ws.shape[0])
    rows = _rows(rows, hs.shape[0])
    out = np.empty(rows.shape[0])
    for i0 in range(0, rows.shape[0], block):
        r = rows[i0:i0 + block]
        ht = mxfp8_dequantize(*mxfp8_quantize(np.asarray(decode(h_t, dtype))[r], "f64"))
        ls = hs[r] @ Ws.T
        lt = ht @ Wt.T
        ls = ls - _lse(ls)[:, None]
        lt = lt - _lse(lt)[:, None]
        out[i0:i0 + block] = (np.exp(lt) * (lt - ls)).sum(axis=1)
    return out


def logprob_entropy_mx(h, packed, scales, V, targets, rows, tau, dtype, block=256):
    """logp, ent, lse, ez per scored row on the block-scaled path: each scored
    row of h quantised to MXFP8 (mxfp8_quantize above), the head in MXFP4
    (blocked layout, decoded by mxfp4_dequantize)."""
    hd = np.asarray(decode(h, dtype))
    Wd = mxfp4_dequantize(packed, scales, V)
    rows = _rows(rows, hd.shape[0])
    tg = np.asarray(targets, dtype=np.int64)[rows]
    hq = mxfp8_dequantize(*mxfp8_quantize(hd[rows], "f64")) if rows.shape[0] else hd[rows]
    lse, ez = row_stats(hq, Wd, np.arange(rows.shape[0]), tau, block)
    logp = np.einsum("ik,ik->i", hq, Wd[tg]) / tau - lse
    return {"logp": logp, "ent": lse - ez, "lse": lse, "ez": ez}
