"""ctypes wrapper around the C float64 oracle (``oracle.c``).

Test infrastructure only (see the package docstring).  Arrays are handed to
C as their raw storage: bf16/fp16 as uint16 bit patterns, float64 as is.
Torch tensors are accepted and viewed as that storage on the host.
"""
import ctypes

import numpy as np

from .build import build_oracle

_TYPES = {"bf16": 0, "fp16": 1, "f64": 2}
_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build_oracle())
        i64, dbl, vp, ip = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        _lib.orc_logprob_entropy.argtypes = [i64, i64, vp, ip, i64, vp, ip, i64,
                                             vp, i64, i64, vp, dbl, vp, vp, vp, vp]
        _lib.orc_kl.argtypes = [i64, i64, vp, vp, vp, vp, ip, i64, i64, vp, i64, vp]
        _lib.orc_backward.argtypes = [i64, i64, vp, ip, i64, vp, ip, i64, vp, i64, i64,
                                      vp, dbl, vp, vp, vp, vp, i64, vp]
        _lib.orc_decode_array.argtypes = [vp, ip, i64, vp]
        _lib.orc_logprob_k.argtypes = [i64, i64, vp, ip, i64, vp, ip, i64, vp, i64, i64, vp, i64,
                                       dbl, vp, vp, vp]
        _lib.orc_logprob_k.restype = ip
        _lib.orc_logprob_entropy_support.argtypes = [i64, i64, vp, ip, i64, vp, ip, i64, vp, i64,
                                                     i64, vp, vp, i64, dbl, vp, vp, vp, vp]
        _lib.orc_logprob_entropy_support.restype = ip
        _lib.orc_backward_support.argtypes = [i64, i64, vp, ip, i64, vp, ip, i64, vp, i64, i64,
                                              vp, vp, i64, dbl, vp, vp, vp, vp, i64, vp]
        _lib.orc_backward_support.restype = ip
        _lib.orc_mxfp4_quantize.argtypes = [vp, ip, i64, i64, i64, i64, vp, vp]
        _lib.orc_mxfp4_quantize.restype = ip
        _lib.orc_mxfp4_dequantize.argtypes = [vp, vp, i64, i64, i64, vp]
        _lib.orc_kl_mxfp4.argtypes = [i64, i64, vp, vp, vp, vp, vp, i64, ip, i64, i64, vp, i64, vp]
        _lib.orc_kl_mxfp4.restype = ip
        _lib.orc_mxfp8_quantize.argtypes = [vp, ip, i64, i64, i64, vp, vp]
        _lib.orc_mxfp8_quantize.restype = ip
        _lib.orc_mxfp8_dequantize.argtypes = [vp, vp, i64, i64, vp]
        _lib.orc_e4m3_value.argtypes = [ip]
        _lib.orc_e4m3_value.restype = dbl
        _lib.orc_kl_mx.argtypes = [i64, i64, vp, vp, vp, vp, vp, i64, ip, i64, i64, vp, i64, vp]
        _lib.orc_kl_mx.restype = ip
        _lib.orc_logprob_entropy_mx.argtypes = [i64, i64, vp, ip, i64, vp, vp, i64, vp, i64,
                                                i64, vp, dbl, vp, vp, vp, vp]
        _lib.orc_logprob_entropy_mx.restype = ip
        _lib.orc_num_threads.restype = ip
        for f in (_lib.orc_logprob_entropy, _lib.orc_kl, _lib.orc_backward):
            f.restype = ip
    return _lib


def num_threads() -> int:
    return int(lib().orc_num_threads())


def storage(x, dtype):
    """Host storage of a 2-D matrix: (contiguous array, element type code, row stride)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype in (torch.bfloat16, torch.float16):
                x = x.contiguous().view(torch.int16).numpy().view(np.uint16)
            else:
                x = x.contiguous().numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.ascontiguousarray(x)
    if dtype in ("bf16", "fp16"):
        if x.dtype != np.uint16:
            raise TypeError("bf16/fp16 oracle inputs are uint16 bit patterns")
    elif dtype == "f64":
        x = np.ascontiguousarray(x, dtype=np.float64)
    else:
        raise ValueError(dtype)
    return x, _TYPES[dtype], (x.shape[1] if x.ndim == 2 else 1)


def _i64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def decode(bits, dtype):
    """Decode a uint16 bit-pattern array (bf16 or fp16) to float64 with the C decoder."""
    x = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.float64)
    lib().orc_decode_array(x.ctypes.data, _TYPES[dtype], x.size, out.ctypes.data)
    return out


def logprob_entropy(h, W, targets, rows, tau, dtype):
    """Per scored row: logp, ent, lse, ez (float64 arrays of len(rows))."""
    hs, ht, ldh = storage(h, dtype)
    ws, wt, ldw = storage(W, dtype)
    T, H = hs.shape[0], ldh
    V = ws.shape[0]
    rows = _i64(rows if rows is not None else np.arange(T))
    tg = _i64(targets)
    n = rows.shape[0]
    out = {k: np.empty(n, dtype=np.float64) for k in ("logp", "ent", "lse", "ez")}
    rc = lib().orc_logprob_entropy(H, V, hs.ctypes.data, ht, ldh, ws.ctypes.data, wt, ldw,
                                   _ptr(rows), n, T, _ptr(tg), float(tau),
                                   out["logp"].ctypes.data, out["ent"].ctypes.data,
                                   out["lse"].ctypes.data, out["ez"].ctypes.data)
    if rc == -2:
        raise MemoryError("oracle allocation failed")
    out["rc"] = rc
    return out


def kl(h_s, W_s, h_t, W_t, rows, dtype):
    """Per scored row KL(teacher || student), float64."""
    a, ty, ldh = storage(h_s, dtype)
    b, _, ldw = storage(W_s, dtype)
    c, _, _ = storage(h_t, dtype)
    d, _, _ = storage(W_t, dtype)
    T, V = a.shape[0], b.shape[0]
    rows = _i64(rows if rows is not None else np.arange(T))
    out = np.empty(rows.shape[0], dtype=np.float64)
    rc = lib().orc_kl(ldh, V, a.ctypes.data, b.ctypes.data, c.ctypes.data, d.ctypes.data,
                      ty, ldh, ldw, _ptr(rows), rows.shape[0], out.ctypes.data)
    if rc:
        raise RuntimeError("oracle kl failed: %d" % rc)
    return out


def backward(h, W, targets, rows, tau, g1, g2, dtype, want_dh=True, vsel=None,
             want_dw=True):
    """Gradients of sum(g1*logp + g2*ent).

    Returns (dh_rows [n,H] or None, dW_sel [nv,H] or None); dh_rows[i] is the
    gradient contribution of scored position i (to be added at h row rows[i]).
    """
    hs, ht, ldh = storage(h, dtype)
    ws, wt, ldw = storage(W, dtype)
    T, H, V = hs.shape[0], ldh, ws.shape[0]
    rows = _i64(rows if rows is not None else np.arange(T))
    n = rows.shape[0]
    g1 = np.ascontiguousarray(g1, dtype=np.float64)
    g2 = np.ascontiguousarray(g2, dtype=np.float64)
    dh = np.zeros((n, H), dtype=np.float64) if want_dh else None
    vs = None if vsel is None else _i64(vsel)
    nv = V if vs is None else vs.shape[0]
    dW = np.zeros((nv, H), dtype=np.float64) if want_dw else None
    rc = lib().orc_backward(H, V, hs.ctypes.data, ht, ldh, ws.ctypes.data, wt, ldw,
                            _ptr(rows), n, T, _ptr(_i64(targets)), float(tau),
                            g1.ctypes.data, g2.ctypes.data, _ptr(dh), _ptr(vs), nv, _ptr(dW))
    if rc:
        raise RuntimeError("oracle backward failed: %d" % rc)
    return dh, dW


def scatter_rows(dh_rows, rows, T):
    """Add per-position gradient rows into a [T,H] array (duplicates add up)."""
    out = np.zeros((T, dh_rows.shape[1]), dtype=np.float64)
    np.add.at(out, _i64(rows), dh_rows)
    return out


def logprob_k(h, W, targets_tk, rows, tau, dtype):
    """K targets per scored row: logp [n, K], ent [n], lse [n] (float64).
    targets_tk is [T, K] (indexed by h row)."""
    hs, ht, ldh = storage(h, dtype)
    ws, wt, ldw = storage(W, dtype)
    T, H, V = hs.shape[0], ldh, ws.shape[0]
    rows = _i64(rows if rows is not None else np.arange(T))
    tg = _i64(targets_tk)
    K = tg.shape[1]
    n = rows.shape[0]
    logp = np.empty((n, K))
    ent = np.empty(n)
    lse = np.empty(n)
    rc = lib().orc_logprob_k(H, V, hs.ctypes.data, ht, ldh, ws.ctypes.data, wt, ldw, _ptr(rows), n,
                             T, _ptr(tg), K, float(tau), logp.ctypes.data, ent.ctypes.data,
                             lse.ctypes.data)
    if rc == -2:
        raise MemoryError("oracle allocation failed")
    return {"logp": logp, "ent": ent, "lse": lse, "rc": rc}


def _words(support):
    w = np.ascontiguousarray(np.asarray(support).view(np.uint32))
    if w.ndim != 2:
        raise ValueError("support is a [T, ld] array of uint32 words")
    return w, w.shape[1]


def logprob_entropy_support(h, W, targets, rows, support, tau, dtype):
    """Per scored row under the row's sampling support (uint32 bitmask [T, ld]
    by h row): logp (-inf for a target off the support), ent, lse, ez."""
    hs, ht, ldh = storage(h, dtype)
    ws, wt, ldw = storage(W, dtype)
    T, H, V = hs.shape[0], ldh, ws.shape[0]
    rows = _i64(rows if rows is not None else np.arange(T))
    sw, lds = _words(support)
    n = rows.shape[0]
    out = {k: np.empty(n, dtype=np.float64) for k in ("logp", "ent", "lse", "ez")}
    rc = lib().orc_logprob_entropy_support(H, V, hs.ctypes.data, ht, ldh, ws.ctypes.data, wt,
                                           ldw, _ptr(rows), n, T, _ptr(_i64(targets)),
                                           sw.ctypes.data, lds, float(tau),
                                           out["logp"].ctypes.data, out["ent"].ctypes.data,
                                           out["lse"].ctypes.data, out["ez"].ctypes.data)
    if rc == -2:
        raise MemoryError("oracle allocation failed")
    out["rc"] = rc
    return out


def backward_support(h, W, targets, rows, support, tau, g1, g2, dtype, vsel=None):
    """Gradients of sum(g1*logp + g2*ent) under the sampling support:
    (dh_rows [n,H], dW_sel [nv,H]) as in :func:`backward`."""
    hs, ht, ldh = storage(h, dtype)
    ws, wt, ldw = storage(W, dtype)
    T, H, V = hs.shape[0], ldh, ws.shape[0]
    rows = _i64(rows if rows is not None else np.arange(T))
    sw, lds = _words(support)
    n = rows.shape[0]
    g1 = np.ascontiguousarray(g1, dtype=np.float64)
    g2 = np.ascontiguousarray(g2, dtype=np.float64)
    vs = None if vsel is None else _i64(vsel)
    nv = V if vs is None else vs.shape[0]
    dh = np.zeros((n, H))
    dW = np.zeros((nv, H))
    rc = lib().orc_backward_support(H, V, hs.ctypes.data, ht, ldh, ws.ctypes.data, wt, ldw,
                                    _ptr(rows), n, T, _ptr(_i64(targets)), sw.ctypes.data, lds,
                                    float(tau), g1.ctypes.data, g2.ctypes.data, dh.ctypes.data,
                                    _ptr(vs), nv, dW.ctypes.data)
    if rc:
        raise RuntimeError("oracle backward_support failed: %d" % rc)
    return dh, dW


def mxfp4_vpad(V):
    """Rows of the blocked MXFP4 layout: V rounded up to a multiple of 256."""
    return -(-V // 256) * 256


def mxfp4_quantize(W, dtype):
    """C quantiser: (packed uint8 [H/64, V_pad, 32], scales uint8 [H/64, V_pad, 2])."""
    ws, wt, ldw = storage(W, dtype)
    V, H = ws.shape[0], ldw
    Vp = mxfp4_vpad(V)
    packed = np.empty((H // 64, Vp, 32), np.uint8)
    scales = np.empty((H // 64, Vp, 2), np.uint8)
    rc = lib().orc_mxfp4_quantize(ws.ctypes.data, wt, V, H, ldw, Vp, packed.ctypes.data,
                                  scales.ctypes.data)
    if rc:
        raise ValueError("H must be a multiple of 64")
    return packed, scales


def mxfp4_dequantize(packed, scales, V):
    packed = np.ascontiguousarray(packed, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    H = packed.shape[0] * 64
    out = np.empty((V, H))
    lib().orc_mxfp4_dequantize(packed.ctypes.data, scales.ctypes.data, V, H, packed.shape[1],
                               out.ctypes.data)
    return out


def kl_mxfp4(h_s, W_s, h_t, packed, scales, rows, dtype):
    """Per scored row KL(teacher || student), the teacher head in MXFP4."""
    a, ty, ldh = storage(h_s, dtype)
    b, _, ldw = storage(W_s, dtype)
    c, _, _ = storage(h_t, dtype)
    packed = np.ascontiguousarray(packed, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    T, V = a.shape[0], b.shape[0]
    rows = _i64(rows if rows is not None else np.arange(T))
    out = np.empty(rows.shape[0], dtype=np.float64)
    rc = lib().orc_kl_mxfp4(ldh, V, a.ctypes.data, b.ctypes.data, c.ctypes.data,
                            packed.ctypes.data, scales.ctypes.data, packed.shape[1], ty, ldh,
                            ldw, _ptr(rows), rows.shape[0], out.ctypes.data)
    if rc:
        raise RuntimeError("oracle kl_mxfp4 failed: %d" % rc)
    return out


def e4m3_value(code):
    """Value of one E4M3 code (0..255) by the C oracle's decoder."""
    return float(lib().orc_e4m3_value(int(code)))


def mxfp8_quantize(X, dtype):
    """C quantiser: (codes uint8 [R, H] E4M3, scales uint8 [R, H/32] E8M0)."""
    xs, xt, ld = storage(X, dtype)
    R, H = xs.shape[0], ld
    codes = np.empty((R, H), np.uint8)
    scales = np.empty((R, H // 32), np.uint8)
    rc = lib().orc_mxfp8_quantize(xs.ctypes.data, xt, R, H, ld, codes.ctypes.data,
                                  scales.ctypes.data)
    if rc:
        raise ValueError("H must be a multiple of 32")
    return codes, scales


def mxfp8_dequantize(codes, scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    R, H = codes.shape
    out = np.empty((R, H))
    lib().orc_mxfp8_dequantize(codes.ctypes.data, scales.ctypes.data, R, H, out.ctypes.data)
    return out


def kl_mx(h_s, W_s, h_t, packed, scales, rows, dtype):
    """Per scored row KL(teacher || student) on the block-scaled teacher path:
    h_t rows quantised to MXFP8, the teacher head in MXFP4 (blocked layout)."""
    a, ty, ldh = storage(h_s, dtype)
    b, _, ldw = storage(W_s, dtype)
    c, _, _ = storage(h_t, dtype)
    packed = np.ascontiguousarray(packed, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    T, V = a.shape[0], b.shape[0]
    rows = _i64(rows if rows is not None else np.arange(T))
    out = np.empty(rows.shape[0], dtype=np.float64)
    rc = lib().orc_kl_mx(ldh, V, a.ctypes.data, b.ctypes.data, c.ctypes.data,
                         packed.ctypes.data, scales.ctypes.data, packed.shape[1], ty, ldh, ldw,
                         _ptr(rows), rows.shape[0], out.ctypes.data)
    if rc:
        raise RuntimeError("oracle kl_mx failed: %d" % rc)
    return out


def logprob_entropy_mx(h, packed, scales, V, targets, rows, tau, dtype):
    """Per scored row logp, ent, lse, ez on the block-scaled path: the rows
    h[rows] quantised to MXFP8, the head in MXFP4 (blocked layout, V rows)."""
    hs, ht, ldh = storage(h, dtype)
    packed = np.ascontiguousarray(packed, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    T, H = hs.shape[0], ldh
    rows = _i64(rows if rows is not None else np.arange(T))
    tg = _i64(targets)
    n = rows.shape[0]
    out = {k: np.empty(n, dtype=np.float64) for k in ("logp", "ent", "lse", "ez")}
    rc = lib().orc_logprob_entropy_mx(H, int(V), hs.ctypes.data, ht, ldh, packed.ctypes.data,
                                      scales.ctypes.data, packed.shape[1], _ptr(rows), n, T,
                                      _ptr(tg), float(tau), out["logp"].ctypes.data,
                                      out["ent"].ctypes.data, out["lse"].ctypes.data,
                                      out["ez"].ctypes.data)
    if rc == -2:
        raise MemoryError("oracle allocation failed")
    out["rc"] = rc
    return out
