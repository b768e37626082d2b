"""Fused LM-head token scoring on GB300 (sm_103a): Python binding of libfusedlogp.

This module only marshals arguments: it checks tensor layouts, allocates the
outputs and the workspace with torch, and passes raw device pointers and the
current CUDA stream to the C ABI declared in ``include/fusedlogp.h``.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
or PyTorch fallback, and a missing library raises.

    logp, ent = logprob_entropy(h, W, targets, row_idx, temperature)
    logp, ent = logprob_entropy(h, W, targets, row_idx, temperature,
                                support=pack_support(mask))        # sampling support
    kl = kl_divergence(h_s, W_s, h_t, W_t, row_idx)
    kl = kl_divergence_mxfp4(h_s, W_s, h_t, *mxfp4_quantize(W_t), row_idx)
    kl = kl_divergence_mx(h_s, W_s, h_t, mx_head_quantize(W_t), row_idx)  # block-scaled MMA
    logp, ent = logprob_entropy_mx(h, mx_head_quantize(W), V, targets, row_idx, temperature)
    dh, dW = backward(h, W, targets, row_idx, temperature, g1, g2)
    logp, ent = FusedLogProbEntropy.apply(h, W, targets, row_idx, temperature)
"""
import ctypes
import os

import torch

from . import _build

__all__ = ["lib", "build", "workspace_size", "logprob_entropy", "logprob_entropy_k",
           "kl_divergence", "backward", "pack_support", "mxfp4_quantize",
           "kl_divergence_mxfp4", "mx_head_quantize", "mxfp8_quantize", "kl_divergence_mx",
           "logprob_entropy_mx",
           "read_device_status", "plan", "set_kernel_events", "set_wait_limit", "row_chunks",
           "FusedLogProbEntropy", "FlpError",
           "OP_LOGPROB_ENTROPY", "OP_KL", "OP_BACKWARD", "OP_KL_MX", "OP_LOGPROB_ENTROPY_MX"]

OP_LOGPROB_ENTROPY, OP_KL, OP_BACKWARD, OP_KL_MX, OP_LOGPROB_ENTROPY_MX = 0, 1, 2, 3, 4
_DTYPES = {torch.bfloat16: 0, torch.float16: 1}


class FlpError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("libfusedlogp: %s (status %d)" % (msg, status))
        self.status = status


class FlpShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("V", ctypes.c_int64),
                ("n_rows", ctypes.c_int64), ("dtype", ctypes.c_int),
                ("ld_h", ctypes.c_int64), ("ld_w", ctypes.c_int64)]


class FlpDeviceStatus(ctypes.Structure):
    _fields_ = [("bad_targets", ctypes.c_uint32), ("bad_rows", ctypes.c_uint32),
                ("timeouts", ctypes.c_uint32), ("empty_supports", ctypes.c_uint32)]


class FlpPlan(ctypes.Structure):
    _fields_ = [("row_tiles", ctypes.c_int32), ("vocab_tiles", ctypes.c_int32),
                ("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("cta_group", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("tiles_per_split", ctypes.c_int32), ("band", ctypes.c_int32),
                ("items", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("max_tiles_per_cta", ctypes.c_int64), ("chunk_rows", ctypes.c_int64),
                ("dh_split", ctypes.c_int32), ("dh_tail_tiles", ctypes.c_int32)]


_lib = None


def build(force=False, verbose=False):
    """Compile libfusedlogp.so in-tree (nvcc, sm_103a)."""
    return _build.build(force=force, verbose=verbose)


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError("libfusedlogp.so is not built; call entropy_tcgen05_vocab_gb300.build()")
    L = ctypes.CDLL(_build.LIB)
    vp, i64, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    shp = ctypes.POINTER(FlpShape)
    L.flp_workspace_size.argtypes = [shp, ctypes.c_int]
    L.flp_workspace_size.restype = sz
    L.flp_logprob_entropy.argtypes = [shp, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp, sz, vp]
    L.flp_kl.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flp_backward.argtypes = [shp, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flp_read_device_status.argtypes = [vp, ctypes.POINTER(FlpDeviceStatus), vp]
    L.flp_status_string.argtypes = [ctypes.c_int]
    L.flp_status_string.restype = ctypes.c_char_p
    L.flp_last_error.restype = ctypes.c_char_p
    L.flp_plan_scoring.argtypes = [shp, ctypes.c_int, ctypes.c_int32, ctypes.POINTER(FlpPlan)]
    L.flp_row_chunks.argtypes = [i64, i64, ctypes.POINTER(ctypes.c_int64), i64]
    L.flp_row_chunks.restype = i64
    L.flp_logprob_entropy_k.argtypes = [shp, vp, vp, vp, ctypes.c_int32, vp, f32, vp, vp, vp, vp,
                                        vp, sz, vp]
    L.flp_logprob_entropy_k.restype = ctypes.c_int
    L.flp_logprob_entropy_noalloc.argtypes = [shp, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp]
    L.flp_logprob_entropy_noalloc.restype = ctypes.c_int
    L.flp_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp, vp]
    L.flp_selftest_wait_timeout.restype = ctypes.c_int
    L.flp_set_kernel_events.argtypes = [vp, vp]
    L.flp_set_kernel_events.restype = ctypes.c_int
    L.flp_set_wait_limit.argtypes = [ctypes.c_uint64]
    L.flp_set_wait_limit.restype = ctypes.c_int
    L.flp_logprob_entropy_support.argtypes = [shp, vp, vp, vp, vp, vp, i64, f32, vp, vp, vp, vp,
                                              vp, sz, vp]
    L.flp_logprob_entropy_support.restype = ctypes.c_int
    L.flp_backward_support.argtypes = [shp, vp, vp, vp, vp, vp, i64, f32, vp, vp, vp, vp, vp, vp,
                                       vp, sz, vp]
    L.flp_backward_support.restype = ctypes.c_int
    L.flp_pack_support.argtypes = [vp, i64, i64, i64, vp, i64, vp]
    L.flp_pack_support.restype = ctypes.c_int
    L.flp_mxfp4_rows.argtypes = [i64]
    L.flp_mxfp4_rows.restype = i64
    L.flp_mxfp4_bytes.argtypes = [i64, i64, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.flp_mxfp4_bytes.restype = sz
    L.flp_mxfp4_quantize.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, vp, vp]
    L.flp_mxfp4_quantize.restype = ctypes.c_int
    L.flp_kl_mxfp4.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flp_kl_mxfp4.restype = ctypes.c_int
    L.flp_mx_head_bytes.argtypes = [i64, i64]
    L.flp_mx_head_bytes.restype = sz
    L.flp_mx_head_quantize.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, vp]
    L.flp_mx_head_quantize.restype = ctypes.c_int
    L.flp_mxfp8_quantize.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, vp, vp]
    L.flp_mxfp8_quantize.restype = ctypes.c_int
    L.flp_kl_mx.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flp_kl_mx.restype = ctypes.c_int
    L.flp_logprob_entropy_mx.argtypes = [shp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp,
                                         sz, vp]
    L.flp_logprob_entropy_mx.restype = ctypes.c_int
    for f in (L.flp_logprob_entropy, L.flp_kl, L.flp_backward, L.flp_read_device_status,
              L.flp_plan_scoring):
        f.restype = ctypes.c_int
    _lib = L
    return L


def _check(status):
    if status != 0:
        L = lib()
        msg = L.flp_last_error().decode() or L.flp_status_string(status).decode()
        raise FlpError(status, msg)


def make_shape(T, H, V, n_rows, dtype, ld_h=None, ld_w=None):
    return FlpShape(T, H, V, n_rows, _DTYPES[dtype] if isinstance(dtype, torch.dtype) else dtype,
                    H if ld_h is None else ld_h, H if ld_w is None else ld_w)


def workspace_size(shape, op):
    return int(lib().flp_workspace_size(ctypes.byref(shape), op))


def plan(shape, op, num_sms):
    """Tiling plan the library would use on a device with ``num_sms`` SMs."""
    out = FlpPlan()
    _check(lib().flp_plan_scoring(ctypes.byref(shape), op, num_sms, ctypes.byref(out)))
    return {k: getattr(out, k) for k, _ in FlpPlan._fields_}


def row_chunks(n_rows, chunk_rows):
    """Row-chunk lengths of the backward (the pages' chunk rule)."""
    k = lib().flp_row_chunks(n_rows, chunk_rows, None, 0)
    buf = (ctypes.c_int64 * max(k, 1))()
    lib().flp_row_chunks(n_rows, chunk_rows, buf, k)
    return [int(buf[i]) for i in range(k)]


def set_kernel_events(before, after):
    """Have the next call on this thread record two torch.cuda.Events around
    its tensor-core kernels (both must have been recorded once, so that they
    exist)."""
    lib().flp_set_kernel_events(ctypes.c_void_p(before.cuda_event), ctypes.c_void_p(after.cuda_event))


def set_wait_limit(limit_ns):
    """Wall-clock limit (ns) of the kernels' barrier waits for later calls from
    this thread; 0 restores the default (4 s).  A wait that runs out ends its
    kernel with a timeout counted in the call's device status."""
    _check(lib().flp_set_wait_limit(int(limit_ns)))


def selftest_wait_timeout(limit_ns, device=None):
    """Run the bounded-wait self-test kernel; returns the device status it left."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    _check(lib().flp_selftest_wait_timeout(int(limit_ns), _ptr(ws), _stream(dev)))
    return read_device_status(ws, dev)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _matrix(x, name):
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if x.dim() != 2 or x.dtype not in _DTYPES or x.stride(1) != 1:
        raise TypeError("%s must be a 2-D bf16/fp16 tensor with unit column stride" % name)
    return x


def _index(x, name, device):
    if x is None:
        return None
    if not isinstance(x, torch.Tensor) or x.device != device:
        raise TypeError("%s must be a tensor on %s" % (name, device))
    return x.to(torch.int64).contiguous()


def _vector(x, name, n, device):
    if x is None:
        return None
    if not isinstance(x, torch.Tensor) or x.device != device or x.numel() != n:
        raise TypeError("%s must be a [%d] tensor on %s" % (name, n, device))
    return x.to(torch.float32).contiguous()


def _support(x, T, V, device):
    """(tensor, row stride in words) of a packed support, or (None, 0)."""
    if x is None:
        return None, 0
    nw = (V + 31) // 32
    if not isinstance(x, torch.Tensor) or x.device != device or x.dim() != 2 or \
            x.dtype != torch.int32 or x.stride(1) != 1 or x.shape[0] != T or x.shape[1] < nw:
        raise TypeError("support must be an int32 [T, >= ceil(V/32)] tensor of packed bits on "
                        "%s (see pack_support)" % device)
    return x, x.stride(0)


def pack_support(mask, words=None):
    """Pack a [T, V] bool/uint8 CUDA mask (True = token in the row's sampling
    support) into int32 words [T, ceil(V/32)] (or ``words`` columns): bit v % 32
    of word v // 32 is token v.  Runs on the GPU (flp_pack_support)."""
    if not isinstance(mask, torch.Tensor) or not mask.is_cuda or mask.dim() != 2 or \
            mask.dtype not in (torch.bool, torch.uint8) or mask.stride(1) != 1:
        raise TypeError("mask must be a 2-D bool/uint8 CUDA tensor with unit column stride")
    T, V = mask.shape
    nw = (V + 31) // 32 if words is None else int(words)
    out = torch.empty((T, nw), dtype=torch.int32, device=mask.device)
    with torch.cuda.device(mask.device):
        _check(lib().flp_pack_support(_ptr(mask), T, V, mask.stride(0), _ptr(out), nw,
                                      _stream(mask.device)))
    return out


def _workspace(shape, op, device, workspace):
    need = workspace_size(shape, op)
    if need == 0:
        raise FlpError(1, "invalid shape")
    if workspace is not None and workspace.numel() >= need:
        return workspace
    return torch.empty(need, dtype=torch.uint8, device=device)


def logprob_entropy(h, W, targets, row_idx=None, temperature=1.0, *, return_stats=False,
                    workspace=None, support=None):
    """Target log-prob and entropy of softmax(h[row_idx] W^T / temperature).

    h [T,H] and W [V,H] bf16/fp16 on the same GPU; targets int64 [T] indexed
    by h row; row_idx int64 [n] (or None: every row).  Returns float32 [n]
    tensors (logp, ent), plus (lse, ez) if ``return_stats``.  ``support``
    (packed by :func:`pack_support`, [T, words] by h row) restricts each row
    to its sampling support (logp = -inf for a target outside it).
    """
    _matrix(h, "h")
    _matrix(W, "W")
    dev = h.device
    if W.device != dev or W.dtype != h.dtype or W.shape[1] != h.shape[1]:
        raise TypeError("W must match h in device, dtype and hidden size")
    tg = _index(targets, "targets", dev)
    ri = _index(row_idx, "row_idx", dev)
    n = h.shape[0] if ri is None else ri.numel()
    shape = make_shape(h.shape[0], h.shape[1], W.shape[0], n, h.dtype, h.stride(0), W.stride(0))
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    ent = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev) if return_stats else None
    ez = torch.empty(n, dtype=torch.float32, device=dev) if return_stats else None
    sup, lds = _support(support, h.shape[0], W.shape[0], dev)
    ws = _workspace(shape, OP_LOGPROB_ENTROPY, dev, workspace)
    with torch.cuda.device(dev):
        if sup is None:
            _check(lib().flp_logprob_entropy(ctypes.byref(shape), _ptr(h), _ptr(W), _ptr(tg),
                                             _ptr(ri), float(temperature), _ptr(logp), _ptr(ent),
                                             _ptr(lse), _ptr(ez), _ptr(ws), ws.numel(),
                                             _stream(dev)))
        else:
            _check(lib().flp_logprob_entropy_support(
                ctypes.byref(shape), _ptr(h), _ptr(W), _ptr(tg), _ptr(ri), _ptr(sup), lds,
                float(temperature), _ptr(logp), _ptr(ent), _ptr(lse), _ptr(ez), _ptr(ws),
                ws.numel(), _stream(dev)))
    if return_stats:
        return logp, ent, lse, ez
    return logp, ent


def logprob_entropy_k(h, W, targets, row_idx=None, temperature=1.0, *, workspace=None):
    """K target tokens per scored row: targets int64 [T, K] (K <= 8) indexed by
    h row.  Returns (logp [n, K], ent [n]) float32."""
    _matrix(h, "h")
    _matrix(W, "W")
    dev = h.device
    if W.device != dev or W.dtype != h.dtype or W.shape[1] != h.shape[1]:
        raise TypeError("W must match h in device, dtype and hidden size")
    if not isinstance(targets, torch.Tensor) or targets.dim() != 2 or targets.device != dev:
        raise TypeError("targets must be a [T, K] tensor on %s" % dev)
    tg = targets.to(torch.int64).contiguous()
    K = tg.shape[1]
    ri = _index(row_idx, "row_idx", dev)
    n = h.shape[0] if ri is None else ri.numel()
    shape = make_shape(h.shape[0], h.shape[1], W.shape[0], n, h.dtype, h.stride(0), W.stride(0))
    logp = torch.empty((n, K), dtype=torch.float32, device=dev)
    ent = torch.empty(n, dtype=torch.float32, device=dev)
    ws = _workspace(shape, OP_LOGPROB_ENTROPY, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib().flp_logprob_entropy_k(ctypes.byref(shape), _ptr(h), _ptr(W), _ptr(tg), K,
                                           _ptr(ri), float(temperature), _ptr(logp), _ptr(ent),
                                           None, None, _ptr(ws), ws.numel(), _stream(dev)))
    return logp, ent


def kl_divergence(h_s, W_s, h_t, W_t, row_idx=None, *, workspace=None):
    """Full-vocabulary KL(teacher || student) per scored row (float32 [n])."""
    for x, nm in ((h_s, "h_s"), (W_s, "W_s"), (h_t, "h_t"), (W_t, "W_t")):
        _matrix(x, nm)
    dev = h_s.device
    if not (h_s.shape == h_t.shape and W_s.shape == W_t.shape and h_s.shape[1] == W_s.shape[1]):
        raise TypeError("student and teacher must share shapes")
    if h_t.stride(0) != h_s.stride(0) or W_t.stride(0) != W_s.stride(0):
        raise TypeError("student and teacher must share row strides")
    if len({x.dtype for x in (h_s, W_s, h_t, W_t)}) != 1:
        raise TypeError("student and teacher must share dtype")
    ri = _index(row_idx, "row_idx", dev)
    n = h_s.shape[0] if ri is None else ri.numel()
    shape = make_shape(h_s.shape[0], h_s.shape[1], W_s.shape[0], n, h_s.dtype, h_s.stride(0),
                       W_s.stride(0))
    out = torch.empty(n, dtype=torch.float32, device=dev)
    ws = _workspace(shape, OP_KL, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib().flp_kl(ctypes.byref(shape), _ptr(h_s), _ptr(W_s), _ptr(h_t), _ptr(W_t),
                            _ptr(ri), _ptr(out), _ptr(ws), ws.numel(), _stream(dev)))
    return out


def backward(h, W, targets, row_idx, temperature, g1, g2, lse=None, ez=None, *, workspace=None,
             support=None, need_dh=True, need_dW=True):
    """dL/dh (dtype of h, [T,H]) and dL/dW (float32 [V,H]) of
    L = sum g1 * logp + g2 * ent, by tile recompute (under each row's
    sampling support if ``support`` is given, as in :func:`logprob_entropy`).
    ``need_dh`` / ``need_dW`` False skips that gradient (returned as None),
    e.g. for a frozen output layer."""
    if not (need_dh or need_dW):
        raise ValueError("need_dh and need_dW are both False")
    _matrix(h, "h")
    _matrix(W, "W")
    dev = h.device
    tg = _index(targets, "targets", dev)
    ri = _index(row_idx, "row_idx", dev)
    n = h.shape[0] if ri is None else ri.numel()
    g1 = _vector(g1, "g1", n, dev)
    g2 = _vector(g2, "g2", n, dev)
    lse = _vector(lse, "lse", n, dev)
    ez = _vector(ez, "ez", n, dev)
    shape = make_shape(h.shape[0], h.shape[1], W.shape[0], n, h.dtype, h.shape[1], W.shape[1])
    dh = torch.empty((h.shape[0], h.shape[1]), dtype=h.dtype, device=dev) if need_dh else None
    dW = (torch.empty((W.shape[0], W.shape[1]), dtype=torch.float32, device=dev)
          if need_dW else None)
    if h.stride(0) != h.shape[1] or W.stride(0) != W.shape[1]:
        h = h.contiguous()
        W = W.contiguous()
    sup, lds = _support(support, h.shape[0], W.shape[0], dev)
    ws = _workspace(shape, OP_BACKWARD, dev, workspace)
    with torch.cuda.device(dev):
        if sup is None:
            _check(lib().flp_backward(ctypes.byref(shape), _ptr(h), _ptr(W), _ptr(tg), _ptr(ri),
                                      float(temperature), _ptr(g1), _ptr(g2), _ptr(lse), _ptr(ez),
                                      _ptr(dh), _ptr(dW), _ptr(ws), ws.numel(), _stream(dev)))
        else:
            _check(lib().flp_backward_support(
                ctypes.byref(shape), _ptr(h), _ptr(W), _ptr(tg), _ptr(ri), _ptr(sup), lds,
                float(temperature), _ptr(g1), _ptr(g2), _ptr(lse), _ptr(ez), _ptr(dh), _ptr(dW),
                _ptr(ws), ws.numel(), _stream(dev)))
    return dh, dW


def mxfp4_quantize(W):
    """Quantise W [V, H] (bf16/fp16 CUDA, H a multiple of 64) to MXFP4 on the
    GPU.  Returns (packed uint8 [H/64, V_pad, 32], scales uint8 [H/64, V_pad, 2])
    in the library's blocked layout (see include/fusedlogp.h)."""
    _matrix(W, "W")
    V, H = W.shape
    if H % 64:
        raise TypeError("H must be a multiple of 64")
    Vp = int(lib().flp_mxfp4_rows(V))
    packed = torch.empty((H // 64, Vp, 32), dtype=torch.uint8, device=W.device)
    scales = torch.empty((H // 64, Vp, 2), dtype=torch.uint8, device=W.device)
    with torch.cuda.device(W.device):
        _check(lib().flp_mxfp4_quantize(_ptr(W), _DTYPES[W.dtype], V, H, W.stride(0), _ptr(packed),
                                        _ptr(scales), _stream(W.device)))
    return packed, scales


def kl_divergence_mxfp4(h_s, W_s, h_t, Wt_packed, Wt_scales, row_idx=None, *, workspace=None):
    """KL(teacher || student) per scored row with the teacher head in MXFP4
    (from :func:`mxfp4_quantize`); bf16 rows and student head."""
    for x, nm in ((h_s, "h_s"), (W_s, "W_s"), (h_t, "h_t")):
        _matrix(x, nm)
    dev = h_s.device
    if h_s.shape != h_t.shape or h_s.shape[1] != W_s.shape[1] or h_t.stride(0) != h_s.stride(0):
        raise TypeError("student and teacher rows must share shape and stride with W_s's H")
    V, H = W_s.shape
    Vp = int(lib().flp_mxfp4_rows(V))
    for x, nm, last in ((Wt_packed, "Wt_packed", 32), (Wt_scales, "Wt_scales", 2)):
        if not isinstance(x, torch.Tensor) or x.device != dev or x.dtype != torch.uint8 or \
                tuple(x.shape) != (H // 64, Vp, last) or not x.is_contiguous():
            raise TypeError("%s must be a contiguous uint8 [%d, %d, %d] tensor on %s"
                            % (nm, H // 64, Vp, last, dev))
    ri = _index(row_idx, "row_idx", dev)
    n = h_s.shape[0] if ri is None else ri.numel()
    shape = make_shape(h_s.shape[0], H, V, n, h_s.dtype, h_s.stride(0), W_s.stride(0))
    out = torch.empty(n, dtype=torch.float32, device=dev)
    ws = _workspace(shape, OP_KL, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib().flp_kl_mxfp4(ctypes.byref(shape), _ptr(h_s), _ptr(W_s), _ptr(h_t),
                                  _ptr(Wt_packed), _ptr(Wt_scales), _ptr(ri), _ptr(out), _ptr(ws),
                                  ws.numel(), _stream(dev)))
    return out


def mx_head_quantize(W):
    """Quantise W [V, H] (bf16/fp16 CUDA, H a multiple of 128) to MXFP4 in the
    layout of the block-scaled KL (E2M1 codes [V, H/2] then the scale atoms;
    see include/fusedlogp.h).  Returns a flat uint8 tensor of
    flp_mx_head_bytes(V, H) bytes."""
    _matrix(W, "W")
    V, H = W.shape
    nbytes = int(lib().flp_mx_head_bytes(V, H))
    if nbytes == 0:
        raise TypeError("H must be a positive multiple of 128")
    head = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    with torch.cuda.device(W.device):
        _check(lib().flp_mx_head_quantize(_ptr(W), _DTYPES[W.dtype], V, H, W.stride(0), _ptr(head),
                                          _stream(W.device)))
    return head


def mxfp8_quantize(X):
    """OCP MXFP8 (E4M3 codes, an E8M0 scale per 32) of X [R, H] (bf16/fp16
    CUDA, H a multiple of 32), on the GPU: (codes uint8 [R, H], scales uint8
    [R, H/32])."""
    _matrix(X, "X")
    R, H = X.shape
    codes = torch.empty((R, H), dtype=torch.uint8, device=X.device)
    scales = torch.empty((R, H // 32), dtype=torch.uint8, device=X.device)
    with torch.cuda.device(X.device):
        _check(lib().flp_mxfp8_quantize(_ptr(X), _DTYPES[X.dtype], R, H, X.stride(0), _ptr(codes),
                                        _ptr(scales), _stream(X.device)))
    return codes, scales


def kl_divergence_mx(h_s, W_s, h_t, Wt_head, row_idx=None, *, workspace=None):
    """KL(teacher || student) per scored row with the teacher forward on the
    block-scaled tensor cores: h_t quantised to MXFP8 per call, the teacher
    head in MXFP4 (from :func:`mx_head_quantize`).  Float32 [n]."""
    for x, nm in ((h_s, "h_s"), (W_s, "W_s"), (h_t, "h_t")):
        _matrix(x, nm)
    dev = h_s.device
    if h_s.shape != h_t.shape or h_s.shape[1] != W_s.shape[1] or h_t.stride(0) != h_s.stride(0) \
            or h_t.dtype != h_s.dtype or W_s.dtype != h_s.dtype:
        raise TypeError("student and teacher rows must share shape, stride and dtype with W_s")
    V, H = W_s.shape
    nbytes = int(lib().flp_mx_head_bytes(V, H))
    if not isinstance(Wt_head, torch.Tensor) or Wt_head.device != dev or \
            Wt_head.dtype != torch.uint8 or Wt_head.numel() < nbytes or not Wt_head.is_contiguous():
        raise TypeError("Wt_head must be a contiguous uint8 tensor of >= %d bytes on %s "
                        "(see mx_head_quantize)" % (nbytes, dev))
    ri = _index(row_idx, "row_idx", dev)
    n = h_s.shape[0] if ri is None else ri.numel()
    shape = make_shape(h_s.shape[0], H, V, n, h_s.dtype, h_s.stride(0), W_s.stride(0))
    out = torch.empty(n, dtype=torch.float32, device=dev)
    ws = _workspace(shape, OP_KL_MX, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib().flp_kl_mx(ctypes.byref(shape), _ptr(h_s), _ptr(W_s), _ptr(h_t), _ptr(Wt_head),
                               _ptr(ri), _ptr(out), _ptr(ws), ws.numel(), _stream(dev)))
    return out


def logprob_entropy_mx(h, head, V, targets, row_idx=None, temperature=1.0, *,
                       return_stats=False, workspace=None):
    """Target log-prob and entropy with the logits on the block-scaled tensor
    cores, for scoring that needs no backward (e.g. the reference model's
    log-probs): the scored rows of h [T, H] (bf16/fp16, H a multiple of 128)
    quantised to MXFP8 per call, times the MXFP4 head of V rows (from
    :func:`mx_head_quantize`).  targets int64 [T] by h row, row_idx int64 [n]
    or None.  Returns float32 [n] (logp, ent), plus (lse, ez) if
    ``return_stats``."""
    _matrix(h, "h")
    dev = h.device
    H = h.shape[1]
    nbytes = int(lib().flp_mx_head_bytes(int(V), H))
    if nbytes == 0:
        raise TypeError("V must be > 0 and H a positive multiple of 128")
    if not isinstance(head, torch.Tensor) or head.device != dev or head.dtype != torch.uint8 \
            or head.numel() < nbytes or not head.is_contiguous():
        raise TypeError("head must be a contiguous uint8 tensor of >= %d bytes on %s "
                        "(see mx_head_quantize)" % (nbytes, dev))
    tg = _index(targets, "targets", dev)
    ri = _index(row_idx, "row_idx", dev)
    n = h.shape[0] if ri is None else ri.numel()
    shape = make_shape(h.shape[0], H, int(V), n, h.dtype, h.stride(0), H)
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    ent = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev) if return_stats else None
    ez = torch.empty(n, dtype=torch.float32, device=dev) if return_stats else None
    ws = _workspace(shape, OP_LOGPROB_ENTROPY_MX, dev, workspace)
    with torch.cuda.device(dev):
        _check(lib().flp_logprob_entropy_mx(ctypes.byref(shape), _ptr(h), _ptr(head), _ptr(tg),
                                            _ptr(ri), float(temperature), _ptr(logp), _ptr(ent),
                                            _ptr(lse), _ptr(ez), _ptr(ws), ws.numel(),
                                            _stream(dev)))
    if return_stats:
        return logp, ent, lse, ez
    return logp, ent


def read_device_status(workspace, device=None):
    """Counters the device recorded on ``workspace`` (synchronises the stream)."""
    dev = workspace.device if device is None else device
    st = FlpDeviceStatus()
    rc = lib().flp_read_device_status(_ptr(workspace), ctypes.byref(st), _stream(dev))
    if rc not in (0, 5):
        _check(rc)
    return {k: getattr(st, k) for k, _ in FlpDeviceStatus._fields_}


class FusedLogProbEntropy(torch.autograd.Function):
    """Autograd op: (h, W) -> (logp, ent); backward by tile recompute."""

    @staticmethod
    def forward(ctx, h, W, targets, row_idx=None, temperature=1.0, support=None):
        logp, ent, lse, ez = logprob_entropy(h, W, targets, row_idx, temperature,
                                             return_stats=True, support=support)
        ctx.save_for_backward(h, W, targets, row_idx, lse, ez, support)
        ctx.temperature = temperature
        return logp, ent

    @staticmethod
    def backward(ctx, g_logp, g_ent):
        h, W, targets, row_idx, lse, ez, support = ctx.saved_tensors
        n = lse.numel()
        g1 = g_logp if g_logp is not None else torch.zeros(n, device=h.device)
        g2 = g_ent if g_ent is not None else torch.zeros(n, device=h.device)
        need_dh, need_dW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if not (need_dh or need_dW):
            return None, None, None, None, None, None
        dh, dW = backward(h, W, targets, row_idx, ctx.temperature, g1, g2, lse, ez,
                          support=support, need_dh=need_dh, need_dW=need_dW)
        return dh, (dW.to(W.dtype) if dW is not None else None), None, None, None, None
