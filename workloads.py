"""Seeded synthetic inputs for the five scoring workloads.

This module only draws inputs.  It holds none of the scoring arithmetic
(no log-sum-exp, entropy, KL or gradient): the CUDA library and the float64
oracle both take their inputs from here and from nowhere else.

Recipe (shapes and distributions of the pages' workloads; no dataset or
checkpoint is involved, the shapes stand in for the Qwen-class LM heads the
miles PR #4645 "Testing" table measures):

  id  workload                 T       H     V        dtype  h        W           targets              tau
  0   tiny                     256     512   8,192    bf16   N(0,1)   N(0,0.02)   U[0,V)               1.0
  1   forward scoring          4,096   4096  151,936  bf16   N(0,1)   N(0,0.05)   ~ softmax(z/0.7)     0.7
  2   long packed micro-batch  49,152  5120  38,016   fp16   N(0,1)   N(0,0.04)   U[0,V)               1.0
  3   distillation KL          8,192   4096  129,280  bf16   h_s N(0,1), h_t = h_s + N(0,0.3); W_s, W_t N(0,0.05)
  4   backward                 16,384  4096  151,936  bf16   N(0,1)   N(0,0.05)   U[0,V)               0.7

Row selection: workload 2 packs sequences of length U[512, 8192] (the last
one truncated to fill T) and scores the last round(0.6 len) positions of
each (prompt first, response last); workload 4 scores a Bernoulli(0.6) row
mask; the others score every row.  Workload 4 also draws g1, g2 ~ N(0,1)
(float32) per scored row.

Sampling supports (the per-row vocabulary masks of the sampling_mask
argument) are drawn by :func:`support_words`: each bit is Bernoulli(2^-j), the
AND of j uniform random words, packed 32 tokens per uint32 word (bit v % 32
of word v // 32), optionally with each row's target forced in.

Random streams: discrete draws (targets, lengths, masks) always come from
``numpy.random.Generator(PCG64([seed, k]))`` on the host, so they do not
depend on the device.  Continuous draws are float32 normals rounded to
bf16/fp16 (round to nearest even); they come from the same NumPy generator
for small tensors and, for tensors of 2**26 elements or more generated on a
GPU, from ``torch.Generator`` on that device (seeded ``seed*100+k``), which
is deterministic for a given device type and torch version.  Workload 1's
targets are drawn by Gumbel-max over z/0.7, z = h W^T from a float32
matmul: that is sampling a target, not scoring one.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

LARGE = 1 << 26


@dataclasses.dataclass(frozen=True)
class Workload:
    id: int
    name: str
    T: int
    H: int
    V: int
    dtype: str          # "bf16" | "fp16"
    h_std: float
    w_std: float
    targets: str        # "uniform" | "softmax"
    tau: float
    seed: int
    rows: str           # "all" | "packed" | "bernoulli"
    kind: str           # "fwd" | "kl" | "bwd"
    teacher_noise: float = 0.0

    def scaled(self, **kw) -> "Workload":
        """Same recipe with some sizes replaced (for small test cases)."""
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    0: Workload(0, "tiny", 256, 512, 8192, "bf16", 1.0, 0.02, "uniform", 1.0, 0, "all", "fwd"),
    1: Workload(1, "forward-scoring", 4096, 4096, 151936, "bf16", 1.0, 0.05, "softmax", 0.7, 1,
                "all", "fwd"),
    2: Workload(2, "long-packed", 49152, 5120, 38016, "fp16", 1.0, 0.04, "uniform", 1.0, 2,
                "packed", "fwd"),
    3: Workload(3, "distill-kl", 8192, 4096, 129280, "bf16", 1.0, 0.05, "uniform", 1.0, 3,
                "all", "kl", teacher_noise=0.3),
    4: Workload(4, "backward", 16384, 4096, 151936, "bf16", 1.0, 0.05, "uniform", 0.7, 4,
                "bernoulli", "bwd"),
}

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "f32": torch.float32}


def _np_rng(seed: int, k: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, k]))


def normal(shape, std, seed, k, dtype, device, generator="auto"):
    """float32 N(0, std^2) draws rounded to ``dtype`` on ``device``."""
    device = torch.device(device)
    numel = int(np.prod(shape))
    use_torch = generator == "device" or (
        generator == "auto" and device.type == "cuda" and numel >= LARGE)
    if use_torch:
        g = torch.Generator(device=device)
        g.manual_seed(seed * 100 + k)
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    else:
        x = torch.from_numpy(_np_rng(seed, k).standard_normal(shape, dtype=np.float32))
        x = x.to(device)
    if std != 1.0:
        x.mul_(std)
    return x.to(TORCH_DTYPES[dtype])


def packed_response_rows(T: int, seed: int, lo: int = 512, hi: int = 8192, frac: float = 0.6):
    """Sequences of length U[lo, hi] packed into T positions (the last one
    truncated); the last round(frac * len) positions of each are scored.
    Returns (row_idx int64 sorted, seq_lens int64)."""
    rng = _np_rng(seed, 10)
    lens = []
    total = 0
    while total < T:
        L = int(rng.integers(lo, hi + 1))
        L = min(L, T - total)
        lens.append(L)
        total += L
    rows = []
    start = 0
    for L in lens:
        r = int(round(frac * L))
        rows.append(np.arange(start + L - r, start + L, dtype=np.int64))
        start += L
    return np.concatenate(rows) if rows else np.zeros(0, np.int64), np.array(lens, np.int64)


def bernoulli_rows(T: int, seed: int, frac: float = 0.6):
    rng = _np_rng(seed, 11)
    return np.nonzero(rng.random(T) < frac)[0].astype(np.int64)


def _softmax_targets(h, W, tau, seed, block=256):
    """Gumbel-max draw from softmax(z / tau) per row, z = h W^T (float32)."""
    T = h.shape[0]
    out = torch.empty(T, dtype=torch.int64, device=h.device)
    g = torch.Generator(device=h.device)
    g.manual_seed(seed * 100 + 20)
    Wf = W.float()
    for i0 in range(0, T, block):
        z = h[i0:i0 + block].float() @ Wf.T
        u = torch.rand(z.shape, generator=g, device=h.device, dtype=torch.float32)
        u.clamp_(min=1e-12, max=1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        out[i0:i0 + block] = torch.argmax(z / tau + gumbel, dim=1)
    return out


def make(w, device="cpu", generator="auto"):
    """Draw workload ``w`` (an id or a :class:`Workload`) on ``device``.

    Returns a dict with h [T,H], W [V,H], targets int64 [T] (indexed by h
    row), row_idx int64 [n] or None (all rows), tau, and for "kl" h_t, W_t;
    for "bwd" g1, g2 float32 [n].
    """
    if isinstance(w, int):
        w = WORKLOADS[w]
    dev = torch.device(device)
    out = {"workload": w, "tau": w.tau}
    out["h"] = normal((w.T, w.H), w.h_std, w.seed, 1, w.dtype, dev, generator)
    out["W"] = normal((w.V, w.H), w.w_std, w.seed, 2, w.dtype, dev, generator)
    if w.rows == "all":
        rows = None
        n = w.T
    elif w.rows == "packed":
        rows, _ = packed_response_rows(w.T, w.seed)
        n = rows.shape[0]
    elif w.rows == "bernoulli":
        rows = bernoulli_rows(w.T, w.seed)
        n = rows.shape[0]
    else:
        raise ValueError(w.rows)
    out["row_idx"] = None if rows is None else torch.from_numpy(rows).to(dev)
    out["n"] = n
    if w.targets == "uniform":
        t = _np_rng(w.seed, 3).integers(0, w.V, size=w.T, dtype=np.int64)
        out["targets"] = torch.from_numpy(t).to(dev)
    elif w.targets == "softmax":
        out["targets"] = _softmax_targets(out["h"], out["W"], w.tau, w.seed)
    else:
        raise ValueError(w.targets)
    if w.kind == "kl":
        noise = normal((w.T, w.H), w.teacher_noise, w.seed, 4, "f32", dev, generator)
        out["h_t"] = (out["h"].float() + noise).to(TORCH_DTYPES[w.dtype])
        out["W_t"] = normal((w.V, w.H), w.w_std, w.seed, 5, w.dtype, dev, generator)
        out["h_s"], out["W_s"] = out["h"], out["W"]
    if w.kind == "bwd":
        r = _np_rng(w.seed, 6)
        out["g1"] = torch.from_numpy(r.standard_normal(n, dtype=np.float32)).to(dev)
        out["g2"] = torch.from_numpy(r.standard_normal(n, dtype=np.float32)).to(dev)
    return out


def support_words(T: int, V: int, j: int, seed: int, targets=None, ld: int | None = None,
                  k: int = 30):
    """A seeded sampling-support bitmask as int32 storage of uint32 words,
    [T, ld] with ld >= ceil(V/32) (default equal): token v is in row r's
    support iff bit v % 32 of word v // 32 of row r is set.  Each bit is set
    with probability 2^-j (j = 0: every token).  Bits past V and words past
    ceil(V/32) are random too (consumers must ignore them).  ``targets``
    (int64 [T], host) are forced into their rows' supports."""
    nw = (V + 31) // 32
    ld = nw if ld is None else ld
    if ld < nw:
        raise ValueError("ld < ceil(V/32)")
    rng = _np_rng(seed, k)
    words = np.full((T, ld), 0xFFFFFFFF, dtype=np.uint32)
    for _ in range(j):
        words &= rng.integers(0, 1 << 32, size=(T, ld), dtype=np.uint32)
    if targets is not None:
        t = np.asarray(targets, dtype=np.int64)
        ok = (t >= 0) & (t < V)
        r = np.nonzero(ok)[0]
        words[r, t[ok] // 32] |= (np.uint32(1) << (t[ok] % 32).astype(np.uint32))
    return words.view(np.int32)


def sample_rows(n: int, k: int, seed: int = 1234):
    """A seeded sample of k distinct positions in [0, n) (sorted)."""
    k = min(k, n)
    return np.sort(_np_rng(seed, 99).choice(n, size=k, replace=False)).astype(np.int64)
