"""Float64 CPU oracle for fused LM-head token scoring.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import anything from this package.
The product path (``entropy_tcgen05_vocab_gb300``) never imports it and has
no CPU fallback.

Two independent restatements of the same definitions live here:

* :mod:`oracle.coracle` -- ctypes wrapper around ``oracle.c`` (plain C
  loops, float64, OpenMP over vocabulary rows);
* :mod:`oracle.ref` -- NumPy float64, with ``numpy.matmul`` as the only
  library step.

They share no code with each other beyond the bit decoding of the inputs'
storage formats (which each does on its own) and none at all with the CUDA
library.  The tests in ``tests/test_oracle.py`` pin both to closed forms,
invariants, 50-digit brute force and finite differences.

Definitions (pages: miles PR #2764 summary, "Implementation breakdown" item
2 and its math_utils.py snippet; miles PR #4645, "How it works"; DeepSeek-V4
book ch. 19, "Never materialize logits" and "TileLang KL kernel"):

    z = h W^T,  z' = z / tau  (in float64 after the exact upcast)
    LSE = logsumexp(z'),  p = exp(z' - LSE)
    logp = z'_tgt - LSE,  ent = LSE - sum p z'
    KL(t || s) = sum p_t (log p_t - log p_s)            (tau = 1)
    G = (g1 (onehot - p) - g2 p (z' - sum p z')) / tau
    dh = G W,  dW = G^T h
"""
