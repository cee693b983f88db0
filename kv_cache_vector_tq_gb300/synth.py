"""Seeded synthetic inputs shaped like the workloads the TurboQuant pages discuss.

This module draws random numbers and lays out arrays; it contains none of the
method's arithmetic (no rotation, no quantization).  The tests feed its output
to both the CUDA library and the CPU oracle, and the benchmark uses it for its
host-side inputs.

Streams: ``np.random.SeedSequence(seed).spawn(8)``
  0  Gaussian matrix G whose QR gives the Haar rotation
  1  QJL matrix S
  2  data vectors (keys, values, bulk rows)
  3  queries
  4  Hadamard sign vector
  5  choice of scaled rows (bulk indexing outliers)
Per-layer KV data of the long-context shape uses SeedSequence([seed, layer]).

Workload shapes (head_dim 128, GQA, outlier channels, 70B-like 80 layers x 8 KV
heads, bulk indexing over d in 64..3072) follow "TurboQuant 详解" (KV cache
example with 128-dim heads), "TurboQuant 和 RotorQuant 的真相" chapter 1
(80 layers, 8 KV heads, 128 dims) and "turboquant-first-principles-
walkthrough" (outlier channels; d from 64 to 3072; 100K-vector indexing).
"""

import numpy as np

N_STREAMS = 8


def _gen(seed, stream):
    return np.random.default_rng(np.random.SeedSequence(seed).spawn(N_STREAMS)[stream])


def gaussian_matrix(seed, d):
    """d x d i.i.d. N(0, 1), fp64 (input of the Haar rotation)."""
    return _gen(seed, 0).standard_normal((d, d))


def qjl_matrix(seed, d):
    """d x d i.i.d. N(0, 1), fp64 (QJL projection S)."""
    return _gen(seed, 1).standard_normal((d, d))


def hadamard_signs(seed, d):
    """d random signs in {-1, +1}, fp64."""
    return np.where(_gen(seed, 4).integers(0, 2, size=d) == 1, 1.0, -1.0)


def gaussian_rows(seed, n, d, outlier_cols=0, outlier_scale=1.0, dtype=np.float32):
    """n x d i.i.d. N(0, 1) rows, the first ``outlier_cols`` columns scaled."""
    x = _gen(seed, 2).standard_normal((n, d), dtype=np.float32)
    if outlier_cols:
        x[:, :outlier_cols] *= np.float32(outlier_scale)
    return x.astype(dtype)


def unit_rows(seed, n, d):
    """n x d Gaussian rows normalised to unit length, fp32."""
    x = _gen(seed, 2).standard_normal((n, d))
    x /= np.sqrt((x * x).sum(axis=1, keepdims=True))
    return x.astype(np.float32)


def queries(seed, m, d, dtype=np.float32):
    """m x d i.i.d. N(0, 1) queries."""
    return _gen(seed, 3).standard_normal((m, d), dtype=np.float32).astype(dtype)


def kv_layer(seed, layer, B, Hkv, T, d, outlier_cols=4, outlier_scale=10.0):
    """fp16 K and V of one layer, [B, Hkv, T, d] each, N(0, 1) with outlier channels."""
    g = np.random.default_rng(np.random.SeedSequence([seed, layer]))
    k = g.standard_normal((B, Hkv, T, d), dtype=np.float32)
    v = g.standard_normal((B, Hkv, T, d), dtype=np.float32)
    k[..., :outlier_cols] *= np.float32(outlier_scale)
    v[..., :outlier_cols] *= np.float32(outlier_scale)
    return k.astype(np.float16), v.astype(np.float16)


def bulk_rows(seed, n, d, frac=0.01, scale=50.0):
    """n x d i.i.d. N(0, 1) fp32 rows; a seeded 1% of the rows scaled by 50."""
    x = _gen(seed, 2).standard_normal((n, d), dtype=np.float32)
    k = max(1, int(round(frac * n)))
    rows = _gen(seed, 5).choice(n, size=k, replace=False)
    x[rows] *= np.float32(scale)
    return x
