"""Inner-product scores and decode attention over TurboQuant codes (oracle, fp64).

Test infrastructure only (see ``oracle/__init__.py``).

Everything here works by EXPLICIT dequantization: every key/value vector is
rebuilt as x̂ = s · Πᵀ ŷ (plus the QJL correction for TurboQuant_Prod) and the
textbook formula is applied to the rebuilt vectors.  The GPU path's
algebraic shortcuts (pre-rotated query, accumulation of V in the rotated
domain, one inverse rotation per head) are therefore checked against an
implementation that does not use them.

Sources
-------
* Decode first dequantizes (unpack, table lookup, multiply by Rᵀ and the
  norm) and then runs ordinary attention: "TurboQuant 详解", section
  "decode 阶段到底怎么“用”这些压缩后的 KV" (first route).
* Attention(Q, K, V) = softmax(Q Kᵀ / √d) V: "TurboQuant 和 RotorQuant 的真相",
  chapter 1 ("为什么压缩 KV 缓存这么难").
* GQA map kv_head = q_head // gqa_ratio: "sub-byte-kv-cache-quantization-
  turboquant", section "工程实现的关键路径".
* Prod inner-product estimator ⟨y, x̂_mse⟩ + ⟨y, corr⟩:
  "TurboQuant 详解", section "TurboQuant_prod：用残差补偿修正内积偏差".
"""

import numpy as np

from .quantizer import mse_dequantize, prod_dequantize


def mse_scores(Q, idx, s, Pi, centroids, scale):
    """ŝ[m, n] = ⟨q_m, x̂_n⟩ with x̂_n = s_n · Πᵀ ŷ_n."""
    Xh = mse_dequantize(idx, s, Pi, centroids, scale)
    return np.asarray(Q, dtype=np.float64) @ Xh.T


def prod_scores(Q, idx, s, bits, gamma, Pi, S, centroids_mse, scale):
    """ŝ[m, n] = ⟨q_m, x̂_prod,n⟩, the unbiased TurboQuant_Prod estimate."""
    Xh = prod_dequantize(idx, s, bits, gamma, Pi, S, centroids_mse, scale)
    return np.asarray(Q, dtype=np.float64) @ Xh.T


def softmax(z):
    """Max-subtracted softmax along the last axis."""
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def decode_attention(q, Khat, Vhat, sm_scale):
    """One decode step: out[b, h] = Σ_t softmax_t(⟨q[b,h], k̂[b,kv,t]⟩·scale) v̂[b,kv,t].

    q     [B, Hq, d]
    Khat  [B, Hkv, T, d]  explicitly dequantized keys
    Vhat  [B, Hkv, T, d]  explicitly dequantized values
    The query head h reads KV head h // (Hq // Hkv).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv = Khat.shape[1]
    gqa = Hq // Hkv
    out = np.zeros((B, Hq, d), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            kv = h // gqa
            z = (Khat[b, kv] @ q[b, h]) * sm_scale
            p = softmax(z)
            out[b, h] = p @ Vhat[b, kv]
    return out


def dequantize_cache(idx, s, Pi, centroids, scale, B, Hkv, T):
    """Rebuild a [B, Hkv, T, d] cache from canonical indices [B*Hkv*T, d]."""
    Xh = mse_dequantize(idx, s, Pi, centroids, scale)
    return Xh.reshape(B, Hkv, T, -1)
