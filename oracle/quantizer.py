"""TurboQuant_MSE and TurboQuant_Prod encode / decode (oracle, fp64).

Test infrastructure only (see ``oracle/__init__.py``).

Sources
-------
* Nearest-centroid quantization, index bit string and dequantization by
  table lookup: "TurboQuant 详解", section "例子" (x = [0.8, -0.5, 0.2, -0.9],
  codebook {-0.6, 0.6}, bit string "1010").
* TurboQuant_MSE: y = Π·u, k*(i) = argmin_k |y_i - c_k|, ŷ = c[k*], x̂ = Πᵀŷ;
  the norm s = ‖x‖ is stored separately and u = x/s is quantized:
  "TurboQuant 详解", sections "TurboQuant_mse 的官方步骤" and "一个具体例子：
  KV Cache 在 prefill 和 decode 里怎么量化" (steps 1-6).
* TurboQuant_Prod: a (b-1)-bit MSE stage, residual r = x - x̂_mse, γ = ‖r‖,
  1-bit QJL code sign(S·r) with sign(0) = +1, and the correction
  γ · √(π/2) / d · Sᵀ·sign(S·r): "TurboQuant 详解", section "TurboQuant_prod：
  用残差补偿修正内积偏差"; "turboquant-first-principles-walkthrough", section
  "内积偏差问题与 QJL 修正器"; "sub-byte-kv-cache-quantization-turboquant",
  section "两阶段量化框架".

Readings where the pages are silent or ambiguous:
* Decisions are taken in unit-variance units v = √d · y against centroids in
  the same units; ties at equal distance go to the higher index.
* A zero vector has s = 0, all indices 0, γ = 0 and all QJL bits 0.
* The Prod residual is taken on the unit vector u (r = u - Πᵀŷ) and every
  estimate is scaled back by s.
* The QJL matrix is square (m = d).
* Canonical packing: the b-bit code of coordinate j occupies bits
  [j·b, j·b + b) of the vector's bit stream, least significant bit first;
  stream bit p is bit p mod 32 of little-endian uint32 word p // 32; each
  vector is padded with zero bits to a whole number of 16-byte units.
  The QJL bit of row j of S is stream bit j of its own padded stream.
* b + 1/2 bits per coordinate ("TurboQuant 详解", section "论文给出的关键数据点":
  3.5 and 2.5 bit/channel; section "decode 阶段到底怎么“用”这些压缩后的 KV":
  672 B per token per layer = 16 vectors x (40 B of codes + a 2 B norm), i.e.
  one rotation and one norm per vector and 320 code bits at d = 128): half of
  the rotated coordinates take b + 1 bits, the other half b, each with the
  Lloyd-Max codebook of its own width for the same coordinate density.  Which
  half is immaterial to the quantizer (the coordinates of Π·u are exchangeable
  under a Haar Π); the reading fixes coordinates j with j mod 16 < 8 at b + 1
  bits.  Packing stays canonical with a width per coordinate: the code of
  coordinate j occupies stream bits [P_j, P_j + w_j), P_j = Σ_{i<j} w_i.
* Near-threshold band: a coordinate is excluded from bit-exact comparison iff
  |v - t_k| <= 1e-6 · max(1, |t_k|) for some threshold t_k (unit-variance
  units).  A QJL bit is excluded iff |(S·r)_j| <= 1e-6 · ‖S_j‖₂ · γ, i.e.
  relative to the Cauchy-Schwarz bound of that dot product.
"""

import math

import numpy as np

BAND_REL = 1e-6


def words_per_vector(d, b):
    """uint32 words per packed vector: ceil(b·d/32) rounded up to 4 words."""
    w = (b * d + 31) // 32
    return (w + 3) // 4 * 4


def nearest_centroid(v, centroids):
    """Exhaustive nearest-centroid index; equal distances go to the higher k."""
    v = np.asarray(v, dtype=np.float64)
    c = np.asarray(centroids, dtype=np.float64)
    flat = v.reshape(-1)
    out = np.empty(flat.shape, dtype=np.int64)
    step = 1 << 20  # row blocks only bound the temporary; the search is per element
    for a in range(0, flat.size, step):
        dist = np.abs(flat[a:a + step, None] - c[None, ::-1])
        out[a:a + step] = (len(c) - 1) - np.argmin(dist, axis=-1)
    return out.reshape(v.shape)


def pack_codes(idx, b):
    """Canonical LSB-first packing of [N, d] indices into [N, W] uint32."""
    idx = np.asarray(idx, dtype=np.int64)
    n, d = idx.shape
    W = words_per_vector(d, b)
    words = np.zeros((n, W), dtype=np.uint64)
    for j in range(d):
        for k in range(b):
            p = j * b + k
            bit = (idx[:, j] >> k) & 1
            words[:, p // 32] |= bit.astype(np.uint64) << np.uint64(p % 32)
    return words.astype(np.uint32)


def unpack_codes(words, d, b):
    """Inverse of ``pack_codes``."""
    words = np.asarray(words, dtype=np.uint64)
    n = words.shape[0]
    idx = np.zeros((n, d), dtype=np.int64)
    for j in range(d):
        for k in range(b):
            p = j * b + k
            bit = (words[:, p // 32] >> np.uint64(p % 32)) & np.uint64(1)
            idx[:, j] |= bit.astype(np.int64) << k
    return idx


def pack_bits(bits):
    """QJL sign bits [N, m] -> [N, W] uint32, bit j of word j // 32 (LSB first)."""
    return pack_codes(np.asarray(bits, dtype=np.int64), 1)


def unpack_bits(words, m):
    return unpack_codes(words, m, 1)


def _unit_rows(X):
    X = np.asarray(X, dtype=np.float64)
    s = np.sqrt((X * X).sum(axis=1))
    U = np.zeros_like(X)
    nz = s > 0.0
    U[nz] = X[nz] / s[nz, None]
    return U, s


def near_threshold(v, centroids):
    """Mask of coordinates within the 1e-6 relative band of a threshold."""
    c = np.asarray(centroids, dtype=np.float64)
    t = 0.5 * (c[:-1] + c[1:])
    v = np.asarray(v, dtype=np.float64)
    mask = np.zeros(v.shape, dtype=bool)
    for tk in t:
        mask |= np.abs(v - tk) <= BAND_REL * max(1.0, abs(tk))
    return mask


def mse_quantize(X, Pi, centroids, scale):
    """TurboQuant_MSE encode of the rows of X.

    X          [N, d] exact input values (fp32/fp16 inputs widened to fp64)
    Pi         [d, d] rotation
    centroids  codebook, in units where a rotated unit-vector coordinate is
               multiplied by ``scale`` (scale = √d for unit-variance codebooks)
    Returns (idx [N, d], s [N], v [N, d]) with v = scale · Π·u.
    Rows with s = 0 get all-zero indices.
    """
    U, s = _unit_rows(X)
    Pi = np.asarray(Pi, dtype=np.float64)
    v = scale * (U @ Pi.T)
    idx = nearest_centroid(v, centroids)
    idx[s == 0.0] = 0
    return idx, s, v


def mse_dequantize(idx, s, Pi, centroids, scale):
    """x̂ = s · Πᵀ · (c[idx] / scale)."""
    c = np.asarray(centroids, dtype=np.float64)
    yhat = c[np.asarray(idx)] / scale
    return np.asarray(s, dtype=np.float64)[:, None] * (yhat @ np.asarray(Pi, dtype=np.float64))


def qjl_encode(R, S):
    """1-bit QJL code of residuals R [N, d]: (bits [N, m], γ [N], p = S·r).

    bit_j = 1 iff (S·r)_j >= 0, i.e. sign(0) = +1.
    """
    R = np.asarray(R, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    p = R @ S.T
    bits = (p >= 0.0).astype(np.int64)
    gamma = np.sqrt((R * R).sum(axis=1))
    return bits, gamma, p


def qjl_correction(bits, gamma, S):
    """γ · √(π/2)/m · Sᵀ · (2·bits - 1): the correction vector of the Prod stage."""
    S = np.asarray(S, dtype=np.float64)
    m = S.shape[0]
    sgn = 2.0 * np.asarray(bits, dtype=np.float64) - 1.0
    return (np.asarray(gamma, dtype=np.float64) * math.sqrt(math.pi / 2.0) / m)[:, None] * (sgn @ S)


def prod_quantize(X, Pi, S, centroids_mse, scale):
    """TurboQuant_Prod encode: (b-1)-bit MSE stage plus a 1-bit QJL stage.

    Returns dict(idx, s, bits, gamma, v, p): idx/v as in ``mse_quantize`` for
    the MSE stage, bits/gamma/p of the QJL stage on r = u - Πᵀŷ.
    Zero rows: idx 0, gamma 0, bits 0.
    """
    U, s = _unit_rows(X)
    Pi = np.asarray(Pi, dtype=np.float64)
    v = scale * (U @ Pi.T)
    idx = nearest_centroid(v, centroids_mse)
    zero = s == 0.0
    idx[zero] = 0
    yhat = np.asarray(centroids_mse, dtype=np.float64)[idx] / scale
    R = U - yhat @ Pi
    R[zero] = 0.0
    bits, gamma, p = qjl_encode(R, S)
    bits[zero] = 0
    return {"idx": idx, "s": s, "bits": bits, "gamma": gamma, "v": v, "p": p}


def qjl_near_zero(p, gamma, S):
    """Mask of QJL bits inside the band |p_j| <= 1e-6 · ‖S_j‖ · γ."""
    S = np.asarray(S, dtype=np.float64)
    rownorm = np.sqrt((S * S).sum(axis=1))
    return np.abs(p) <= BAND_REL * rownorm[None, :] * np.asarray(gamma)[:, None]


def prod_dequantize(idx, s, bits, gamma, Pi, S, centroids_mse, scale):
    """x̂_prod = s · (Πᵀ ŷ + γ √(π/2)/m · Sᵀ sign)."""
    c = np.asarray(centroids_mse, dtype=np.float64)
    base = (c[np.asarray(idx)] / scale) @ np.asarray(Pi, dtype=np.float64)
    return np.asarray(s, dtype=np.float64)[:, None] * (base + qjl_correction(bits, gamma, S))


# ------------------------------------------------------------ b + 1/2 bits
def mixed_widths(d, b):
    """Bits of rotated coordinate j at b + 1/2 bits per coordinate: b + 1 where
    j mod 16 < 8, b elsewhere."""
    j = np.arange(d)
    return np.where(j % 16 < 8, b + 1, b).astype(np.int64)


def mixed_words_per_vector(d, b):
    """uint32 words per packed vector: the Σ w_j bits, rounded up to whole words."""
    return (int(mixed_widths(d, b).sum()) + 31) // 32


def pack_varwidth(idx, widths):
    """Canonical LSB-first packing of [N, n] indices with a width per position:
    position j occupies stream bits [P_j, P_j + w_j), P_j = Σ_{i<j} w_i."""
    idx = np.asarray(idx, dtype=np.int64)
    widths = [int(w) for w in widths]
    n = idx.shape[0]
    W = (sum(widths) + 31) // 32
    words = np.zeros((n, W), dtype=np.uint64)
    p = 0
    for j, w in enumerate(widths):
        for k in range(w):
            bit = (idx[:, j] >> k) & 1
            words[:, p // 32] |= bit.astype(np.uint64) << np.uint64(p % 32)
            p += 1
    return words.astype(np.uint32)


def unpack_varwidth(words, widths):
    """Inverse of ``pack_varwidth``."""
    words = np.asarray(words, dtype=np.uint64)
    widths = [int(w) for w in widths]
    idx = np.zeros((words.shape[0], len(widths)), dtype=np.int64)
    p = 0
    for j, w in enumerate(widths):
        for k in range(w):
            bit = (words[:, p // 32] >> np.uint64(p % 32)) & np.uint64(1)
            idx[:, j] |= bit.astype(np.int64) << k
            p += 1
    return idx


def pack_mixed_pairs(idx, b):
    """Pair blocks of a b + 1/2-bit V cache: vectors 2i and 2i+1 share one stream
    in which coordinate j holds the even vector's code then the odd vector's,
    w_j bits each ([N, d] indices, N even -> [N/2, 2W] words)."""
    idx = np.asarray(idx, dtype=np.int64)
    d = idx.shape[1]
    inter = np.zeros((idx.shape[0] // 2, 2 * d), dtype=np.int64)
    inter[:, 0::2] = idx[0::2]
    inter[:, 1::2] = idx[1::2]
    return pack_varwidth(inter, np.repeat(mixed_widths(d, b), 2))


def mixed_quantize(X, Pi, centroids_lo, centroids_hi, b, scale):
    """TurboQuant_MSE at b + 1/2 bits: as ``mse_quantize``, but coordinate j is
    quantized with the (b+1)-bit codebook where w_j = b + 1 and with the b-bit
    codebook elsewhere.  Returns (idx [N, d], s [N], v [N, d])."""
    U, s = _unit_rows(X)
    Pi = np.asarray(Pi, dtype=np.float64)
    v = scale * (U @ Pi.T)
    hi = mixed_widths(v.shape[1], b) == b + 1
    idx = np.where(hi[None, :], nearest_centroid(v, centroids_hi), nearest_centroid(v, centroids_lo))
    idx[s == 0.0] = 0
    return idx, s, v


def mixed_dequantize(idx, s, Pi, centroids_lo, centroids_hi, b, scale):
    """x̂ = s · Πᵀ · (c_j[idx_j] / scale), c_j the codebook of coordinate j's width."""
    idx = np.asarray(idx, dtype=np.int64)
    hi = mixed_widths(idx.shape[1], b) == b + 1
    c_lo = np.asarray(centroids_lo, dtype=np.float64)
    c_hi = np.asarray(centroids_hi, dtype=np.float64)
    yhat = np.where(hi[None, :], c_hi[np.minimum(idx, len(c_hi) - 1)], c_lo[np.minimum(idx, len(c_lo) - 1)])
    yhat = yhat / scale
    return np.asarray(s, dtype=np.float64)[:, None] * (yhat @ np.asarray(Pi, dtype=np.float64))


def mixed_near_threshold(v, centroids_lo, centroids_hi, b):
    """The near-threshold band of each coordinate against its own codebook."""
    v = np.asarray(v, dtype=np.float64)
    hi = mixed_widths(v.shape[-1], b) == b + 1
    return np.where(hi, near_threshold(v, centroids_hi), near_threshold(v, centroids_lo))
