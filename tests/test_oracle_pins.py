"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test names the fact it checks.  None of them re-types the oracle's own
formula: they use values printed on the pages (tests/golden), closed forms,
library routines (scipy quadrature, scipy.linalg.hadamard, torch SDPA,
numpy searchsorted) or invariants that a dropped term, a wrong sign or a
transposed operand would break.
"""

import math

import numpy as np
import pytest
import scipy.linalg
from scipy import integrate

from oracle import attention as oatt
from oracle import codebook as ocb
from oracle import quantizer as oq
from kv_cache_vector_tq_gb300 import synth
from oracle import rotation as orot
from tests.conftest import golden


def _rounded(x, digits):
    return float(np.round(x, digits))


# ---------------------------------------------------------------- T1 Lloyd
def test_lloyd_worked_example():
    g = golden("lloyd_1_2_8_9.json")
    hist, final = ocb.lloyd_max(g["data"], np.ones(4), g["init"])
    assert len(hist) == g["converged_after"]
    for (t, c), ref in zip(hist, g["iterations"]):
        np.testing.assert_array_equal(t, ref["threshold"])
        np.testing.assert_array_equal(c, ref["centroids"])
    np.testing.assert_array_equal(final, g["final"])


def test_lloyd_assign_upper_cell_on_tie():
    # a sample exactly on the midpoint goes to the upper cell
    assert list(ocb.lloyd_assign([4.5, 4.4999], [4.5])) == [1, 0]


# ------------------------------------------------- T2/T3 nearest + metrics
def test_uniform_vs_nonuniform_two_bit():
    g = golden("uniform_vs_nonuniform_2bit.json")
    x = np.array(g["x"])
    for cbk, xh_key, mse_key, ip_key in (
        ("codebook_uniform", "xhat_uniform", "mse_uniform", "ip_uniform"),
        ("codebook_nonuniform", "xhat_nonuniform", "mse_nonuniform", "ip_nonuniform"),
    ):
        c = np.array(g[cbk])
        idx = oq.nearest_centroid(x, c)
        xh = c[idx]
        np.testing.assert_allclose(xh, g[xh_key], atol=1e-15)
        mse = float(np.mean((x - xh) ** 2))
        assert _rounded(mse, g["printed_digits_mse"]) == g[mse_key]
        ip = float(np.dot(g["query_y"], xh))
        assert _rounded(ip, g["printed_digits_ip"]) == g[ip_key]
    assert _rounded(float(np.dot(g["query_y"], x)), 3) == g["ip_true"]


def test_nearest_equals_searchsorted_bucketize():
    # exhaustive nearest centroid == counting thresholds t_k <= v (midpoints),
    # computed by numpy's searchsorted; ties go to the higher index
    rng = np.random.default_rng(5)
    c = np.sort(rng.standard_normal(16))
    t = 0.5 * (c[:-1] + c[1:])
    v = rng.standard_normal(5000) * 2
    idx = oq.nearest_centroid(v, c)
    ref = np.searchsorted(t, v, side="right")
    np.testing.assert_array_equal(idx, ref)
    # exact ties (dyadic centroids, so the distances are exactly equal)
    c = np.array([-3.0, -1.0, 1.0, 3.0])
    v = np.array([-2.0, 0.0, 2.0, -2.5, 2.5])
    np.testing.assert_array_equal(oq.nearest_centroid(v, c), [1, 2, 3, 0, 3])


# ------------------------------------------------------- T4 1-bit + packing
def test_one_bit_toy_and_bitstring():
    g = golden("one_bit_toy.json")
    c = np.array(g["codebook"])
    idx = oq.nearest_centroid(np.array(g["x"]), c)
    assert list(idx) == g["indices"]
    np.testing.assert_allclose(c[idx], g["xhat"])
    words = oq.pack_codes(idx[None, :], 1)
    bits = "".join(str((int(words[0, 0]) >> j) & 1) for j in range(len(idx)))
    assert bits == g["bitstring"]


@pytest.mark.parametrize("d,b", [(4, 1), (32, 3), (64, 2), (96, 3), (128, 3), (128, 4), (160, 1)])
def test_pack_matches_big_integer_stream(d, b):
    rng = np.random.default_rng(d * 10 + b)
    idx = rng.integers(0, 1 << b, size=(3, d))
    words = oq.pack_codes(idx, b)
    W = oq.words_per_vector(d, b)
    assert words.shape == (3, W) and W % 4 == 0 and W * 32 >= b * d
    for r in range(3):
        stream = 0
        for j in range(d):
            stream |= int(idx[r, j]) << (j * b)
        ref = [(stream >> (32 * w)) & 0xFFFFFFFF for w in range(W)]
        assert [int(v) for v in words[r]] == ref
    np.testing.assert_array_equal(oq.unpack_codes(words, d, b), idx)


# ------------------------------------------------------ T5 2-D MSE pipeline
def test_mse_rotation_2d_example():
    g = golden("mse_rotation_2d.json")
    R = np.array(g["R"])
    c = np.array(g["codebook"])
    idx, s, v = oq.mse_quantize(np.array([g["x"]]), R, c, 1.0)
    np.testing.assert_allclose(v[0], g["y"], atol=1e-12)
    assert list(idx[0]) == g["indices"]
    np.testing.assert_allclose(c[idx[0]], g["yhat"])
    xh = oq.mse_dequantize(idx, s, R, c, 1.0)
    np.testing.assert_allclose(xh[0], g["xhat"], atol=1e-12)


# ------------------------------------------------------- T6 Prod / QJL toy
def test_prod_qjl_2d_example():
    g = golden("prod_qjl_2d.json")
    S = np.array(g["S"])
    r = np.array([g["r"]])
    bits, gamma, p = oq.qjl_encode(r, S)
    assert _rounded(gamma[0], 4) == g["gamma"]
    np.testing.assert_allclose(np.round(p[0], 4), g["Sr"], atol=0)
    assert abs(p[0, 1]) < 1e-15 and bits[0, 1] == 1
    # sign(0) = +1 on an exact zero (dyadic operands, exact products)
    b0, _, p0 = oq.qjl_encode(np.array([[0.25, -0.25]]), np.array([[0.5, -0.5], [0.5, 0.5]]))
    assert p0[0, 1] == 0.0 and b0[0, 1] == 1 and b0[0, 0] == 1
    b1, _, _ = oq.qjl_encode(np.array([[-0.25, 0.125]]), np.array([[1.0, 0.0], [0.0, 1.0]]))
    assert list(b1[0]) == [0, 1]
    assert list(2 * bits[0] - 1) == g["signs"]
    np.testing.assert_allclose(np.round((2 * bits[0] - 1) @ S, 3), g["St_signs"])
    assert _rounded(gamma[0] * math.sqrt(math.pi / 2) / 2, 4) == g["scale"]
    corr = oq.qjl_correction(bits, gamma, S)[0]
    np.testing.assert_allclose(np.round(corr, 3), g["corr"])
    xh = np.array(g["xhat_mse"]) + corr
    np.testing.assert_allclose(np.round(xh, 3), g["xhat_prod"])
    y = np.array(g["query_y"])
    assert _rounded(float(y @ xh), 3) == g["ip_prod"]
    assert _rounded(float(y @ np.array(g["xhat_mse"])), 3) == g["ip_mse"]
    assert _rounded(float(y @ np.array(g["x"])), 3) == g["ip_true"]


# ---------------------------------------------------- T7/T8 codebook values
def test_centroids_gaussian_limit_match_printed():
    g = golden("centroids_unit_variance.json")
    c1 = ocb.build_codebook(128, 1, "gauss")["centroids"]
    assert abs(c1[1] - math.sqrt(2 / math.pi)) < 1e-4
    np.testing.assert_allclose(c1, g["b1"], atol=0.5e-4 + 1e-12)
    c2 = ocb.build_codebook(128, 2, "gauss")["centroids"]
    np.testing.assert_allclose(np.round(c2, g["printed_digits"]), g["b2"], atol=1e-12)


@pytest.mark.parametrize("d", [16, 64, 128, 1536])
def test_one_bit_beta_centroid_closed_form(d):
    cbk = ocb.build_codebook(d, 1, "beta")
    ref = math.sqrt(d) * ocb.beta_abs_mean(d)
    assert abs(cbk["centroids"][1] - ref) < 1e-5
    assert abs(cbk["centroids"][0] + ref) < 1e-5
    assert cbk["thresholds"][0] == 0.0


def test_beta_density_is_a_density_with_variance_one_over_d():
    for d in (8, 128, 1024):
        m0 = integrate.quad(lambda x: ocb.beta_coordinate_density(np.array([x]), d)[0], -1, 1)[0]
        m2 = integrate.quad(lambda x: x * x * ocb.beta_coordinate_density(np.array([x]), d)[0], -1, 1)[0]
        assert abs(m0 - 1) < 1e-9
        assert abs(m2 * d - 1) < 1e-9


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_codebook_stationarity_by_quadrature(b):
    """Each centroid is (close to) the conditional mean of its cell and each
    threshold the midpoint, checked on the continuous density by adaptive
    quadrature; the grid distortion equals the quadrature distortion."""
    d = 128
    cbk = ocb.build_codebook(d, b, "beta")
    c, t = cbk["centroids_raw"], cbk["thresholds_raw"]
    np.testing.assert_allclose(t, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(c, -c[::-1], atol=1e-15)
    edges = np.concatenate([[-1.0], t, [1.0]])
    f = lambda x: ocb.beta_coordinate_density(np.array([x]), d)[0]  # noqa: E731
    dist = 0.0
    for k in range(len(c)):
        m0 = integrate.quad(f, edges[k], edges[k + 1], epsabs=1e-14, epsrel=1e-12, limit=200)[0]
        m1 = integrate.quad(lambda x: x * f(x), edges[k], edges[k + 1], epsabs=1e-14, epsrel=1e-12, limit=200)[0]
        # 300 iterations leave Lloyd ~1e-4 (unit-variance units) from the fixed point
        assert abs(m1 / m0 - c[k]) * math.sqrt(d) < 3e-4
        dist += integrate.quad(lambda x: (x - c[k]) ** 2 * f(x), edges[k], edges[k + 1],
                               epsabs=1e-15, epsrel=1e-12, limit=200)[0]
    assert abs(dist * d - cbk["distortion"]) < 1e-6


# ------------------------------------------------------- T9/T10 distortion
def test_dmse_table_and_bound():
    g = golden("dmse_table.json")
    for b, printed in zip(g["b"], g["dmse_printed"]):
        dg = ocb.build_codebook(128, b, "gauss")["distortion"]
        db = ocb.build_codebook(128, b, "beta")["distortion"]
        digits = len(repr(printed).split(".")[1])
        # the printed table is the Gaussian-limit Lloyd-Max distortion cut to its digits
        assert math.floor(dg * 10 ** digits) / 10 ** digits == pytest.approx(printed, abs=1e-12)
        # exact-d Beta codebook: slightly lower, within 2 %
        assert db <= dg and (dg - db) / dg < 0.02
        assert db <= ocb.mse_upper_bound(b)
        # lower bound 4^-b (Shannon) holds too
        assert db >= 4.0 ** (-b)


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_empirical_mse_matches_codebook_and_bound(b):
    d, n = 128, 3000
    rng = np.random.default_rng(100 + b)
    Pi = orot.haar_rotation(rng.standard_normal((d, d)))
    X = rng.standard_normal((n, d)) * np.exp(rng.standard_normal((n, 1)))  # any norms
    cbk = ocb.build_codebook(d, b, "beta")
    idx, s, _ = oq.mse_quantize(X, Pi, cbk["centroids"], math.sqrt(d))
    Xh = oq.mse_dequantize(idx, s, Pi, cbk["centroids"], math.sqrt(d))
    err = ((X - Xh) ** 2).sum(axis=1) / s ** 2
    mean, sem = err.mean(), err.std() / math.sqrt(n)
    assert abs(mean - cbk["distortion"]) < 5 * sem
    assert mean <= ocb.mse_upper_bound(b)
    # rotation does not change the error: ‖x - x̂‖ = ‖y - ŷ‖ (unit-vector units)
    yh = cbk["centroids"][idx] / math.sqrt(d)
    y = (X / s[:, None]) @ Pi.T
    np.testing.assert_allclose(((y - yh) ** 2).sum(axis=1), err, rtol=1e-9)


@pytest.mark.parametrize("b", [2, 3, 4])
def test_hadamard_rotation_distortion_on_kv_rows(b):
    """The randomized Hadamard rotation H·diag(σ)/√d at d = 128 against the Haar
    rotation on the same KV-like rows (fp16 N(0, 1) with channels 0-3 x10):
    both stay under the (√3π/2)·4^-b guarantee, and the Hadamard rotation's
    distortion is within 20 % of the Haar one (on these rows it is lower: the
    outlier channels spread evenly over every coordinate).  On rows without
    outlier channels both match the codebook distortion."""
    d = 128
    cbk = ocb.build_codebook(d, b, "beta")
    Pi_haar = orot.haar_rotation(synth.gaussian_matrix(7, d))
    Pi_had = orot.hadamard_rotation(d, synth.hadamard_signs(7, d))

    def mse(X, Pi):
        idx, s, _ = oq.mse_quantize(X, Pi, cbk["centroids"], math.sqrt(d))
        Xh = oq.mse_dequantize(idx, s, Pi, cbk["centroids"], math.sqrt(d))
        err = ((X - Xh) ** 2).sum(axis=1) / s ** 2
        return err.mean(), err.std() / math.sqrt(len(err))

    K, _ = synth.kv_layer(7, 0, 1, 4, 1000, d)
    X = K.reshape(-1, d).astype(np.float64)
    m_haar, _ = mse(X, Pi_haar)
    m_had, _ = mse(X, Pi_had)
    assert m_haar <= ocb.mse_upper_bound(b) and m_had <= ocb.mse_upper_bound(b)
    assert abs(m_had - m_haar) <= 0.2 * m_haar
    G = synth.gaussian_rows(8, 4000, d).astype(np.float64)
    for Pi in (Pi_haar, Pi_had):
        m, sem = mse(G, Pi)
        assert abs(m - cbk["distortion"]) < 5 * sem


def test_zero_vector_encodes_to_zero():
    d = 32
    Pi = orot.haar_rotation(np.random.default_rng(1).standard_normal((d, d)))
    cbk = ocb.build_codebook(d, 3)
    X = np.zeros((2, d))
    X[1, 3] = 2.0
    idx, s, _ = oq.mse_quantize(X, Pi, cbk["centroids"], math.sqrt(d))
    assert s[0] == 0 and not idx[0].any()
    assert np.all(oq.mse_dequantize(idx, s, Pi, cbk["centroids"], math.sqrt(d))[0] == 0)


# --------------------------------------------------------- T11 rotation
@pytest.mark.parametrize("d", [2, 32, 128, 1536])
def test_haar_rotation_invariants(d):
    G = np.random.default_rng(d).standard_normal((d, d))
    Pi = orot.haar_rotation(G)
    assert np.abs(Pi.T @ Pi - np.eye(d)).max() < 1e-13 * max(1, d / 128)
    # sign fix: Πᵀ G is upper triangular with a positive diagonal
    R = Pi.T @ G
    assert np.abs(np.tril(R, -1)).max() < 1e-10 * d
    assert np.all(np.diag(R) > 0)
    x, q = np.random.default_rng(d + 1).standard_normal((2, d))
    assert abs(np.linalg.norm(Pi @ x) - np.linalg.norm(x)) < 1e-12 * np.linalg.norm(x)
    assert abs((Pi @ q) @ (Pi @ x) - q @ x) < 1e-11 * np.linalg.norm(q) * np.linalg.norm(x)


# --------------------------------------------------------- T12 shrinkage
def test_one_bit_inner_product_shrinkage():
    """E_Π ⟨q, x̂⟩ = d·c₁²·⟨q, x⟩ exactly for the b=1 codebook c₁ = E|X|, and
    d·c₁² -> 2/π as d grows (the 2/π shrinkage of the pages)."""
    d, trials = 64, 1500
    rng = np.random.default_rng(7)
    x = rng.standard_normal(d)
    x /= np.linalg.norm(x)
    q = x + 0.7 * rng.standard_normal(d)
    cbk = ocb.build_codebook(d, 1)
    vals = []
    for _ in range(trials):
        Pi = orot.haar_rotation(rng.standard_normal((d, d)))
        idx, s, _ = oq.mse_quantize(x[None], Pi, cbk["centroids"], math.sqrt(d))
        vals.append(oq.mse_dequantize(idx, s, Pi, cbk["centroids"], math.sqrt(d))[0] @ q)
    vals = np.array(vals)
    factor = d * ocb.beta_abs_mean(d) ** 2
    assert abs(vals.mean() - factor * (q @ x)) < 4 * vals.std() / math.sqrt(trials)
    assert abs(4096 * ocb.beta_abs_mean(4096) ** 2 - 2 / math.pi) < 1e-4


# --------------------------------------------------------- T13 QJL
def test_qjl_inner_product_is_unbiased():
    d, trials = 48, 4000
    rng = np.random.default_rng(11)
    r = rng.standard_normal(d) * 0.3
    q = rng.standard_normal(d)
    est = []
    for _ in range(trials):
        S = rng.standard_normal((d, d))
        bits, gamma, _ = oq.qjl_encode(r[None], S)
        est.append(oq.qjl_correction(bits, gamma, S)[0] @ q)
    est = np.array(est)
    assert abs(est.mean() - q @ r) < 4 * est.std() / math.sqrt(trials)
    # variance bound (π/2)·γ²‖q‖²/m
    assert est.var() <= math.pi / 2 * (r @ r) * (q @ q) / d * 1.1


def test_prod_estimator_is_unbiased_over_S():
    """The full Prod estimate ⟨q, x̂_prod⟩ is unbiased for ⟨q, x⟩ (Π fixed,
    S random), while the MSE-only estimate is biased."""
    d, trials = 32, 3000
    rng = np.random.default_rng(21)
    Pi = orot.haar_rotation(rng.standard_normal((d, d)))
    x = rng.standard_normal(d) * 2.0
    q = x + rng.standard_normal(d)
    cb2 = ocb.build_codebook(d, 1)
    est = []
    for _ in range(trials):
        S = rng.standard_normal((d, d))
        e = oq.prod_quantize(x[None], Pi, S, cb2["centroids"], math.sqrt(d))
        est.append(oatt.prod_scores(q[None], e["idx"], e["s"], e["bits"], e["gamma"], Pi, S,
                                    cb2["centroids"], math.sqrt(d))[0, 0])
    est = np.array(est)
    assert abs(est.mean() - q @ x) < 4 * est.std() / math.sqrt(trials)
    idx, s, _ = oq.mse_quantize(x[None], Pi, cb2["centroids"], math.sqrt(d))
    mse_only = oatt.mse_scores(q[None], idx, s, Pi, cb2["centroids"], math.sqrt(d))[0, 0]
    assert abs(mse_only - q @ x) > 8 * est.std() / math.sqrt(trials)


def test_prod_residual_in_rotated_domain_identity():
    # r = u - Πᵀŷ equals Πᵀ(y - ŷ) and γ = ‖y - ŷ‖ (rotation invariance)
    d = 64
    rng = np.random.default_rng(3)
    Pi = orot.haar_rotation(rng.standard_normal((d, d)))
    S = rng.standard_normal((d, d))
    X = rng.standard_normal((50, d))
    cb2 = ocb.build_codebook(d, 2)
    e = oq.prod_quantize(X, Pi, S, cb2["centroids"], math.sqrt(d))
    y = e["v"] / math.sqrt(d)
    yh = cb2["centroids"][e["idx"]] / math.sqrt(d)
    np.testing.assert_allclose(e["gamma"], np.linalg.norm(y - yh, axis=1), rtol=1e-12)
    np.testing.assert_allclose(e["p"], (y - yh) @ Pi @ S.T, atol=1e-12)


# --------------------------------------------------------- T14 attention
def test_decode_attention_matches_torch_sdpa():
    torch = pytest.importorskip("torch")
    B, Hq, Hkv, T, d, b = 2, 8, 2, 37, 32, 3
    rng = np.random.default_rng(9)
    Pi = orot.haar_rotation(rng.standard_normal((d, d)))
    cbk = ocb.build_codebook(d, b)
    K = rng.standard_normal((B * Hkv * T, d)) * 3
    V = rng.standard_normal((B * Hkv * T, d))
    q = rng.standard_normal((B, Hq, d))
    ki, ks, _ = oq.mse_quantize(K, Pi, cbk["centroids"], math.sqrt(d))
    vi, vs, _ = oq.mse_quantize(V, Pi, cbk["centroids"], math.sqrt(d))
    Kh = oatt.dequantize_cache(ki, ks, Pi, cbk["centroids"], math.sqrt(d), B, Hkv, T)
    Vh = oatt.dequantize_cache(vi, vs, Pi, cbk["centroids"], math.sqrt(d), B, Hkv, T)
    out = oatt.decode_attention(q, Kh, Vh, 1 / math.sqrt(d))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, :, None, :],
        torch.from_numpy(Kh).repeat_interleave(Hq // Hkv, dim=1),
        torch.from_numpy(Vh).repeat_interleave(Hq // Hkv, dim=1),
        scale=1 / math.sqrt(d))[:, :, 0, :].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_decode_attention_degenerate_cases():
    d = 16
    rng = np.random.default_rng(4)
    Vh = rng.standard_normal((1, 1, 5, d))
    q = rng.standard_normal((1, 2, d))
    # one token: output is that value
    out = oatt.decode_attention(q, rng.standard_normal((1, 1, 1, d)), Vh[:, :, :1], 0.3)
    np.testing.assert_allclose(out[0, 0], Vh[0, 0, 0], rtol=1e-14)
    # identical keys: output is the mean of the values
    Kh = np.repeat(rng.standard_normal((1, 1, 1, d)), 5, axis=2)
    out = oatt.decode_attention(q, Kh, Vh, 0.3)
    np.testing.assert_allclose(out[0, 1], Vh[0, 0].mean(axis=0), rtol=1e-12)
    # a key far ahead of the rest: output is its value
    Kh = np.zeros((1, 1, 5, d))
    Kh[0, 0, 3] = 1e3 * q[0, 0]
    out = oatt.decode_attention(q[:, :1], Kh, Vh, 1.0)
    np.testing.assert_allclose(out[0, 0], Vh[0, 0, 3], rtol=1e-12)


def test_mse_scores_equal_reconstruction_inner_products():
    # score = ⟨q, x̂⟩ with x̂ rebuilt independently by rotating ŷ back
    d = 32
    rng = np.random.default_rng(12)
    Pi = orot.haar_rotation(rng.standard_normal((d, d)))
    cbk = ocb.build_codebook(d, 2)
    X = rng.standard_normal((20, d))
    Q = rng.standard_normal((3, d))
    idx, s, _ = oq.mse_quantize(X, Pi, cbk["centroids"], math.sqrt(d))
    sc = oatt.mse_scores(Q, idx, s, Pi, cbk["centroids"], math.sqrt(d))
    yh = cbk["centroids"][idx] / math.sqrt(d)
    ref = np.einsum("md,nd->mn", Q @ Pi.T, yh) * s[None, :]  # ⟨Πq, ŷ⟩ s
    np.testing.assert_allclose(sc, ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------- T15 Hadamard
@pytest.mark.parametrize("d", [1, 2, 8, 128, 256])
def test_sylvester_matches_scipy(d):
    np.testing.assert_array_equal(orot.hadamard(d), scipy.linalg.hadamard(d))


@pytest.mark.parametrize("d", [12, 24, 96, 1536, 3072])
def test_hadamard_orthogonality(d):
    H = orot.hadamard(d)
    assert set(np.unique(H)) == {-1.0, 1.0}
    np.testing.assert_array_equal(H @ H.T, d * np.eye(d))


def test_paley_twelve_structure():
    H = orot.paley_hadamard_12()
    np.testing.assert_array_equal(H @ H.T, 12 * np.eye(12))
    S = H - np.eye(12)
    np.testing.assert_array_equal(S, -S.T)  # skew Hadamard
    assert np.all(H[0] == 1)


def test_hadamard_rotation_is_orthogonal():
    d = 1536
    signs = np.where(np.random.default_rng(0).integers(0, 2, d) == 1, 1.0, -1.0)
    P = orot.hadamard_rotation(d, signs)
    assert np.abs(P @ P.T - np.eye(d)).max() < 1e-12


# ------------------------------------------------ near-threshold bands
# The parity tests excuse an index mismatch only inside the band
# |v - t_k| <= 1e-6 · max(1, |t_k|) around a codebook threshold, and a QJL bit
# only inside |(S·r)_j| <= 1e-6 · ‖S_j‖₂ · γ.  These values are built by hand so
# that a band that is absolute instead of relative, relative to plain |t_k|
# (no band at t = 0), uses column norms of S, drops γ or takes < for <= selects
# different coordinates.
def test_near_threshold_band_selects_exactly_the_hand_built_coordinates():
    c = np.array([-5.0, -3.0, 3.0, 5.0])  # thresholds -4, 0, 4
    v = np.array([
        1.0e-6,          # t = 0, on the band edge (1e-6 · max(1, 0)): inside
        0.5e-6,          # t = 0, inside (a band of 1e-6·|t| would be empty here)
        -0.99e-6,        # t = 0, inside from below
        1.01e-6,         # t = 0, outside
        4.0 + 3.9e-6,    # t = 4: band 4e-6, inside (an absolute 1e-6 band would miss it)
        4.0 - 3.9e-6,    # inside from below
        4.0 + 4.1e-6,    # outside
        -4.0 - 2.0e-6,   # t = -4, inside
        -4.0 + 4.2e-6,   # outside
        2.0,             # far from every threshold
    ])
    want = [True, True, True, False, True, True, False, True, False, False]
    assert list(oq.near_threshold(v, c)) == want


def test_near_threshold_band_keeps_the_unit_floor_below_one():
    c = np.array([-0.3, -0.1, 0.1, 0.3])  # thresholds -0.2, 0, 0.2: all |t| < 1
    v = np.array([0.2 + 0.9e-6, 0.2 + 1.1e-6, -0.2 - 0.95e-6, 0.2 + 0.15e-6])
    # the band is 1e-6 absolute here (max(1, 0.2) = 1), not 0.2e-6
    assert list(oq.near_threshold(v, c)) == [True, False, True, True]


def test_near_threshold_shape_and_dtype():
    c = np.array([-1.0, 1.0])
    v = np.zeros((3, 4))
    m = oq.near_threshold(v, c)
    assert m.shape == (3, 4) and m.dtype == bool and m.all()


def test_qjl_band_uses_row_norms_of_s_and_gamma():
    # rows of S with norms 5 and 1; its column norms are 5 and 4, so a
    # column-norm band differs in the second coordinate
    S = np.array([[3.0, 4.0], [0.0, 1.0]])
    assert np.allclose(np.sqrt((S * S).sum(1)), [5.0, 1.0])
    gamma = np.array([2.0, 2.0, 2.0, 0.5, 1.0])
    # bands per row: 1e-6·5·γ and 1e-6·1·γ
    p = np.array([
        [0.99e-5, 1.99e-6],    # both inside (γ = 2: 1e-5, 2e-6)
        [1.01e-5, 2.01e-6],    # both outside
        [-0.99e-5, -2.1e-6],   # first inside from below, second outside
        [2.4e-6, 0.49e-6],     # γ = 0.5: bands 2.5e-6 and 0.5e-6, both inside
        [5.1e-6, 1.0e-6],      # γ = 1: first outside; second exactly on its band (<=)
    ])
    want = np.array([[True, True], [False, False], [True, False], [True, True], [False, True]])
    np.testing.assert_array_equal(oq.qjl_near_zero(p, gamma, S), want)


def test_qjl_band_is_empty_for_a_zero_residual():
    # γ = 0 (a zero vector or an exact MSE code) gives a band of width zero:
    # only an exactly zero projection lies in it
    S = np.eye(3)
    m = oq.qjl_near_zero(np.array([[0.0, 1e-30, -1e-30]]), np.array([0.0]), S)
    assert m.tolist() == [[True, False, False]]


def test_band_width_by_uniform_draws_near_each_threshold():
    # Draws uniform within ±1e-5 of each threshold of the b = 3 codebook fall in
    # the band with probability 1e-6·max(1,|t_k|) / 1e-5 (binomial count).
    cb = ocb.build_codebook(128, 3, density="gauss")
    t = 0.5 * (cb["centroids"][:-1] + cb["centroids"][1:])
    assert np.diff(t).min() > 1e-3  # no draw reaches a neighbour's band
    rng = np.random.default_rng(7)
    width, n = 1e-5, 500_000
    for tk in t:
        v = tk + rng.uniform(-width, width, n)
        hits = int(oq.near_threshold(v, cb["centroids"]).sum())
        pr = 1e-6 * max(1.0, abs(tk)) / width
        assert abs(hits - n * pr) <= 6 * math.sqrt(n * pr * (1 - pr)), (tk, hits, n * pr)


# ------------------------------------------------ b + 1/2 bits per coordinate
def test_half_bit_widths_give_the_pages_bytes_per_token():
    """The pages' 672 B per token and layer against 4 KB uncompressed: 16 vectors
    of 42 B, i.e. 40 B of codes (2.5 bits x 128) and a 2-byte norm."""
    g = golden("kv_bytes_per_token.json")
    vectors = g["uncompressed_bytes"] // (g["head_dim"] * g["uncompressed_bytes_per_value"])
    assert vectors == 16
    per_vec = g["compressed_bytes"] / vectors
    w = oq.mixed_widths(128, 2)
    assert int(w.sum()) == 320 and oq.mixed_words_per_vector(128, 2) * 4 == 40
    assert per_vec == 40 + 2
    assert int(oq.mixed_widths(128, 1).sum()) == 192 and int(oq.mixed_widths(128, 3).sum()) == 448
    # exactly half of every block of 16 coordinates carries the extra bit, the first eight
    assert ((w == 3).reshape(-1, 16).sum(axis=1) == 8).all() and (w.reshape(-1, 16)[:, :8] == 3).all()


def test_varwidth_packing_hand_example():
    """d = 16, b = 1: coordinates 0-7 take two bits, 8-15 one bit.  Stream bits
    0-15 are 11 00 10 01 00 00 00 00 (codes 3, 0, 1, 2, 0, 0, 0, 0, LSB first),
    bits 16-23 are 1 0 1 0 0 0 0 1."""
    idx = np.array([[3, 0, 1, 2, 0, 0, 0, 0, 1, 0, 1, 0, 0, 0, 0, 1]])
    expect = (1 << 0) | (1 << 1) | (1 << 4) | (1 << 7) | (1 << 16) | (1 << 18) | (1 << 23)
    words = oq.pack_varwidth(idx, oq.mixed_widths(16, 1))
    assert words.shape == (1, 1) and int(words[0, 0]) == expect
    np.testing.assert_array_equal(oq.unpack_varwidth(words, oq.mixed_widths(16, 1)), idx)


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_varwidth_packing_with_one_width_is_the_canonical_packing(b):
    rng = np.random.default_rng(40 + b)
    idx = rng.integers(0, 1 << b, size=(50, 128))
    a = oq.pack_varwidth(idx, [b] * 128)
    c = oq.pack_codes(idx, b)
    np.testing.assert_array_equal(a, c[:, :a.shape[1]])
    assert not c[:, a.shape[1]:].any()


def test_half_bit_pair_blocks_interleave_the_two_vectors():
    """b = 2: coordinate 0 (3 bits) holds the even vector's code in block bits
    0-2 and the odd vector's in 3-5; coordinate 8 (2 bits) starts at block bit
    2·(8·3) = 48, i.e. word 1 bit 16."""
    idx = np.zeros((2, 128), dtype=np.int64)
    idx[0, 0], idx[1, 0], idx[0, 8], idx[1, 8] = 5, 2, 1, 3
    words = oq.pack_mixed_pairs(idx, 2)
    assert words.shape == (1, 20)
    assert int(words[0, 0]) == 5 | (2 << 3)
    assert int(words[0, 1]) == (1 << 16) | (3 << 18)
    assert not words[0, 2:].any()


def test_half_bit_quantize_is_a_brute_force_nearest_search_per_width():
    d, b = 16, 1
    rng = np.random.default_rng(7)
    X = rng.standard_normal((40, d))
    Pi = orot.haar_rotation(rng.standard_normal((d, d)))
    lo, hi = ocb.build_codebook(d, b)["centroids"], ocb.build_codebook(d, b + 1)["centroids"]
    idx, s, v = oq.mixed_quantize(X, Pi, lo, hi, b, math.sqrt(d))
    for n in range(X.shape[0]):
        for j in range(d):
            cb = hi if j % 16 < 8 else lo
            best = min(range(len(cb)), key=lambda k: abs(v[n, j] - cb[k]))
            assert idx[n, j] == best
    # and the rotated coordinates are √d·Π·x/‖x‖
    np.testing.assert_allclose(v, math.sqrt(d) * (X / np.linalg.norm(X, axis=1, keepdims=True)) @ Pi.T,
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("b", [1, 2, 3])
def test_half_bit_distortion_is_the_mean_of_the_two_codebooks(b):
    """Per-coordinate errors add, and each half of the (exchangeable) rotated
    coordinates carries its own codebook's distortion: E‖u - û‖² =
    (D_b + D_(b+1)) / 2, with D_(b+1)/2 on the (b+1)-bit half."""
    d, n = 128, 3000
    rng = np.random.default_rng(300 + b)
    Pi = orot.haar_rotation(rng.standard_normal((d, d)))
    X = rng.standard_normal((n, d)) * np.exp(rng.standard_normal((n, 1)))
    cl, ch = ocb.build_codebook(d, b), ocb.build_codebook(d, b + 1)
    idx, s, _ = oq.mixed_quantize(X, Pi, cl["centroids"], ch["centroids"], b, math.sqrt(d))
    Xh = oq.mixed_dequantize(idx, s, Pi, cl["centroids"], ch["centroids"], b, math.sqrt(d))
    err = ((X - Xh) ** 2).sum(axis=1) / s ** 2
    want = 0.5 * (cl["distortion"] + ch["distortion"])
    assert abs(err.mean() - want) < 5 * err.std() / math.sqrt(n)
    assert ch["distortion"] < err.mean() < cl["distortion"]
    # the (b+1)-bit half alone, in the rotated domain
    y = (X / s[:, None]) @ Pi.T
    yh = (Xh / s[:, None]) @ Pi.T
    hi = oq.mixed_widths(d, b) == b + 1
    e_hi = ((y - yh)[:, hi] ** 2).sum(axis=1)
    assert abs(e_hi.mean() - ch["distortion"] / 2) < 5 * e_hi.std() / math.sqrt(n)


def test_half_bit_band_uses_each_coordinates_own_codebook():
    d, b = 16, 2
    lo, hi = ocb.build_codebook(d, b)["centroids"], ocb.build_codebook(d, b + 1)["centroids"]
    t_lo, t_hi = 0.5 * (lo[1:] + lo[:-1]), 0.5 * (hi[1:] + hi[:-1])
    v = np.full((1, d), 5.0)        # far from every threshold
    v[0, 0] = t_hi[2]               # a (b+1)-bit coordinate on its own threshold
    v[0, 8] = t_lo[0]               # a b-bit coordinate on its own threshold
    v[0, 9] = t_hi[0]               # a b-bit coordinate on a threshold of the other codebook
    v[0, 1] = t_lo[0]               # and the reverse
    band = oq.mixed_near_threshold(v, lo, hi, b)
    assert band[0, 0] and band[0, 8]
    assert not band[0, 9] and not band[0, 1]
    assert band.sum() == 2
