"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bars (from the benchmark spec of the method's build):
  * packed indices bit-exact except coordinates within 1e-6 (relative) of a
    decision threshold; that fraction is reported and must be <= 1e-5;
  * QJL bits bit-exact except |(S r)_j| <= 1e-6·‖S_j‖·γ, for vectors whose MSE
    indices match;
  * norms within 1e-6 relative; scores within 1e-4·‖q‖‖x‖; attention outputs
    within 2e-3·‖out‖ per head.
Scores and attention are evaluated by the oracle on the GPU's own codes, so
encode parity and read-path parity are checked separately.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import kv_cache_vector_tq_gb300 as tq  # noqa: E402
from kv_cache_vector_tq_gb300 import synth  # noqa: E402
from oracle import attention as oatt  # noqa: E402
from oracle import codebook as ocb  # noqa: E402
from oracle import quantizer as oq  # noqa: E402
from oracle import rotation as orot  # noqa: E402

pytestmark = pytest.mark.gpu

BAND_FRAC_MAX = 1e-5


def expected_band_frac(centroids):
    """Expected share of coordinates in the 1e-6 band for v ~ N(0, 1) (the
    large-d law of a rotated unit-vector coordinate in unit-variance units):
    Σ_k 2·1e-6·max(1, |t_k|)·φ(t_k)."""
    c = np.asarray(centroids, dtype=np.float64)
    t = 0.5 * (c[:-1] + c[1:])
    return float(np.sum(2e-6 * np.maximum(1.0, np.abs(t)) * np.exp(-0.5 * t * t) / math.sqrt(2 * math.pi)))


def band_count_ok(band, centroids):
    """The band holds at most 1e-5 of the coordinates: the codebook's expected
    share is below 1e-5, and the observed count is within a Poisson bound of
    that expectation (small samples see zero, one or two such coordinates)."""
    ef = expected_band_frac(centroids)
    mean = ef * band.size
    return ef <= BAND_FRAC_MAX and band.sum() <= mean + 5 * math.sqrt(mean) + 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()


_cb_cache = {}


def oracle_codebook(d, b):
    if (d, b) not in _cb_cache:
        _cb_cache[(d, b)] = ocb.build_codebook(d, b)
    return _cb_cache[(d, b)]


def make_pair(seed, d, b, mode=tq.TQ_MSE, rot="dense"):
    """Product context and the oracle's own rotation/QJL matrices for one seed
    (rot "dense": Haar rotation from QR; "hadamard": H·diag(σ)/√d)."""
    S = synth.qjl_matrix(seed, d) if mode == tq.TQ_PROD else None
    if rot == "hadamard":
        sig = synth.hadamard_signs(seed, d)
        ctx = tq.Context(d, b, mode, tq.TQ_ROT_HADAMARD, sig, S)
        return ctx, orot.hadamard_rotation(d, sig), S
    G = synth.gaussian_matrix(seed, d)
    ctx = tq.Context(d, b, mode, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(G), S)
    return ctx, orot.haar_rotation(G), S


def gpu_encode(ctx, x_np, layout=tq.TQ_LAYOUT_TOKEN, n=None):
    x = torch.from_numpy(np.ascontiguousarray(x_np)).cuda()
    cs = tq.CodeSet(ctx, n or x_np.shape[0], layout)
    tq.tq_encode(ctx, x, cs)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    return cs


def check_mse_encode(ctx, Pi, X, b, cs=None, first=0):
    d = X.shape[1]
    cb = oracle_codebook(d, b)
    idx_ref, s_ref, v = oq.mse_quantize(X.astype(np.float64), Pi, cb["centroids"], math.sqrt(d))
    band = oq.near_threshold(v, cb["centroids"])
    band[s_ref == 0.0] = False  # zero vectors are coded 0 by definition, not by a threshold test
    idx = tq.tq_unpack_indices(cs, first, X.shape[0]).astype(np.int64)
    mism = (idx != idx_ref) & ~band
    assert not mism.any(), f"{mism.sum()} index mismatches outside the band, rows {np.nonzero(mism.any(1))[0][:10]}"
    frac = band.mean()
    assert band_count_ok(band, cb["centroids"]), f"near-threshold fraction {frac} ({band.sum()} of {band.size})"
    norm = cs.norm[first:first + X.shape[0]].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(norm, s_ref, rtol=1e-6, atol=0)
    return idx_ref, band, frac


# ------------------------------------------------------------------ encode
@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_encode_mse_fp32_config1(b):
    """TurboQuant_MSE, d=128, N=4096 fp32 N(0,1) keys with channels 0-3 x20
    (the first workload; b=3 is its own bit width, the others widen it)."""
    ctx, Pi, _ = make_pair(0, 128, b)
    X = synth.gaussian_rows(0, 4096, 128, outlier_cols=4, outlier_scale=20.0)
    cs = gpu_encode(ctx, X)
    idx_ref, band, frac = check_mse_encode(ctx, Pi, X, b, cs)
    # raw words equal the canonical packing wherever no coordinate is in the band
    words = cs.codes.view(torch.int32).cpu().numpy().view(np.uint32).reshape(4096, -1)
    ok = ~band.any(axis=1)
    np.testing.assert_array_equal(words[ok], oq.pack_codes(idx_ref[ok], b))


@pytest.mark.parametrize("d", [32, 64, 96])
@pytest.mark.parametrize("b", [1, 3, 4])
def test_encode_small_dims(d, b):
    ctx, Pi, _ = make_pair(3, d, b)
    X = synth.gaussian_rows(3, 333, d, outlier_cols=2, outlier_scale=5.0)
    cs = gpu_encode(ctx, X)
    idx_ref, band, _ = check_mse_encode(ctx, Pi, X, b, cs)
    words = cs.codes.view(torch.int32).cpu().numpy().view(np.uint32).reshape(333, -1)
    ok = ~band.any(axis=1)
    np.testing.assert_array_equal(words[ok], oq.pack_codes(idx_ref[ok], b))


@pytest.mark.parametrize("N", [1, 31, 33, 129, 1000])
def test_encode_ragged_and_zero_rows(N):
    ctx, Pi, _ = make_pair(5, 128, 3)
    X = synth.gaussian_rows(5, N, 128)
    X[N // 2] = 0.0  # zero vector: s = 0, all codes 0
    cs = gpu_encode(ctx, X)
    check_mse_encode(ctx, Pi, X, 3, cs)
    idx = tq.tq_unpack_indices(cs, N // 2, 1)
    assert not idx.any() and cs.norm[N // 2].item() == 0.0


def test_encode_extreme_magnitudes():
    """Rows scaled by 1e-20, 1e-25 (squares below the fp32 range) and 1e22
    (above it), and rows with a single non-zero value: the norm and the codes
    follow the definition at any magnitude."""
    ctx, Pi, _ = make_pair(6, 128, 3)
    X = synth.gaussian_rows(6, 64, 128)
    X[1] *= 1e-20
    X[2] *= 1e-25
    X[3] *= 1e22
    X[4] = 0.0
    X[4, 77] = 2.5e-30
    X[5] = 0.0
    X[5, 0] = -3e30
    cs = gpu_encode(ctx, X)
    check_mse_encode(ctx, Pi, X, 3, cs)


def test_encode_fp16_extreme_rows():
    """fp16 rows at the ends of the fp16 range, which the tensor cores take
    unscaled: full of 65504, of subnormals (6e-8), a single subnormal, a zero
    row, and mixed magnitudes."""
    d, b = 128, 3
    ctx, Pi, _ = make_pair(45, d, b)
    X = synth.gaussian_rows(45, 40, d).astype(np.float16)
    X[0] = np.float16(65504.0) * np.sign(X[0] + np.float16(1e-3))
    X[1] = np.float16(6e-8) * np.sign(X[1] + np.float16(1e-3))
    X[2] = 0.0
    X[2, 17] = np.float16(6e-8)
    X[3] = 0.0
    X[4, :64] = np.float16(65504.0)
    X[4, 64:] = np.float16(1e-4)
    cs = gpu_encode(ctx, X)
    check_mse_encode(ctx, Pi, X.astype(np.float32), b, cs)


@pytest.mark.parametrize("b", [2, 3, 4])
def test_encode_fp16_kv_token_and_pair_layouts(b):
    """fp16 K/V with 4 outlier channels x10 (the KV workloads), both layouts."""
    ctx, Pi, _ = make_pair(0, 128, b)
    K, V = synth.kv_layer(0, 0, 1, 2, 1000, 128)
    for arr, layout in ((K, tq.TQ_LAYOUT_TOKEN), (V, tq.TQ_LAYOUT_PAIR)):
        X = arr.reshape(-1, 128)
        cs = gpu_encode(ctx, X, layout)
        idx_ref, band, _ = check_mse_encode(ctx, Pi, X.astype(np.float32), b, cs)
        if layout == tq.TQ_LAYOUT_PAIR:
            # pair block i: coordinate j of vector 2i+q at bits (2j+q)·b of the block
            words = cs.codes.view(torch.int32).cpu().numpy().view(np.uint32).reshape(-1, 2 * cs.words_per_vec)
            inter = np.zeros((idx_ref.shape[0] // 2, 2 * 128), dtype=np.int64)
            inter[:, 0::2] = idx_ref[0::2]
            inter[:, 1::2] = idx_ref[1::2]
            ok = ~(band[0::2].any(1) | band[1::2].any(1))
            np.testing.assert_array_equal(words[ok], oq.pack_codes(inter[ok], b))


@pytest.mark.parametrize("b", [1, 2, 3, 4])
@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("offset", [0, 1])
def test_encode_pair_layout_widths_and_offsets(b, f16, offset):
    """PAIR layout at every width, fp32 and fp16 rows: an odd row count (the
    last pair block half written) at an even offset (row pairs fill whole
    blocks) and at an odd one (every row shares its block with a row written by
    no one: masked writes).  Slots this call does not own keep what was there
    (the code set starts as all ones)."""
    d, N = 128, 301
    ctx, Pi, _ = make_pair(40 + b, d, b)
    X = synth.gaussian_rows(40 + b, N, d, outlier_cols=4, outlier_scale=10.0)
    if f16:
        X = X.astype(np.float16)
    cs = tq.CodeSet(ctx, N + offset + 1, tq.TQ_LAYOUT_PAIR)
    cs.codes.fill_(-1)
    tq.tq_encode(ctx, torch.from_numpy(np.ascontiguousarray(X)).cuda(), cs, offset=offset)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    check_mse_encode(ctx, Pi, X.astype(np.float32), b, cs, first=offset)
    full = (1 << b) - 1
    untouched = [0] if offset else []
    untouched += [N + offset]
    for v in untouched:
        assert (tq.tq_unpack_indices(cs, v, 1) == full).all()


def test_encode_append_mapping_pair_layout():
    """Cache append: one token per (batch, head) block at position t (odd and
    even), written next to tokens encoded earlier into the same pair blocks."""
    b, cap, blocks = 3, 64, 6
    ctx, Pi, _ = make_pair(2, 128, b)
    X = synth.gaussian_rows(2, blocks * 40, 128).reshape(blocks, 40, 128)
    cs = tq.CodeSet(ctx, blocks * cap, tq.TQ_LAYOUT_PAIR)
    # prefill 37 tokens per block (odd count: the last pair is half written)
    pre = torch.from_numpy(np.ascontiguousarray(X[:, :37].reshape(-1, 128))).cuda()
    tq.tq_encode(ctx, pre, cs, offset=0, group_rows=37, group_stride=cap)
    for t in (37, 38, 39):
        new = torch.from_numpy(np.ascontiguousarray(X[:, t])).cuda()
        tq.tq_encode(ctx, new, cs, offset=t, group_rows=1, group_stride=cap)
    torch.cuda.synchronize()
    cb = oracle_codebook(128, b)
    idx_ref, s_ref, v = oq.mse_quantize(X.reshape(-1, 128).astype(np.float64), Pi, cb["centroids"], math.sqrt(128))
    band = oq.near_threshold(v, cb["centroids"])
    for blk in range(blocks):
        got = tq.tq_unpack_indices(cs, blk * cap, 40).astype(np.int64)
        ref = idx_ref[blk * 40:(blk + 1) * 40]
        bb = band[blk * 40:(blk + 1) * 40]
        assert not ((got != ref) & ~bb).any()
        np.testing.assert_allclose(cs.norm[blk * cap: blk * cap + 40].cpu().numpy(), s_ref[blk * 40:(blk + 1) * 40], rtol=1e-6)


@pytest.mark.parametrize("b,f16", [(3, False), (3, True), (2, True), (4, False)])
def test_encode_prod_config3_sample(b, f16):
    """TurboQuant_Prod (b - 1-bit MSE + 1-bit QJL), unit-norm Gaussian keys, fp32
    and fp16 rows (the fp16 instance reads the rows straight from the TMA tile)."""
    d, N = 128, 20000
    ctx, Pi, S = make_pair(0, d, b, tq.TQ_PROD)
    X = synth.unit_rows(0, N, d)
    if f16:
        X = X.astype(np.float16).astype(np.float32)
        cs = gpu_encode(ctx, X.astype(np.float16))
    else:
        cs = gpu_encode(ctx, X)
    cb = oracle_codebook(d, b - 1)
    e = oq.prod_quantize(X.astype(np.float64), Pi, S, cb["centroids"], math.sqrt(d))
    band = oq.near_threshold(e["v"], cb["centroids"])
    idx, bits = tq.tq_unpack_indices(cs, 0, N, with_bits=True)
    mism = (idx.astype(np.int64) != e["idx"]) & ~band
    assert not mism.any()
    assert band.mean() <= BAND_FRAC_MAX
    rows_ok = (idx.astype(np.int64) == e["idx"]).all(axis=1)
    qband = oq.qjl_near_zero(e["p"], e["gamma"], S)
    bmism = (bits.astype(np.int64) != e["bits"]) & ~qband & rows_ok[:, None]
    assert not bmism.any(), f"{bmism.sum()} QJL bit mismatches"
    # band |p_j| <= 1e-6·‖S_j‖·γ: for a random residual direction p_j/(γ‖S_j‖/√d) ~ N(0,1),
    # so the expected excluded fraction is 2·φ(0)·1e-6·√d (9.0e-6 at d = 128); on this
    # sample the count must lie within 5 Poisson σ of it
    expected = qband.size * 2 * 0.3989422804014327 * 1e-6 * math.sqrt(d)
    assert qband.sum() <= expected + 5 * math.sqrt(expected) + 1
    g = cs.rnorm[:N].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(g[rows_ok], e["gamma"][rows_ok], rtol=1e-5, atol=1e-7)


def _shifted_codebook(d, bm):
    """A codebook that is not symmetric about 0: the Lloyd-Max centroids moved
    by 0.02..0.08, thresholds at the new midpoints (the nearest-centroid rule,
    "TurboQuant 详解", section "痛点 2")."""
    cb = tq.tq_codebook_build(d, bm)
    K = 1 << bm
    c = np.array([cb.centroid[k] for k in range(K)]) + 0.02 + 0.06 * np.arange(K) / K
    for k in range(K):
        cb.centroid[k] = float(c[k])
    for k in range(K - 1):
        cb.threshold[k] = float(0.5 * (c[k] + c[k + 1]))
    return cb, c


@pytest.mark.parametrize("mode", [tq.TQ_MSE, tq.TQ_PROD])
def test_encode_nonsymmetric_codebook(mode):
    """A caller's codebook without the ± symmetry (d = 128, b = 3): the codes
    still follow the nearest-centroid rule and (Prod) the QJL stage."""
    d, b, N = 128, 3, 3000
    bm = b - 1 if mode == tq.TQ_PROD else b
    cb, cen = _shifted_codebook(d, bm)
    S = synth.qjl_matrix(4, d) if mode == tq.TQ_PROD else None
    G = synth.gaussian_matrix(4, d)
    ctx = tq.Context(d, b, mode, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(G), S, codebook=cb)
    Pi = orot.haar_rotation(G)
    X = synth.unit_rows(4, N, d) if mode == tq.TQ_PROD else synth.gaussian_rows(4, N, d, outlier_cols=4,
                                                                                  outlier_scale=10.0)
    cs = gpu_encode(ctx, X)
    if mode == tq.TQ_MSE:
        idx_ref, s_ref, v = oq.mse_quantize(X.astype(np.float64), Pi, cen, math.sqrt(d))
        band = oq.near_threshold(v, cen)
        idx = tq.tq_unpack_indices(cs, 0, N).astype(np.int64)
        assert not ((idx != idx_ref) & ~band).any()
        np.testing.assert_allclose(cs.norm[:N].cpu().numpy(), s_ref, rtol=1e-6)
    else:
        e = oq.prod_quantize(X.astype(np.float64), Pi, S, cen, math.sqrt(d))
        band = oq.near_threshold(e["v"], cen)
        idx, bits = tq.tq_unpack_indices(cs, 0, N, with_bits=True)
        assert not ((idx.astype(np.int64) != e["idx"]) & ~band).any()
        rows_ok = (idx.astype(np.int64) == e["idx"]).all(axis=1)
        qband = oq.qjl_near_zero(e["p"], e["gamma"], S)
        assert not ((bits.astype(np.int64) != e["bits"]) & ~qband & rows_ok[:, None]).any()
        g = cs.rnorm[:N].cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(g[rows_ok], e["gamma"][rows_ok], rtol=1e-5, atol=1e-7)
    assert band.mean() <= BAND_FRAC_MAX


# ------------------------------------------------------------------ scores
def _scores_check(ctx, Pi, S, X, Q, b_mse, prod):
    d = X.shape[1]
    N, M = X.shape[0], Q.shape[0]
    cs = gpu_encode(ctx, X)
    q = torch.from_numpy(np.ascontiguousarray(Q)).cuda()
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(tq.tq_scores_workspace_size(ctx, M) // 4 + 4, dtype=torch.float32, device="cuda")
    tq.tq_scores(ctx, q, cs, out, ws)
    torch.cuda.synchronize()
    cb = oracle_codebook(d, b_mse)
    s = cs.norm[:N].cpu().numpy().astype(np.float64)
    if prod:
        idx, bits = tq.tq_unpack_indices(cs, 0, N, with_bits=True)
        gam = cs.rnorm[:N].cpu().numpy().astype(np.float64)
        ref = oatt.prod_scores(Q.astype(np.float64), idx, s, bits, gam, Pi, S, cb["centroids"], math.sqrt(d))
    else:
        idx = tq.tq_unpack_indices(cs, 0, N)
        ref = oatt.mse_scores(Q.astype(np.float64), idx, s, Pi, cb["centroids"], math.sqrt(d))
    got = out.cpu().numpy().astype(np.float64)
    bound = 1e-4 * np.linalg.norm(Q, axis=1)[:, None] * np.linalg.norm(X.astype(np.float64), axis=1)[None, :]
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"max err/bound {np.max(err / np.maximum(bound, 1e-30))}"
    return np.max(err / np.maximum(bound, 1e-30))


def test_scores_mse_config1():
    ctx, Pi, _ = make_pair(0, 128, 3)
    X = synth.gaussian_rows(0, 4096, 128, outlier_cols=4, outlier_scale=20.0)
    Q = synth.queries(0, 1, 128)
    _scores_check(ctx, Pi, None, X, Q, 3, False)


@pytest.mark.parametrize("b", [1, 2, 4])
def test_scores_mse_bits_and_ragged(b):
    ctx, Pi, _ = make_pair(7, 128, b)
    X = synth.gaussian_rows(7, 1237, 128, outlier_cols=4, outlier_scale=20.0)
    Q = synth.queries(7, 70, 128)  # more than one 64-query launch, ragged
    _scores_check(ctx, Pi, None, X, Q, b, False)


@pytest.mark.parametrize("first,N,M,prod", [
    (0, 1, 1, False),       # one key, one query
    (37, 100, 3, True),     # a key range inside the code set, less than one 128-key tile
    (5, 1000, 130, True),   # three query launches (64, 64, 2), ragged last key tile
    (0, 4096, 64, False),   # whole tiles, a full query launch
])
def test_scores_key_ranges_and_query_counts(first, N, M, prod):
    """Scores over keys [first, first + N) of a larger code set: tiny and
    ragged key counts, key counts that are not multiples of 4, more than one
    64-query launch."""
    d = 128
    mode = tq.TQ_PROD if prod else tq.TQ_MSE
    b = 3
    ctx, Pi, S = make_pair(21, d, b, mode)
    total = first + N + 11
    X = synth.unit_rows(21, total, d) if prod else synth.gaussian_rows(21, total, d, outlier_cols=4, outlier_scale=20.0)
    cs = gpu_encode(ctx, X)
    Q = synth.queries(21, M, d)
    q = torch.from_numpy(np.ascontiguousarray(Q)).cuda()
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(tq.tq_scores_workspace_size(ctx, M) // 4 + 4, dtype=torch.float32, device="cuda")
    tq.tq_scores(ctx, q, cs, out, ws, first=first, N=N)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    b_mse = b - 1 if prod else b
    cb = oracle_codebook(d, b_mse)
    s = cs.norm[first:first + N].cpu().numpy().astype(np.float64)
    if prod:
        idx, bits = tq.tq_unpack_indices(cs, first, N, with_bits=True)
        gam = cs.rnorm[first:first + N].cpu().numpy().astype(np.float64)
        ref = oatt.prod_scores(Q.astype(np.float64), idx, s, bits, gam, Pi, S, cb["centroids"], math.sqrt(d))
    else:
        idx = tq.tq_unpack_indices(cs, first, N)
        ref = oatt.mse_scores(Q.astype(np.float64), idx, s, Pi, cb["centroids"], math.sqrt(d))
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()  # every (query, key) written, nothing outside
    Xs = X[first:first + N].astype(np.float64)
    bound = 1e-4 * np.linalg.norm(Q, axis=1)[:, None] * np.linalg.norm(Xs, axis=1)[None, :]
    assert (np.abs(got - ref) <= bound).all()


@pytest.mark.parametrize("b,M,prod,first,N", [
    (1, 1, False, 0, 4096), (2, 5, False, 3, 777), (3, 1, False, 0, 30001), (3, 8, False, 0, 9000),
    (4, 2, False, 11, 129), (2, 1, True, 0, 4096), (3, 8, True, 5, 1001), (4, 3, True, 0, 65),
    (3, 9, False, 0, 300),  # one query past the small path: the tensor-core scorer
    (3, 1, False, 0, 40000),  # more keys than the small path takes
])
def test_scores_small_query_counts(b, M, prod, first, N):
    """Up to 8 queries over up to ~10^5/(M + 2) keys take the one-launch scorer
    (each CTA rotates the queries, four threads per key): every bit width, MSE
    and Prod, key ranges with an offset, ragged key counts, more keys than one
    pass of its grid; and both sides of its limits."""
    d = 128
    mode = tq.TQ_PROD if prod else tq.TQ_MSE
    ctx, Pi, S = make_pair(31 + b, d, b, mode)
    total = first + N + 7
    X = synth.unit_rows(31, total, d) if prod else synth.gaussian_rows(31, total, d, outlier_cols=4,
                                                                       outlier_scale=20.0)
    cs = gpu_encode(ctx, X)
    Q = synth.queries(31, M, d)
    q = torch.from_numpy(np.ascontiguousarray(Q)).cuda()
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(tq.tq_scores_workspace_size(ctx, M) // 4 + 4, dtype=torch.float32, device="cuda")
    tq.tq_scores(ctx, q, cs, out, ws, first=first, N=N)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    b_mse = b - 1 if prod else b
    cb = oracle_codebook(d, b_mse)
    s = cs.norm[first:first + N].cpu().numpy().astype(np.float64)
    if prod:
        idx, bits = tq.tq_unpack_indices(cs, first, N, with_bits=True)
        gam = cs.rnorm[first:first + N].cpu().numpy().astype(np.float64)
        ref = oatt.prod_scores(Q.astype(np.float64), idx, s, bits, gam, Pi, S, cb["centroids"], math.sqrt(d))
    else:
        idx = tq.tq_unpack_indices(cs, first, N)
        ref = oatt.mse_scores(Q.astype(np.float64), idx, s, Pi, cb["centroids"], math.sqrt(d))
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    Xs = X[first:first + N].astype(np.float64)
    bound = 1e-4 * np.linalg.norm(Q, axis=1)[:, None] * np.linalg.norm(Xs, axis=1)[None, :]
    assert (np.abs(got - ref) <= bound).all(), f"max err/bound {np.max(np.abs(got - ref) / bound)}"


@pytest.mark.parametrize("prod", [False, True])
@pytest.mark.parametrize("M", [3, 70])
def test_scores_hadamard(prod, M):
    """Scores over keys encoded with the randomized Hadamard rotation, through
    the one-launch scorer (3 queries) and the tensor-core scorer (70)."""
    d, b = 128, 3
    ctx, Pi, S = make_pair(44, d, b, tq.TQ_PROD if prod else tq.TQ_MSE, rot="hadamard")
    X = synth.unit_rows(44, 999, d) if prod else synth.gaussian_rows(44, 999, d, outlier_cols=4, outlier_scale=20.0)
    Q = synth.queries(44, M, d)
    _scores_check(ctx, Pi, S, X, Q, b - 1 if prod else b, prod)


def test_scores_prod_config3_sample():
    ctx, Pi, S = make_pair(0, 128, 3, tq.TQ_PROD)
    X = synth.unit_rows(0, 8192, 128)
    Q = synth.queries(0, 64, 128)
    _scores_check(ctx, Pi, S, X, Q, 2, True)


# ------------------------------------------------------------------ decode
def run_decode(b_k, b_v, B, Hq, Hkv, seq, cap=None, seed=0, q_dtype=torch.float16, rot="dense"):
    d = 128
    cap = cap or (seq + 15) // 16 * 16
    kctx, Pi_k, _ = make_pair(seed, d, b_k, rot=rot)
    if b_v == b_k:
        vctx, Pi_v = kctx, Pi_k
    else:
        vctx, Pi_v, _ = make_pair(seed, d, b_v, rot=rot)
    Kh, Vh = synth.kv_layer(seed, 0, B, Hkv, seq, d)
    Kc = tq.CodeSet(kctx, B * Hkv * cap, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(vctx, B * Hkv * cap, tq.TQ_LAYOUT_PAIR)
    kx = torch.from_numpy(np.ascontiguousarray(Kh.reshape(-1, d))).cuda()
    vx = torch.from_numpy(np.ascontiguousarray(Vh.reshape(-1, d))).cuda()
    tq.tq_encode(kctx, kx, Kc, offset=0, group_rows=seq, group_stride=cap)
    tq.tq_encode(vctx, vx, Vc, offset=0, group_rows=seq, group_stride=cap)
    q_np = synth.queries(seed, B * Hq, d).reshape(B, Hq, d)
    q = torch.from_numpy(q_np).cuda().to(q_dtype)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(kctx, B, Hq, Hkv, seq) // 4 + 4, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    tq.tq_decode_attention(kctx, vctx, q, Kc, Vc, B, Hq, Hkv, seq, cap, scale, out, ws)
    torch.cuda.synchronize()
    assert kctx.poll() == tq.TQ_OK
    # oracle on the GPU's own codes
    kidx = np.concatenate([tq.tq_unpack_indices(Kc, blk * cap, seq) for blk in range(B * Hkv)])
    vidx = np.concatenate([tq.tq_unpack_indices(Vc, blk * cap, seq) for blk in range(B * Hkv)])
    kn = Kc.norm.cpu().numpy().reshape(B * Hkv, cap)[:, :seq].reshape(-1).astype(np.float64)
    vn = Vc.norm.cpu().numpy().reshape(B * Hkv, cap)[:, :seq].reshape(-1).astype(np.float64)
    cbk, cbv = oracle_codebook(d, b_k), oracle_codebook(d, b_v)
    Khat = oatt.dequantize_cache(kidx, kn, Pi_k, cbk["centroids"], math.sqrt(d), B, Hkv, seq)
    Vhat = oatt.dequantize_cache(vidx, vn, Pi_v, cbv["centroids"], math.sqrt(d), B, Hkv, seq)
    qref = q.float().cpu().numpy().astype(np.float64)
    ref = oatt.decode_attention(qref, Khat, Vhat, scale)
    got = out.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() <= 2e-3, f"max per-head relative error {rel.max()}"
    return rel.max()


@pytest.mark.parametrize("b", [2, 4])
def test_decode_config2(b):
    """One layer, B=1, 32 query / 8 KV heads, d=128, seq 16384, fp16 K/V with
    4 outlier channels x10, K and V TurboQuant_MSE at b."""
    run_decode(b, b, 1, 32, 8, 16384)


@pytest.mark.parametrize("seq", [1, 15, 17, 33, 1000])
def test_decode_ragged_seq(seq):
    run_decode(3, 3, 2, 8, 2, seq, cap=((seq + 15) // 16 + 1) * 16)


@pytest.mark.parametrize("gqa", [1, 2, 8])
def test_decode_gqa_variants(gqa):
    run_decode(3, 3, 1, 4 * gqa, 4, 777, q_dtype=torch.float32)


@pytest.mark.parametrize("b_k,b_v,B,Hq,Hkv,seq", [(3, 3, 1, 32, 4, 6007), (4, 4, 1, 64, 8, 5000),
                                                   (4, 2, 2, 16, 2, 9001)])
def test_decode_gqa8_long(b_k, b_v, B, Hq, Hkv, seq):
    """8 query heads per KV head over caches past 4096 tokens (the 8-head
    kernel, 8 warps per SM), table and byte-row lookups, asymmetric bits,
    ragged last tiles."""
    run_decode(b_k, b_v, B, Hq, Hkv, seq)


def test_decode_asymmetric_bits():
    run_decode(4, 2, 1, 16, 4, 2048)


@pytest.mark.parametrize("b_k,b_v,Hq,Hkv,seq", [(1, 1, 32, 8, 4099), (1, 3, 16, 4, 2001), (3, 1, 64, 8, 5003)])
def test_decode_one_bit(b_k, b_v, Hq, Hkv, seq):
    """1-bit keys and/or values (sign codes, centroids ±√(2/π)): GQA 4 and 8,
    asymmetric widths, ragged lengths."""
    run_decode(b_k, b_v, 1, Hq, Hkv, seq)


@pytest.mark.parametrize("b", [2, 3, 4])
def test_decode_hadamard_rotation(b):
    """Decode attention over K/V caches encoded with the randomized Hadamard
    rotation Π = H·diag(σ)/√d ("TurboQuant 和 RotorQuant 的真相", chapter 7,
    WHT vs random rotation): keys (TOKEN) and values (PAIR) by the d = 128
    tensor-memory encoder with the materialized Π; the oracle rotates with its
    own Hadamard matrix."""
    run_decode(b, b, 1, 32, 8, 3001, seed=5, rot="hadamard")


def test_decode_hadamard_gqa8_long():
    """8 query heads per KV head over a Hadamard-rotated cache longer than
    4096 tokens (the 8-head kernel)."""
    run_decode(3, 3, 1, 64, 8, 8191, seed=6, rot="hadamard")


def run_decode_prod(b_k, b_v, B, Hq, Hkv, seq, cap=None, seed=0, q_dtype=torch.float16, rot="dense"):
    """Decode attention with TurboQuant_Prod keys ((b_k - 1)-bit MSE codes plus
    QJL sign bits and γ) and TurboQuant_MSE values, against attention over the
    explicitly dequantized Prod keys x̂ = s·(Πᵀŷ + γ·√(π/2)/d·Sᵀ·sign) built
    from the GPU's own codes."""
    d = 128
    cap = cap or (seq + 15) // 16 * 16
    kctx, Pi_k, S = make_pair(seed, d, b_k, tq.TQ_PROD, rot=rot)
    vctx, Pi_v, _ = make_pair(seed + 100, d, b_v, rot=rot)
    Kh, Vh = synth.kv_layer(seed, 0, B, Hkv, seq, d)
    Kc = tq.CodeSet(kctx, B * Hkv * cap, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(vctx, B * Hkv * cap, tq.TQ_LAYOUT_PAIR)
    kx = torch.from_numpy(np.ascontiguousarray(Kh.reshape(-1, d))).cuda()
    vx = torch.from_numpy(np.ascontiguousarray(Vh.reshape(-1, d))).cuda()
    tq.tq_encode(kctx, kx, Kc, offset=0, group_rows=seq, group_stride=cap)
    tq.tq_encode(vctx, vx, Vc, offset=0, group_rows=seq, group_stride=cap)
    q_np = synth.queries(seed, B * Hq, d).reshape(B, Hq, d)
    q = torch.from_numpy(q_np).cuda().to(q_dtype)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(kctx, B, Hq, Hkv, seq) // 4 + 4, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    tq.tq_decode_attention(kctx, vctx, q, Kc, Vc, B, Hq, Hkv, seq, cap, scale, out, ws)
    torch.cuda.synchronize()
    assert kctx.poll() == tq.TQ_OK and vctx.poll() == tq.TQ_OK
    kidx, kbits = [], []
    for blk in range(B * Hkv):
        i, bt = tq.tq_unpack_indices(Kc, blk * cap, seq, with_bits=True)
        kidx.append(i)
        kbits.append(bt)
    kidx, kbits = np.concatenate(kidx), np.concatenate(kbits)
    vidx = np.concatenate([tq.tq_unpack_indices(Vc, blk * cap, seq) for blk in range(B * Hkv)])
    kn = Kc.norm.cpu().numpy().reshape(B * Hkv, cap)[:, :seq].reshape(-1).astype(np.float64)
    kg = Kc.rnorm.cpu().numpy()[:B * Hkv * cap].reshape(B * Hkv, cap)[:, :seq].reshape(-1).astype(np.float64)
    vn = Vc.norm.cpu().numpy().reshape(B * Hkv, cap)[:, :seq].reshape(-1).astype(np.float64)
    cbk, cbv = oracle_codebook(d, b_k - 1), oracle_codebook(d, b_v)
    Khat = oq.prod_dequantize(kidx, kn, kbits, kg, Pi_k, S, cbk["centroids"], math.sqrt(d)).reshape(B, Hkv, seq, d)
    Vhat = oatt.dequantize_cache(vidx, vn, Pi_v, cbv["centroids"], math.sqrt(d), B, Hkv, seq)
    qref = q.float().cpu().numpy().astype(np.float64)
    ref = oatt.decode_attention(qref, Khat, Vhat, scale)
    got = out.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() <= 2e-3, f"max per-head relative error {rel.max()}"
    # the QJL term matters: attention over the MSE part alone is measurably different
    Kmse = oq.mse_dequantize(kidx, kn, Pi_k, cbk["centroids"], math.sqrt(d)).reshape(B, Hkv, seq, d)
    alt = oatt.decode_attention(qref, Kmse, Vhat, scale)
    assert np.linalg.norm(alt - ref) > 10 * np.linalg.norm(got - ref)
    return rel.max()


@pytest.mark.parametrize("b_k,b_v,B,Hq,Hkv,seq", [
    (3, 3, 1, 32, 8, 4096),   # GQA 4, the config-2 head shape
    (4, 2, 2, 8, 4, 1000),    # ragged tail, two batches
    (2, 4, 1, 4, 4, 33),      # GQA 1, a few tiles
    (3, 2, 1, 16, 8, 777),    # GQA 2
])
def test_decode_prod_keys(b_k, b_v, B, Hq, Hkv, seq):
    run_decode_prod(b_k, b_v, B, Hq, Hkv, seq)


def test_decode_prod_keys_hadamard():
    """Prod keys and MSE values with randomized Hadamard rotations (the Prod
    stage's S·Πᵀ built from the materialized H·D/√d)."""
    run_decode_prod(3, 3, 1, 16, 4, 2001, seed=12, rot="hadamard")


def test_decode_prod_keys_rejected_where_unsupported():
    """Prod keys: no fused append (the step encodes MSE keys only) and at most
    4 query heads per KV head."""
    d, seq, cap = 128, 64, 64
    kctx, _, _ = make_pair(3, d, 3, tq.TQ_PROD)
    vctx, _, _ = make_pair(4, d, 3)
    Kc = tq.CodeSet(kctx, 8 * cap, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(vctx, 8 * cap, tq.TQ_LAYOUT_PAIR)
    ws = torch.zeros(tq.tq_decode_workspace_size(kctx, 1, 64, 8, seq) // 4 + 4, dtype=torch.float32, device="cuda")
    q = torch.zeros((1, 64, d), dtype=torch.float16, device="cuda")
    out = torch.empty((1, 64, d), dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TqError) as err:  # GQA 8
        tq.tq_decode_attention(kctx, vctx, q, Kc, Vc, 1, 64, 8, seq, cap, 1 / math.sqrt(d), out, ws)
    assert err.value.status == tq.TQ_ERR_UNSUPPORTED
    q4 = torch.zeros((1, 32, d), dtype=torch.float16, device="cuda")
    out4 = torch.empty((1, 32, d), dtype=torch.float32, device="cuda")
    kn = torch.zeros((8, d), dtype=torch.float16, device="cuda")
    with pytest.raises(tq.TqError) as err:  # fused append
        tq.tq_decode_step(kctx, vctx, q4, kn, kn, Kc, Vc, 1, 32, 8, seq, cap, 1 / math.sqrt(d), out4, ws)
    assert err.value.status == tq.TQ_ERR_UNSUPPORTED


# ------------------------------------------------------------------ full sizes
def test_prod_full_config3_sampled():
    """1M unit-norm keys, 64 queries, Prod b=3: encode and scores at full size,
    checked on a seeded sample of keys (the oracle evaluates them one by one)."""
    d, b, N, M = 128, 3, 1 << 20, 64
    ctx, Pi, S = make_pair(0, d, b, tq.TQ_PROD)
    X = synth.unit_rows(0, N, d)
    cs = gpu_encode(ctx, X)
    q = torch.from_numpy(synth.queries(0, M, d)).cuda()
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(tq.tq_scores_workspace_size(ctx, M) // 4 + 4, dtype=torch.float32, device="cuda")
    tq.tq_scores(ctx, q, cs, out, ws)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(1).choice(N, size=8192, replace=False))
    cb = oracle_codebook(d, b - 1)
    e = oq.prod_quantize(X[rows].astype(np.float64), Pi, S, cb["centroids"], math.sqrt(d))
    band = oq.near_threshold(e["v"], cb["centroids"])
    idx = np.zeros((len(rows), d), np.int64)
    bits = np.zeros((len(rows), d), np.int64)
    for k, r in enumerate(rows):
        i1, b1 = tq.tq_unpack_indices(cs, int(r), 1, with_bits=True)
        idx[k], bits[k] = i1[0], b1[0]
    assert not ((idx != e["idx"]) & ~band).any()
    ok = (idx == e["idx"]).all(axis=1)
    qband = oq.qjl_near_zero(e["p"], e["gamma"], S)
    assert not ((bits != e["bits"]) & ~qband & ok[:, None]).any()
    s = cs.norm.cpu().numpy()[rows].astype(np.float64)
    g = cs.rnorm.cpu().numpy()[rows].astype(np.float64)
    Q = synth.queries(0, M, d).astype(np.float64)
    ref = oatt.prod_scores(Q, idx, s, bits, g, Pi, S, cb["centroids"], math.sqrt(d))
    got = out.cpu().numpy()[:, rows].astype(np.float64)
    bound = 1e-4 * np.linalg.norm(Q, axis=1)[:, None] * np.linalg.norm(X[rows].astype(np.float64), axis=1)[None, :]
    assert (np.abs(got - ref) <= bound).all()


def test_decode_config4_layer_subset():
    """Long-context shape: 64 query / 8 KV heads, seq 131072, b=3 K/V.  The
    prefill encode of the layer (2 x 8 x 131072 fp16 vectors) is checked on a
    seeded sample of 4096 tokens of every KV head (codes outside the band and
    norms against the oracle's encoder); the oracle checks the attention of
    the query heads of two KV heads on the full sequence."""
    d, b, Hq, Hkv, seq = 128, 3, 64, 8, 131072
    cap = seq
    ctx, Pi, _ = make_pair(0, d, b)
    Kh, Vh = synth.kv_layer(0, 0, 1, Hkv, seq, d)
    Kc = tq.CodeSet(ctx, Hkv * cap, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(ctx, Hkv * cap, tq.TQ_LAYOUT_PAIR)
    tq.tq_encode(ctx, torch.from_numpy(Kh.reshape(-1, d)).cuda(), Kc, 0, seq, cap)
    tq.tq_encode(ctx, torch.from_numpy(Vh.reshape(-1, d)).cuda(), Vc, 0, seq, cap)
    q_np = synth.queries(0, Hq, d).reshape(1, Hq, d)
    q = torch.from_numpy(q_np).cuda().half()
    out = torch.empty((1, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(ctx, 1, Hq, Hkv, seq) // 4 + 4, dtype=torch.float32, device="cuda")
    tq.tq_decode_attention(ctx, ctx, q, Kc, Vc, 1, Hq, Hkv, seq, cap, 1 / math.sqrt(d), out, ws)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    cb = oracle_codebook(d, b)
    # prefill encode: sampled tokens of every KV head, K and V
    rng = np.random.default_rng(44)
    for arr, cs in ((Kh, Kc), (Vh, Vc)):
        for kvh in range(Hkv):
            toks = np.sort(rng.choice(seq, 4096, replace=False))
            X = arr[0, kvh, toks].astype(np.float64)
            ref, s_ref, v = oq.mse_quantize(X, Pi, cb["centroids"], math.sqrt(d))
            band = oq.near_threshold(v, cb["centroids"])
            allidx = tq.tq_unpack_indices(cs, kvh * cap, seq)
            got = allidx[toks].astype(np.int64)
            assert not ((got != ref) & ~band).any(), (kvh, int(((got != ref) & ~band).sum()))
            assert band_count_ok(band, cb["centroids"])
            nrm = cs.norm[kvh * cap: kvh * cap + seq].cpu().numpy()[toks].astype(np.float64)
            np.testing.assert_allclose(nrm, s_ref, rtol=1e-6)
    gqa = Hq // Hkv
    for kvh in (0, 5):
        ki = tq.tq_unpack_indices(Kc, kvh * cap, seq)
        vi = tq.tq_unpack_indices(Vc, kvh * cap, seq)
        kn = Kc.norm[kvh * cap: kvh * cap + seq].cpu().numpy().astype(np.float64)
        vn = Vc.norm[kvh * cap: kvh * cap + seq].cpu().numpy().astype(np.float64)
        Khat = oatt.dequantize_cache(ki, kn, Pi, cb["centroids"], math.sqrt(d), 1, 1, seq)
        Vhat = oatt.dequantize_cache(vi, vn, Pi, cb["centroids"], math.sqrt(d), 1, 1, seq)
        qq = q.float().cpu().numpy().astype(np.float64)[:, kvh * gqa:(kvh + 1) * gqa]
        ref = oatt.decode_attention(qq, Khat, Vhat, 1 / math.sqrt(d))
        got = out.cpu().numpy()[:, kvh * gqa:(kvh + 1) * gqa].astype(np.float64)
        rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
        assert rel.max() <= 2e-3, rel.max()


# ------------------------------------------------------------------ fused decode step (append + attend)
@pytest.mark.parametrize("b,B,Hq,Hkv,seq,rot", [(4, 1, 32, 8, 16384, "dense"), (2, 1, 32, 8, 16383, "dense"),
                                                 (3, 2, 16, 2, 1001, "dense"), (3, 1, 64, 8, 4096, "dense"),
                                                 (4, 1, 8, 8, 17, "dense"), (3, 1, 32, 8, 2047, "hadamard"),
                                                 (3, 1, 64, 8, 6001, "dense"),
                                                 (4, 1, 32, 8, 16384, "hadamard")])
def test_decode_step_appends_then_attends(b, B, Hq, Hkv, seq, rot):
    """The step encodes the new token's K and V into position seq-1 (same codes
    as the oracle's encoder, outside the near-threshold band) and attends over
    all seq tokens including it (dense Haar or randomized Hadamard rotation)."""
    d = 128
    cap = (seq + 15) // 16 * 16 + 16
    ctx, Pi, _ = make_pair(1, d, b, rot=rot)
    Kh, Vh = synth.kv_layer(1, 0, B, Hkv, seq, d)
    Kc = tq.CodeSet(ctx, B * Hkv * cap, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(ctx, B * Hkv * cap, tq.TQ_LAYOUT_PAIR)
    if seq > 1:
        tq.tq_encode(ctx, torch.from_numpy(np.ascontiguousarray(Kh[:, :, :seq - 1].reshape(-1, d))).cuda(),
                     Kc, 0, seq - 1, cap)
        tq.tq_encode(ctx, torch.from_numpy(np.ascontiguousarray(Vh[:, :, :seq - 1].reshape(-1, d))).cuda(),
                     Vc, 0, seq - 1, cap)
    kn = torch.from_numpy(np.ascontiguousarray(Kh[:, :, seq - 1])).cuda()
    vn = torch.from_numpy(np.ascontiguousarray(Vh[:, :, seq - 1])).cuda()
    q = torch.from_numpy(synth.queries(1, B * Hq, d).reshape(B, Hq, d)).cuda().half()
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(ctx, B, Hq, Hkv, seq) // 4 + 4, dtype=torch.float32, device="cuda")
    tq.tq_decode_step(ctx, ctx, q, kn, vn, Kc, Vc, B, Hq, Hkv, seq, cap, 1 / math.sqrt(d), out, ws)
    torch.cuda.synchronize()
    cb = oracle_codebook(d, b)
    # appended codes and norms
    for arr, cs in ((Kh, Kc), (Vh, Vc)):
        X = arr[:, :, seq - 1].reshape(-1, d).astype(np.float64)
        ref, s_ref, v = oq.mse_quantize(X, Pi, cb["centroids"], math.sqrt(d))
        band = oq.near_threshold(v, cb["centroids"])
        got = np.stack([tq.tq_unpack_indices(cs, blk * cap + seq - 1, 1)[0] for blk in range(B * Hkv)])
        assert not ((got.astype(np.int64) != ref) & ~band).any()
        norms = cs.norm.cpu().numpy().reshape(B * Hkv, cap)[:, seq - 1].astype(np.float64)
        np.testing.assert_allclose(norms, s_ref, rtol=1e-6)
    # attention over all tokens, oracle on the GPU's codes
    kidx = np.concatenate([tq.tq_unpack_indices(Kc, blk * cap, seq) for blk in range(B * Hkv)])
    vidx = np.concatenate([tq.tq_unpack_indices(Vc, blk * cap, seq) for blk in range(B * Hkv)])
    knr = Kc.norm.cpu().numpy().reshape(B * Hkv, cap)[:, :seq].reshape(-1).astype(np.float64)
    vnr = Vc.norm.cpu().numpy().reshape(B * Hkv, cap)[:, :seq].reshape(-1).astype(np.float64)
    Khat = oatt.dequantize_cache(kidx, knr, Pi, cb["centroids"], math.sqrt(d), B, Hkv, seq)
    Vhat = oatt.dequantize_cache(vidx, vnr, Pi, cb["centroids"], math.sqrt(d), B, Hkv, seq)
    ref = oatt.decode_attention(q.float().cpu().numpy().astype(np.float64), Khat, Vhat, 1 / math.sqrt(d))
    got = out.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() <= 2e-3, rel.max()
