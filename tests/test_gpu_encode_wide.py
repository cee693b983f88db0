"""GPU parity of the encoders for the bulk-indexing workload (b = 4, d = 1536
and 3072, fp32 rows N(0, 1) with a seeded 1 % of the rows scaled by 50) and of
the randomized-Hadamard fast transform at every supported order, against the
fp64 oracle.  Same bars as the other encode parity tests: indices exact
outside the 1e-6 band around the thresholds (band fraction <= 1e-5), norms
within 1e-6 relative.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import kv_cache_vector_tq_gb300 as tq  # noqa: E402
from kv_cache_vector_tq_gb300 import synth  # noqa: E402
from oracle import codebook as ocb  # noqa: E402
from oracle import quantizer as oq  # noqa: E402
from oracle import rotation as orot  # noqa: E402

pytestmark = pytest.mark.gpu

BAND_FRAC_MAX = 1e-5
_cb = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()


def codebook(d, b):
    if (d, b) not in _cb:
        _cb[(d, b)] = ocb.build_codebook(d, b)
    return _cb[(d, b)]


def hadamard_pair(seed, d, b):
    sg = synth.hadamard_signs(seed, d)
    return tq.Context(d, b, tq.TQ_MSE, tq.TQ_ROT_HADAMARD, sg), orot.hadamard_rotation(d, sg)


def encode(ctx, X, dtype=torch.float32):
    x = torch.from_numpy(np.ascontiguousarray(X)).to(dtype).cuda()
    cs = tq.CodeSet(ctx, X.shape[0], tq.TQ_LAYOUT_TOKEN)
    tq.tq_encode(ctx, x, cs)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    return cs


def check(cs, Pi, X, b, rows=None):
    """Oracle on the (sampled) rows; rows = None means all."""
    rows = np.arange(X.shape[0]) if rows is None else np.asarray(rows)
    return check_rows(cs, Pi, X[rows], rows, b, all_rows=len(rows) == X.shape[0])


def check_rows(cs, Pi, Xs, rows, b, all_rows=False):
    """Oracle on the rows Xs, which the code set holds at indices `rows`."""
    d = Xs.shape[1]
    Xs = Xs.astype(np.float64)
    cb = codebook(d, b)
    idx_ref, s_ref, v = oq.mse_quantize(Xs, Pi, cb["centroids"], math.sqrt(d))
    band = oq.near_threshold(v, cb["centroids"])
    band[s_ref == 0.0] = False
    idx = tq.tq_unpack_indices(cs, 0, len(rows)) if all_rows \
        else np.stack([tq.tq_unpack_indices(cs, int(r), 1)[0] for r in rows])
    mism = (idx.astype(np.int64) != idx_ref) & ~band
    assert not mism.any(), f"{mism.sum()} mismatches outside the band (rows {rows[np.nonzero(mism.any(1))[0][:8]]})"
    # the band is a rare event: on small samples allow a Poisson fluctuation
    # above the 1e-5 cap (mean + 4 sigma + 2)
    lam = BAND_FRAC_MAX * band.size
    assert band.mean() <= BAND_FRAC_MAX or band.sum() <= lam + 4 * math.sqrt(lam) + 2, band.mean()
    norm = cs.norm.cpu().numpy().astype(np.float64)[rows]
    np.testing.assert_allclose(norm, s_ref, rtol=1e-6, atol=0)
    return idx_ref, band


@pytest.mark.parametrize("d", [32, 64, 128, 256, 384, 768, 1536, 3072])
@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_hadamard_fast_transform(d, b):
    """Orders 2^k and 12·2^k with 32 <= 2^k <= 256 run the fast transform
    (d = 128: the tensor-memory encoder with the materialized H·D/√d)."""
    n = 257 if d <= 384 else 96
    ctx, Pi = hadamard_pair(7, d, b)
    X = synth.bulk_rows(7, n, d)
    X[n // 3] = 0.0  # zero vector: s = 0, codes 0
    cs = encode(ctx, X)
    idx_ref, band = check(cs, Pi, X, b)
    # raw words equal the canonical packing wherever no coordinate is in the band
    words = cs.codes.view(torch.int32).cpu().numpy().view(np.uint32).reshape(n, -1)
    ok = ~band.any(axis=1)
    np.testing.assert_array_equal(words[ok], oq.pack_codes(idx_ref[ok], b))


def test_hadamard_fast_transform_fp16_rows():
    ctx, Pi = hadamard_pair(8, 128, 3)
    X = synth.gaussian_rows(8, 500, 128, outlier_cols=4, outlier_scale=10.0, dtype=np.float16)
    cs = encode(ctx, X, torch.float16)
    check(cs, Pi, X.astype(np.float32), 3)


@pytest.mark.parametrize("b", [2, 3, 4])
@pytest.mark.parametrize("f16", [False, True])
def test_hadamard_d128_pair_layout(b, f16):
    """d = 128 Hadamard contexts into PAIR caches (the tensor-memory encoder's
    slot-placed kernel with H·D/√d as its matrix), an odd row count."""
    ctx, Pi = hadamard_pair(9, 128, b)
    X = synth.gaussian_rows(9, 333, 128, outlier_cols=4, outlier_scale=10.0)
    if f16:
        X = X.astype(np.float16)
    cs = tq.CodeSet(ctx, X.shape[0], tq.TQ_LAYOUT_PAIR)
    tq.tq_encode(ctx, torch.from_numpy(np.ascontiguousarray(X)).cuda(), cs)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    check(cs, Pi, X.astype(np.float32), b)


@pytest.mark.parametrize("d", [256, 3072])
def test_hadamard_extreme_magnitudes(d):
    """Rows scaled by 1e-20, 1e-25 and 1e22 and rows with a single non-zero
    value, through the fast transform (one block, and twelve)."""
    ctx, Pi = hadamard_pair(16, d, 4)
    X = synth.bulk_rows(16, 40, d)
    X[1] *= 1e-20
    X[2] *= 1e-25
    X[3] *= 1e22
    X[4] = 0.0
    X[4, d // 3] = 2.5e-30
    X[5] = 0.0
    X[5, 0] = -3e30
    cs = encode(ctx, X)
    check(cs, Pi, X, 4)


@pytest.mark.parametrize("d", [1536, 3072])
def test_hadamard_bulk_indexing_full_size_sampled(d):
    """N = 100K rows of the bulk-indexing workload, 512 rows checked."""
    N = 100_000
    ctx, Pi = hadamard_pair(0, d, 4)
    X = synth.bulk_rows(0, N, d)
    cs = encode(ctx, X)
    rows = np.random.default_rng(1).choice(N, size=512, replace=False)
    check(cs, Pi, X, 4, rows)


_haar = {}


def haar_pair(seed, d, b):
    if (seed, d) not in _haar:
        G = synth.gaussian_matrix(seed, d)
        _haar[(seed, d)] = (tq.tq_rotation_haar(G), orot.haar_rotation(G))
    pi_lib, pi_ref = _haar[(seed, d)]
    return tq.Context(d, b, tq.TQ_MSE, tq.TQ_ROT_DENSE, pi_lib), pi_ref


@pytest.mark.parametrize("d", [256, 384, 1536, 3072])
@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_dense_wide_encode(d, b):
    """Dense Haar rotation for d > 128 (tcgen05 GEMM over 128-row tiles plus
    the exact recomputation of near-threshold coordinates): a ragged row
    count (three tiles, the last one partial), a zero row and a row scaled by
    1e4."""
    n = 300
    ctx, Pi = haar_pair(11, d, b)
    X = synth.bulk_rows(11, n, d)
    X[7] = 0.0
    X[150] *= 1e4
    cs = encode(ctx, X)
    idx_ref, band = check(cs, Pi, X, b)
    words = cs.codes.view(torch.int32).cpu().numpy().view(np.uint32).reshape(n, -1)
    ok = ~band.any(axis=1)
    np.testing.assert_array_equal(words[ok], oq.pack_codes(idx_ref[ok], b))


@pytest.mark.parametrize("d", [256, 1536])
def test_dense_wide_encode_magnitude_edges(d):
    """Rows whose magnitudes vary along the row or are extreme: zero leading
    chunks, a small first chunk, a single huge or single non-zero value, rows
    scaled by 1e-20, 1e-25 and 1e22 (squares below the fp32 normal range,
    below its range, above it)."""
    b = 4
    X = synth.bulk_rows(15, 140, d)
    X[3, :64] = 0.0          # first chunk zero
    X[4, :128] = 0.0         # first two chunks zero
    X[5, :64] *= 1e-2        # small first chunk, later values ~100x larger
    X[6, :64] *= 1e-6        # later values ~1e6x larger
    X[7, 64:] = 0.0          # only the first chunk non-zero
    X[8] *= 1e-20            # a tiny row
    X[9, :64] *= 1e-35       # a first chunk far below the rest
    X[10, -1] = 1e6          # one huge last value
    X[11] = 0.0
    X[11, d - 1] = -3.0      # a single non-zero value, in the last chunk
    X[12] *= 1e-25           # squares below the fp32 range
    X[13] *= 1e22            # squares above the fp32 range
    ctx, Pi = haar_pair(15, d, b)
    cs = encode(ctx, X)
    check(cs, Pi, X, b)


def test_dense_wide_encode_fp16_rows():
    ctx, Pi = haar_pair(12, 1536, 4)
    X = synth.gaussian_rows(12, 200, 1536, outlier_cols=4, outlier_scale=10.0, dtype=np.float16)
    cs = encode(ctx, X, torch.float16)
    check(cs, Pi, X.astype(np.float32), 4)


@pytest.mark.parametrize("d", [1536, 3072])
def test_dense_bulk_indexing_full_size_sampled(d):
    """N = 100K rows of the bulk-indexing workload with the dense Haar
    rotation, 512 rows checked."""
    N = 100_000
    ctx, Pi = haar_pair(0, d, 4)
    X = synth.bulk_rows(0, N, d)
    cs = encode(ctx, X)
    rows = np.random.default_rng(2).choice(N, size=512, replace=False)
    check(cs, Pi, X, 4, rows)


@pytest.mark.parametrize("d,b", [(256, 4), (384, 1), (384, 3)])
def test_dense_wide_encode_grouped_destination(d, b):
    """Rows scattered into a larger code set (group_rows / group_stride /
    offset), as when appending to (batch, head) blocks of a cache; tiles of
    128 (d = 256) and 192 (d = 384) output coordinates."""
    n = 200
    ctx, Pi = haar_pair(14, d, b)
    X = synth.bulk_rows(14, n, d)
    x = torch.from_numpy(X).cuda()
    cs = tq.CodeSet(ctx, 1000, tq.TQ_LAYOUT_TOKEN)
    tq.tq_encode(ctx, x, cs, offset=3, group_rows=50, group_stride=240)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    dst = np.array([(r // 50) * 240 + 3 + r % 50 for r in range(n)])
    cb = codebook(d, b)
    idx_ref, s_ref, v = oq.mse_quantize(X.astype(np.float64), Pi, cb["centroids"], math.sqrt(d))
    band = oq.near_threshold(v, cb["centroids"])
    idx = np.stack([tq.tq_unpack_indices(cs, int(r), 1)[0] for r in dst])
    assert not ((idx.astype(np.int64) != idx_ref) & ~band).any()
    np.testing.assert_allclose(cs.norm.cpu().numpy().astype(np.float64)[dst], s_ref, rtol=1e-6, atol=0)


def test_wide_encode_rejects_unsupported():
    """d > 128 with the dense rotation: MSE and TOKEN layout only."""
    ctx, _ = haar_pair(13, 256, 3)
    x = torch.zeros((4, 256), dtype=torch.float32, device="cuda")
    cs = tq.CodeSet(ctx, 4, tq.TQ_LAYOUT_PAIR)
    with pytest.raises(tq.TqError) as err:
        tq.tq_encode(ctx, x, cs)
    assert err.value.status == tq.TQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("rot", ["dense", "hadamard"])
def test_bulk_indexing_ten_million_rows_sampled(rot):
    """N = 10M rows of the bulk-indexing workload at d = 3072 (123 GB of fp32
    rows, generated on the device by torch's seeded generator with the
    workload's distribution: N(0, 1), a seeded 1 % of the rows x50), encoded in
    one call; 256 random rows plus the first and last are copied back and
    checked against the oracle."""
    d, N = 3072, 10_000_000
    if torch.cuda.mem_get_info()[0] < 150e9:
        pytest.skip("needs 150 GB of free device memory")
    ctx, Pi = haar_pair(0, d, 4) if rot == "dense" else hadamard_pair(0, d, 4)
    gen = torch.Generator(device="cuda").manual_seed(20)
    x = torch.randn((N, d), generator=gen, device="cuda")
    x[torch.randperm(N, generator=gen, device="cuda")[: N // 100]] *= 50.0
    cs = tq.CodeSet(ctx, N, tq.TQ_LAYOUT_TOKEN)
    tq.tq_encode(ctx, x, cs)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    rows = np.concatenate([[0, N - 1], np.random.default_rng(3).choice(N, size=256, replace=False)])
    Xs = x[torch.from_numpy(rows).cuda()].cpu().numpy()
    del x
    torch.cuda.empty_cache()
    check_rows(cs, Pi, Xs, rows, 4)
    del cs
    torch.cuda.empty_cache()
