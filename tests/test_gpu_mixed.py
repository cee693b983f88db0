"""GPU parity at b + 1/2 bits per coordinate (TQ_MIXED) through the C ABI,
against the fp64 oracle.

The reading ("TurboQuant 详解", sections "论文给出的关键数据点" and "decode 阶段：
写入少，但每步都要读取历史 cache"): one rotation and one norm per vector, the
rotated coordinates j with j mod 16 < 8 quantized with the (b+1)-bit Lloyd-Max
codebook and the others with the b-bit one, codes packed canonically with a
width per coordinate.  Bars as for the other modes: indices and raw words
bit-exact outside the 1e-6 near-threshold band of each coordinate's own
codebook, norms within 1e-6 relative, scores within 1e-4·‖q‖‖x‖, attention
outputs within 2e-3·‖out‖ per head.
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
D = 128

_cb = {}


def codebooks(b):
    if b not in _cb:
        _cb[b] = (ocb.build_codebook(D, b)["centroids"], ocb.build_codebook(D, b + 1)["centroids"])
    return _cb[b]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()


def mixed_pair(seed, b):
    G = synth.gaussian_matrix(seed, D)
    return tq.Context(D, b, tq.TQ_MIXED, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(G)), orot.haar_rotation(G)


def oracle_codes(X, Pi, b):
    lo, hi = codebooks(b)
    idx, s, v = oq.mixed_quantize(np.asarray(X, dtype=np.float64), Pi, lo, hi, b, math.sqrt(D))
    band = oq.mixed_near_threshold(v, lo, hi, b)
    band[s == 0.0] = False
    return idx, s, band


@pytest.mark.parametrize("b", [1, 3])
def test_mixed_encode_hadamard(b):
    """b + 1/2 bits with the randomized Hadamard rotation (d = 128: the
    tensor-memory encoder with H·D/√d), fp16 rows, both layouts."""
    sg = synth.hadamard_signs(5, D)
    ctx = tq.Context(D, b, tq.TQ_MIXED, tq.TQ_ROT_HADAMARD, sg)
    Pi = orot.hadamard_rotation(D, sg)
    K, V = synth.kv_layer(5, 0, 1, 2, 500, D)
    for arr, layout in ((K, tq.TQ_LAYOUT_TOKEN), (V, tq.TQ_LAYOUT_PAIR)):
        X = arr.reshape(-1, D)
        cs = tq.CodeSet(ctx, X.shape[0], layout)
        tq.tq_encode(ctx, torch.from_numpy(np.ascontiguousarray(X)).cuda(), cs)
        torch.cuda.synchronize()
        assert ctx.poll() == tq.TQ_OK
        idx, s, band = oracle_codes(X.astype(np.float32), Pi, b)
        got = tq.tq_unpack_indices(cs).astype(np.int64)
        assert not ((got != idx) & ~band).any()
        np.testing.assert_allclose(cs.norm[:X.shape[0]].cpu().numpy().astype(np.float64), s, rtol=1e-6, atol=0)
    # scores over the TOKEN keys against the oracle's dequantization
    Q = synth.queries(5, 3, D)
    out = torch.empty((3, X.shape[0]), dtype=torch.float32, device="cuda")
    Kc = tq.CodeSet(ctx, X.shape[0], tq.TQ_LAYOUT_TOKEN)
    Kx = K.reshape(-1, D)
    tq.tq_encode(ctx, torch.from_numpy(np.ascontiguousarray(Kx)).cuda(), Kc)
    ws = torch.empty(tq.tq_scores_workspace_size(ctx, 3) // 4 + 4, dtype=torch.float32, device="cuda")
    tq.tq_scores(ctx, torch.from_numpy(np.ascontiguousarray(Q)).cuda(), Kc, out, ws)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    lo, hi = codebooks(b)
    idx = tq.tq_unpack_indices(Kc).astype(np.int64)
    Xh = oq.mixed_dequantize(idx, Kc.norm[:Kx.shape[0]].cpu().numpy().astype(np.float64), Pi, lo, hi, b, math.sqrt(D))
    ref = Q.astype(np.float64) @ Xh.T
    bound = 1e-4 * np.linalg.norm(Q, axis=1)[:, None] * np.linalg.norm(Kx.astype(np.float64), axis=1)[None, :]
    assert (np.abs(out.cpu().numpy().astype(np.float64) - ref) <= bound).all()


def words_of(cs, n_words):
    return cs.codes.view(torch.int32).cpu().numpy().view(np.uint32)[:n_words]


def test_mixed_layout_sizes():
    for b, nbytes in ((1, 24), (2, 40), (3, 56)):
        ctx, _ = mixed_pair(0, b)
        cs = tq.CodeSet(ctx, 10, tq.TQ_LAYOUT_TOKEN)
        assert cs.words_per_vec * 4 == nbytes == oq.mixed_words_per_vector(D, b) * 4


@pytest.mark.parametrize("b", [1, 2, 3])
@pytest.mark.parametrize("f16", [False, True])
def test_mixed_encode_token_and_pair_words(b, f16):
    """K/V-like rows (fp16 N(0,1), channels 0-3 x10), 2 heads x 1000 tokens;
    fp32 rows are the same values widened.  TOKEN words against the oracle's
    variable-width packing, PAIR blocks against its pair interleave."""
    ctx, Pi = mixed_pair(3, b)
    K, V = synth.kv_layer(3, 0, 1, 2, 1000, D)
    for arr, layout in ((K, tq.TQ_LAYOUT_TOKEN), (V, tq.TQ_LAYOUT_PAIR)):
        X = arr.reshape(-1, D)
        Xin = X if f16 else X.astype(np.float32)
        cs = tq.CodeSet(ctx, X.shape[0], layout)
        tq.tq_encode(ctx, torch.from_numpy(np.ascontiguousarray(Xin)).cuda(), cs)
        torch.cuda.synchronize()
        assert ctx.poll() == tq.TQ_OK
        idx, s, band = oracle_codes(X.astype(np.float32), Pi, b)
        got = tq.tq_unpack_indices(cs).astype(np.int64)
        assert not ((got != idx) & ~band).any()
        assert band.mean() <= 1e-5 or band.sum() <= 3
        np.testing.assert_allclose(cs.norm[:X.shape[0]].cpu().numpy().astype(np.float64), s, rtol=1e-6, atol=0)
        W = cs.words_per_vec
        words = words_of(cs, X.shape[0] * W)
        if layout == tq.TQ_LAYOUT_TOKEN:
            ok = ~band.any(1)
            ref = oq.pack_varwidth(idx, oq.mixed_widths(D, b))
            np.testing.assert_array_equal(words.reshape(-1, W)[ok], ref[ok])
        else:
            ok = ~(band[0::2].any(1) | band[1::2].any(1))
            ref = oq.pack_mixed_pairs(idx, b)
            np.testing.assert_array_equal(words.reshape(-1, 2 * W)[ok], ref[ok])


@pytest.mark.parametrize("N", [1, 127, 129, 1000])
def test_mixed_encode_ragged_and_zero_rows(N):
    b = 2
    ctx, Pi = mixed_pair(4, b)
    X = synth.gaussian_rows(4, N, D).astype(np.float32)
    X[::7] = 0.0
    cs = tq.CodeSet(ctx, N, tq.TQ_LAYOUT_TOKEN)
    tq.tq_encode(ctx, torch.from_numpy(X).cuda(), cs)
    torch.cuda.synchronize()
    idx, s, band = oracle_codes(X, Pi, b)
    got = tq.tq_unpack_indices(cs).astype(np.int64)
    assert not ((got != idx) & ~band).any()
    assert not got[::7].any()
    np.testing.assert_allclose(cs.norm[:N].cpu().numpy().astype(np.float64), s, rtol=1e-6, atol=0)


def test_mixed_encode_append_into_pair_blocks():
    """Cache append at b + 1/2 bits: one token per (batch, head) block at
    positions 37, 38, 39, next to 37 tokens encoded earlier (the half-written
    pair goes through the masked-atomic path)."""
    b, cap, blocks = 3, 64, 6
    ctx, Pi = mixed_pair(5, b)
    X = synth.gaussian_rows(5, blocks * 40, D).reshape(blocks, 40, D).astype(np.float32)
    cs = tq.CodeSet(ctx, blocks * cap, tq.TQ_LAYOUT_PAIR)
    pre = torch.from_numpy(np.ascontiguousarray(X[:, :37].reshape(-1, D))).cuda()
    tq.tq_encode(ctx, pre, cs, offset=0, group_rows=37, group_stride=cap)
    for t in (37, 38, 39):
        tq.tq_encode(ctx, torch.from_numpy(np.ascontiguousarray(X[:, t])).cuda(), cs, offset=t, group_rows=1,
                     group_stride=cap)
    torch.cuda.synchronize()
    idx, s, band = oracle_codes(X.reshape(-1, D), Pi, b)
    W = cs.words_per_vec
    words = words_of(cs, blocks * cap * W).reshape(blocks, cap // 2, 2 * W)
    for blk in range(blocks):
        got = tq.tq_unpack_indices(cs, blk * cap, 40).astype(np.int64)
        ref = idx[blk * 40:(blk + 1) * 40]
        bb = band[blk * 40:(blk + 1) * 40]
        assert not ((got != ref) & ~bb).any()
        ok = ~(bb[0::2].any(1) | bb[1::2].any(1))
        np.testing.assert_array_equal(words[blk, :20][ok], oq.pack_mixed_pairs(ref, b)[ok])
        assert not words[blk, 20:].any()  # nothing beyond position 39


@pytest.mark.parametrize("b,N,M", [(1, 1237, 70), (2, 4096, 64), (3, 129, 3), (2, 1, 1)])
def test_mixed_scores(b, N, M):
    """Inner products over b + 1/2-bit keys (rows with 4 outlier channels x20),
    against the oracle's ⟨q, x̂⟩ on the GPU's own codes: ragged key tiles, more
    than one 64-query launch, one key and one query."""
    ctx, Pi = mixed_pair(7, b)
    X = synth.gaussian_rows(7, N, D, outlier_cols=4, outlier_scale=20.0).astype(np.float32)
    Q = synth.queries(7, M, D)
    cs = tq.CodeSet(ctx, N, tq.TQ_LAYOUT_TOKEN)
    tq.tq_encode(ctx, torch.from_numpy(X).cuda(), cs)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(tq.tq_scores_workspace_size(ctx, M) // 4 + 4, dtype=torch.float32, device="cuda")
    tq.tq_scores(ctx, torch.from_numpy(np.ascontiguousarray(Q)).cuda(), cs, out, ws)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    lo, hi = codebooks(b)
    idx = tq.tq_unpack_indices(cs).astype(np.int64)
    Xh = oq.mixed_dequantize(idx, cs.norm[:N].cpu().numpy().astype(np.float64), Pi, lo, hi, b, math.sqrt(D))
    ref = Q.astype(np.float64) @ Xh.T
    got = out.cpu().numpy().astype(np.float64)
    bound = 1e-4 * np.linalg.norm(Q, axis=1)[:, None] * np.linalg.norm(X.astype(np.float64), axis=1)[None, :]
    assert (np.abs(got - ref) <= bound).all(), f"max err/bound {np.max(np.abs(got - ref) / bound)}"


def hadamard_mixed_pair(seed, b):
    sg = synth.hadamard_signs(seed, D)
    return tq.Context(D, b, tq.TQ_MIXED, tq.TQ_ROT_HADAMARD, sg), orot.hadamard_rotation(D, sg)


def run_decode_mixed(b, B, Hq, Hkv, seq, cap=None, seed=0, q_dtype=torch.float16, hadamard=False):
    """Decode attention over b + 1/2-bit K (TOKEN) and V (PAIR) caches, each with
    its own Haar (or randomized Hadamard) rotation, against fp64 attention over
    the oracle's dequantization of the GPU's own codes (2e-3·‖out‖ per head)."""
    cap = cap or (seq + 15) // 16 * 16
    make = hadamard_mixed_pair if hadamard else mixed_pair
    kctx, Pk = make(seed, b)
    vctx, Pv = make(seed + 1000, b)
    Kh, Vh = synth.kv_layer(seed, 0, B, Hkv, seq, D)
    Kc = tq.CodeSet(kctx, B * Hkv * cap, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(vctx, B * Hkv * cap, tq.TQ_LAYOUT_PAIR)
    tq.tq_encode(kctx, torch.from_numpy(np.ascontiguousarray(Kh.reshape(-1, D))).cuda(), Kc, offset=0,
                 group_rows=seq, group_stride=cap)
    tq.tq_encode(vctx, torch.from_numpy(np.ascontiguousarray(Vh.reshape(-1, D))).cuda(), Vc, offset=0,
                 group_rows=seq, group_stride=cap)
    q_np = synth.queries(seed, B * Hq, D).reshape(B, Hq, D)
    q = torch.from_numpy(q_np).cuda().to(q_dtype)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(kctx, B, Hq, Hkv, seq) // 4 + 4, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    tq.tq_decode_attention(kctx, vctx, q, Kc, Vc, B, Hq, Hkv, seq, cap, scale, out, ws)
    torch.cuda.synchronize()
    assert kctx.poll() == tq.TQ_OK and vctx.poll() == tq.TQ_OK
    lo, hi = codebooks(b)

    def rebuild(cs, Pi):
        idx = np.concatenate([tq.tq_unpack_indices(cs, blk * cap, seq) for blk in range(B * Hkv)]).astype(np.int64)
        nrm = cs.norm.cpu().numpy().reshape(B * Hkv, cap)[:, :seq].reshape(-1).astype(np.float64)
        return oq.mixed_dequantize(idx, nrm, Pi, lo, hi, b, math.sqrt(D)).reshape(B, Hkv, seq, D)

    from oracle import attention as oatt
    ref = oatt.decode_attention(q.float().cpu().numpy().astype(np.float64), rebuild(Kc, Pk), rebuild(Vc, Pv), scale)
    got = out.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() <= 2e-3, f"max per-head relative error {rel.max()}"
    return rel.max()


@pytest.mark.parametrize("b", [2, 3])
def test_mixed_decode_hadamard(b):
    """b + 1/2-bit caches with randomized Hadamard rotations: GQA 4, a ragged
    sequence."""
    run_decode_mixed(b, 1, 16, 4, 3001, seed=8, hadamard=True)


@pytest.mark.parametrize("b", [1, 2, 3])
def test_mixed_decode_one_layer(b):
    """One layer, B = 1, 32 query / 8 KV heads, seq 16384: the decode workload at
    1.5, 2.5 and 3.5 bits per coordinate."""
    run_decode_mixed(b, 1, 32, 8, 16384)


@pytest.mark.parametrize("seq", [1, 15, 17, 33, 1000])
def test_mixed_decode_ragged_seq(seq):
    run_decode_mixed(2, 2, 8, 2, seq, cap=((seq + 15) // 16 + 1) * 16)


@pytest.mark.parametrize("gqa", [1, 2, 4, 8])
def test_mixed_decode_gqa(gqa):
    run_decode_mixed(3, 1, 4 * gqa, 4, 777, q_dtype=torch.float32)


def test_mixed_decode_refusals():
    """b + 1/2-bit caches decode in the attention entry with K and V at the same
    b; the fused append and mixed/uniform pairs are refused."""
    kctx, _ = mixed_pair(0, 2)
    vctx, _ = mixed_pair(1, 3)
    uctx = tq.Context(D, 2, tq.TQ_MSE, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(synth.gaussian_matrix(2, D)))
    cap, seq = 32, 20
    Kc = tq.CodeSet(kctx, 4 * cap, tq.TQ_LAYOUT_TOKEN)
    q = torch.zeros((1, 8, D), dtype=torch.float16, device="cuda")
    out = torch.empty((1, 8, D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(kctx, 1, 8, 4, seq) // 4 + 4, dtype=torch.float32, device="cuda")
    for vc in (vctx, uctx):
        Vc = tq.CodeSet(vc, 4 * cap, tq.TQ_LAYOUT_PAIR)
        with pytest.raises(tq.TqError) as e:
            tq.tq_decode_attention(kctx, vc, q, Kc, Vc, 1, 8, 4, seq, cap, 0.1, out, ws)
        assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    Vc = tq.CodeSet(kctx, 4 * cap, tq.TQ_LAYOUT_PAIR)
    new = torch.zeros((4, D), dtype=torch.float16, device="cuda")
    with pytest.raises(tq.TqError) as e:
        tq.tq_decode_step(kctx, kctx, q, new, new, Kc, Vc, 1, 8, 4, seq, cap, 0.1, out, ws)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
