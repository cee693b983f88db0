"""Reconstruction quality with asymmetric K/V bit widths, on synthetic KV rows.

"sub-byte-kv-cache-quantization-turboquant", section 生产级精度 - 吞吐权衡参数,
reports on model KV caches an inner-product correlation of 0.995 and a cosine
similarity of 0.995 at 4 bits, and 0.945 / 0.940 at 2 bits; "TurboQuant 和
RotorQuant 的真相", chapter 7, recommends more bits for K than for V.  Those
model caches are not here; these tests measure the same two quantities on the
seeded stand-in (fp16 N(0,1) rows with 4 outlier channels x10) through the
product path, and check them against what the MSE quantizer fixes in closed
form: a reconstruction x̂ = E[x | code] has an error orthogonal to it on
average, so both the cosine ⟨x, x̂⟩/(‖x‖‖x̂‖) and the correlation of ⟨q, x̂⟩
with ⟨q, x⟩ are √(1 − D_b), D_b the codebook distortion (0.995 at b = 4,
0.940 at b = 2).

  * cosine of K and V reconstructions: the GPU's codes and norms, rebuilt by
    the oracle (x̂ = s·Πᵀŷ);
  * inner-product correlation: tq_scores over the GPU's key codes against the
    exact ⟨q, x⟩ of the fp16 rows;
  * attention output cosine: tq_decode_attention over (K bits, V bits) caches
    against fp64 attention over the unquantized rows (reported; the softmax
    amplifies key error on these outlier-heavy rows, so it orders by key bits).
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

D, HQ, HKV, T = 128, 32, 8, 2048


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()


def _ctx(seed, b):
    G = synth.gaussian_matrix(seed, D)
    return tq.Context(D, b, tq.TQ_MSE, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(G)), orot.haar_rotation(G)


def _cos_rows(X, Xh):
    return np.sum(X * Xh, axis=1) / (np.linalg.norm(X, axis=1) * np.linalg.norm(Xh, axis=1))


def _measure(bk, bv):
    Kh, Vh = synth.kv_layer(21, 0, 1, HKV, T, D)
    cap = T
    kctx, Pk = _ctx(21, bk)
    vctx, Pv = (kctx, Pk) if bv == bk else _ctx(22, bv)
    Kc = tq.CodeSet(kctx, HKV * cap, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(vctx, HKV * cap, tq.TQ_LAYOUT_PAIR)
    tq.tq_encode(kctx, torch.from_numpy(Kh.reshape(-1, D)).cuda(), Kc, 0, T, cap)
    tq.tq_encode(vctx, torch.from_numpy(Vh.reshape(-1, D)).cuda(), Vc, 0, T, cap)
    cbk, cbv = ocb.build_codebook(D, bk), ocb.build_codebook(D, bv)
    # reconstruction cosine, K and V (all 8 x 2048 rows)
    K = Kh.reshape(-1, D).astype(np.float64)
    V = Vh.reshape(-1, D).astype(np.float64)
    kidx = tq.tq_unpack_indices(Kc).astype(np.int64)
    vidx = tq.tq_unpack_indices(Vc).astype(np.int64)
    Khat = oq.mse_dequantize(kidx, Kc.norm[:HKV * cap].cpu().numpy(), Pk, cbk["centroids"], math.sqrt(D))
    Vhat = oq.mse_dequantize(vidx, Vc.norm[:HKV * cap].cpu().numpy(), Pv, cbv["centroids"], math.sqrt(D))
    r = {"cos_k": float(_cos_rows(K, Khat).mean()), "cos_v": float(_cos_rows(V, Vhat).mean()),
         "want_k": math.sqrt(1 - cbk["distortion"]), "want_v": math.sqrt(1 - cbv["distortion"])}
    # inner-product correlation: GPU scores of 32 queries against the 2048 keys of head 0
    Q = synth.queries(21, HQ, D)
    ws = torch.empty(tq.tq_scores_workspace_size(kctx, HQ) // 4 + 4, device="cuda")
    sc = torch.empty((HQ, T), device="cuda")
    Kt = tq.CodeSet(kctx, T, tq.TQ_LAYOUT_TOKEN)
    tq.tq_encode(kctx, torch.from_numpy(np.ascontiguousarray(Kh[0, 0])).cuda(), Kt)
    tq.tq_scores(kctx, torch.from_numpy(Q).cuda(), Kt, sc, ws)
    exact = Q.astype(np.float64) @ Kh[0, 0].astype(np.float64).T
    r["ip_corr"] = float(np.corrcoef(exact.ravel(), sc.cpu().numpy().astype(np.float64).ravel())[0, 1])
    # attention output cosine against fp64 attention over the unquantized rows
    q = torch.from_numpy(Q.reshape(1, HQ, D)).cuda()
    out = torch.empty((1, HQ, D), device="cuda")
    wsd = torch.zeros(tq.tq_decode_workspace_size(kctx, 1, HQ, HKV, T) // 4 + 4, device="cuda")
    tq.tq_decode_attention(kctx, vctx, q, Kc, Vc, 1, HQ, HKV, T, cap, 1 / math.sqrt(D), out, wsd)
    torch.cuda.synchronize()
    assert kctx.poll() == tq.TQ_OK and vctx.poll() == tq.TQ_OK
    ref = oatt.decode_attention(Q.reshape(1, HQ, D).astype(np.float64), Kh.astype(np.float64),
                                Vh.astype(np.float64), 1 / math.sqrt(D))
    got = out.cpu().numpy().astype(np.float64)
    r["attn_cos"] = float(np.mean(np.sum(got * ref, -1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))))
    return r


def test_asymmetric_kv_quality_matches_the_distortion():
    res = {}
    for bk, bv in [(4, 4), (4, 2), (3, 3), (2, 2)]:
        r = _measure(bk, bv)
        res[(bk, bv)] = r
        print(f"\nK {bk} bit / V {bv} bit: cos(K) {r['cos_k']:.4f} (sqrt(1-D) {r['want_k']:.4f}), "
              f"cos(V) {r['cos_v']:.4f} (sqrt(1-D) {r['want_v']:.4f}), IP correlation {r['ip_corr']:.4f}, "
              f"attention output cosine {r['attn_cos']:.4f}")
        assert abs(r["cos_k"] - r["want_k"]) < 0.004 and abs(r["cos_v"] - r["want_v"]) < 0.004
        assert abs(r["ip_corr"] - r["want_k"]) < 0.01
    # the pages' figures on model caches ("sub-byte-kv-cache-quantization-turboquant",
    # 生产级精度 - 吞吐权衡参数): 4 bits 0.995 / 0.995, 2 bits 0.945 / 0.940
    assert abs(res[(4, 4)]["ip_corr"] - 0.995) < 0.003 and abs(res[(4, 4)]["cos_k"] - 0.995) < 0.003
    assert abs(res[(2, 2)]["ip_corr"] - 0.945) < 0.01 and abs(res[(2, 2)]["cos_k"] - 0.940) < 0.003
    # the softmax amplifies key error on these outlier-heavy rows, so the output
    # follows the key bits first: more K bits, better output, at any V bits
    a = {k: v["attn_cos"] for k, v in res.items()}
    assert a[(4, 4)] > a[(4, 2)] > a[(2, 2)] and a[(4, 4)] > a[(3, 3)] > a[(2, 2)]
