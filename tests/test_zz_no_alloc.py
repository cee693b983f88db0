"""tq_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (and so cannot pass a workspace either), e.g. code that
runs where cudaMalloc is unavailable or forbidden.  Its scratch is an array
built into the library.

This file is collected last on purpose.  Each case calls the entry point
through the C ABI twice in a row and compares each result with
tq_decode_attention (the call with a caller-provided workspace): the same
kernel runs on the same inputs, so the outputs must be bit-identical, which
would expose stale partial states or arrival counters left in the shared
array.  It also checks that a shape needing more scratch than the built-in
array is refused before anything runs.
"""

import math

import pytest

torch = pytest.importorskip("torch")

import kv_cache_vector_tq_gb300 as tq  # noqa: E402
from kv_cache_vector_tq_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()


def _context(seed, d, b):
    G = synth.gaussian_matrix(seed, d)
    return tq.Context(d, b, tq.TQ_MSE, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(G))


@pytest.mark.parametrize("case", ["mse_b4_gqa4", "mse_b3_gqa8", "prod_keys_gqa4"])
def test_noalloc_matches_workspace_call_twice(case):
    d, B, Hkv, seq = 128, 1, 8, 4099
    Hq = 64 if case == "mse_b3_gqa8" else 32
    cap = (seq + 15) // 16 * 16
    vctx = _context(11, d, 3 if case == "mse_b3_gqa8" else 4)
    if case == "prod_keys_gqa4":
        G = synth.gaussian_matrix(11, d)
        kctx = tq.Context(d, 3, tq.TQ_PROD, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(G), synth.qjl_matrix(11, d))
    else:
        kctx = vctx
    Kh, Vh = synth.kv_layer(11, 0, B, Hkv, seq, d)
    Kc = tq.CodeSet(kctx, B * Hkv * cap, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(vctx, B * Hkv * cap, tq.TQ_LAYOUT_PAIR)
    tq.tq_encode(kctx, torch.from_numpy(Kh.reshape(-1, d)).cuda(), Kc, 0, seq, cap)
    tq.tq_encode(vctx, torch.from_numpy(Vh.reshape(-1, d)).cuda(), Vc, 0, seq, cap)
    scale = 1.0 / math.sqrt(d)
    ws = torch.zeros(tq.tq_decode_workspace_size(kctx, B, Hq, Hkv, seq) // 4 + 4, dtype=torch.float32,
                     device="cuda")
    for call in range(2):
        q = torch.from_numpy(synth.queries(20 + call, B * Hq, d).reshape(B, Hq, d)).cuda().half()
        ref = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
        tq.tq_decode_attention(kctx, vctx, q, Kc, Vc, B, Hq, Hkv, seq, cap, scale, ref, ws)
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
        tq.tq_decode_attention_noalloc(kctx, vctx, q, Kc, Vc, B, Hq, Hkv, seq, cap, scale, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert torch.equal(out, ref), (
            f"call {call}: max difference {(out - ref).abs().max().item()} between the calls with "
            "and without a workspace")
    assert kctx.poll() == tq.TQ_OK and vctx.poll() == tq.TQ_OK


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 4096 sequences x 128 KV heads need more counters than the 2 MiB built in;
    # the size check comes before anything touches the (tiny) code sets
    d, b, B, Hq, Hkv, seq, cap = 128, 2, 4096, 128, 128, 16, 16
    ctx = _context(12, d, b)
    assert tq.tq_decode_workspace_size(ctx, B, Hq, Hkv, seq) > (2 << 20)
    Kc = tq.CodeSet(ctx, 16, tq.TQ_LAYOUT_TOKEN)
    Vc = tq.CodeSet(ctx, 16, tq.TQ_LAYOUT_PAIR)
    q = torch.zeros((B, Hq, d), dtype=torch.float16, device="cuda")
    out = torch.zeros((1, 1, d), dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TqError) as err:
        tq.tq_decode_attention_noalloc(ctx, ctx, q, Kc, Vc, B, Hq, Hkv, seq, cap, 1.0, out)
    assert err.value.status == tq.TQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (out == 0).all()
