"""Empty and degenerate sizes at the C ABI: no rows to encode, no keys or no
queries to score, no cached tokens.  Calls with nothing to do return TQ_OK and
write nothing; attention over zero tokens is undefined and is refused."""

import math

import numpy as np
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


def _ctx(d=128, b=3):
    return tq.Context(d, b, tq.TQ_MSE, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(synth.gaussian_matrix(0, d)))


def test_encode_zero_rows_writes_nothing():
    ctx = _ctx()
    cs = tq.CodeSet(ctx, 64, tq.TQ_LAYOUT_TOKEN)
    cs.codes.fill_(0x5A5A5A5A)
    cs.norm.fill_(7.0)
    x = torch.empty((0, 128), dtype=torch.float32, device="cuda")
    tq.tq_encode(ctx, x, cs)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    assert bool((cs.codes == 0x5A5A5A5A).all()) and bool((cs.norm == 7.0).all())


def test_scores_with_no_keys_or_no_queries():
    ctx = _ctx()
    cs = tq.CodeSet(ctx, 256, tq.TQ_LAYOUT_TOKEN)
    x = torch.from_numpy(synth.gaussian_rows(1, 256, 128)).cuda()
    tq.tq_encode(ctx, x, cs)
    q = torch.from_numpy(synth.gaussian_rows(2, 4, 128)).cuda()
    ws = torch.empty(tq.tq_scores_workspace_size(ctx, 4) // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((4, 8), -1.0, dtype=torch.float32, device="cuda")
    tq.tq_scores(ctx, q, cs, out, ws, first=10, N=0)  # no keys
    q0 = torch.empty((0, 128), dtype=torch.float32, device="cuda")
    tq.tq_scores(ctx, q0, cs, out, ws, first=0, N=256)  # no queries
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
    assert bool((out == -1.0).all())


def test_decode_over_zero_tokens_is_refused():
    ctx = _ctx()
    B, Hq, Hkv, cap, d = 1, 8, 2, 16, 128
    K = tq.CodeSet(ctx, B * Hkv * cap, tq.TQ_LAYOUT_TOKEN)
    V = tq.CodeSet(ctx, B * Hkv * cap, tq.TQ_LAYOUT_PAIR)
    q = torch.zeros((B, Hq, d), dtype=torch.float16, device="cuda")
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(ctx, B, Hq, Hkv, 1) // 4 + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(Exception):
        tq.tq_decode_attention(ctx, ctx, q, K, V, B, Hq, Hkv, 0, cap, 1 / math.sqrt(d), out, ws)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK
