"""Bounded device waits that run out (the one form of failure detection that
needs no GPU fault): with tq_ctx_set_wait_limit(ctx, 0) every pipeline wait of
the tensor-memory encoders (d = 128 and d > 128) and of the scorer gives up before its first
poll.  The kernel must then stop, wait for its own copies in flight, free its
tensor memory and return; tq_status_poll reports TQ_ERR_TIMEOUT once and TQ_OK
after that, and the same context works again with the default bound (its
results then equal those of a context that never timed out).
"""

import math

import pytest

torch = pytest.importorskip("torch")

import kv_cache_vector_tq_gb300 as tq  # noqa: E402
from kv_cache_vector_tq_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT = 1 << 22


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()


def _pair(seed, d, b, mode=tq.TQ_MSE):
    G = synth.gaussian_matrix(seed, d)
    S = synth.qjl_matrix(seed, d) if mode == tq.TQ_PROD else None
    Pi = tq.tq_rotation_haar(G)
    return (tq.Context(d, b, mode, tq.TQ_ROT_DENSE, Pi, S), tq.Context(d, b, mode, tq.TQ_ROT_DENSE, Pi, S))


@pytest.mark.parametrize("d,b,mode,f16", [(256, 4, tq.TQ_MSE, False), (256, 4, tq.TQ_MSE, True),
                                          (128, 3, tq.TQ_MSE, False), (128, 4, tq.TQ_MSE, True),
                                          (128, 3, tq.TQ_PROD, False), (128, 3, tq.TQ_PROD, True)])
def test_encoder_wait_limit_zero_times_out_then_recovers(d, b, mode, f16):
    n = 300
    ctx, clean = _pair(31, d, b, mode)
    x = torch.from_numpy(synth.bulk_rows(31, n, d)).cuda()
    if f16:
        x = x.half()
    ref = tq.CodeSet(clean, n)
    tq.tq_encode(clean, x, ref)
    cs = tq.CodeSet(ctx, n)
    ctx.set_wait_limit(0)
    tq.tq_encode(ctx, x, cs)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_ERR_TIMEOUT
    assert ctx.poll() == tq.TQ_OK  # read once, then cleared
    ctx.set_wait_limit(DEFAULT_LIMIT)
    cs.codes.zero_()
    tq.tq_encode(ctx, x, cs)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK and clean.poll() == tq.TQ_OK
    assert torch.equal(cs.codes, ref.codes) and torch.equal(cs.norm, ref.norm)
    if mode == tq.TQ_PROD:
        assert torch.equal(cs.qjl, ref.qjl) and torch.equal(cs.rnorm, ref.rnorm)


@pytest.mark.parametrize("mode", [tq.TQ_MSE, tq.TQ_PROD])
def test_scorer_wait_limit_zero_times_out_then_recovers(mode):
    # 9 queries: past the one-launch scorer for up to 8 (it has no pipeline
    # waits), so the tensor-core scorer with its bounded waits runs
    d, b, n, M = 128, 3, 1000, 9
    ctx, clean = _pair(32, d, b, mode)
    keys = torch.from_numpy(synth.unit_rows(32, n, d)).cuda()
    cs = tq.CodeSet(clean, n)
    tq.tq_encode(clean, keys, cs)
    q = torch.from_numpy(synth.queries(32, M, d)).cuda()
    ws = torch.empty(tq.tq_scores_workspace_size(ctx, M) // 4 + 4, device="cuda")
    ref = torch.empty((M, n), device="cuda")
    tq.tq_scores(clean, q, cs, ref, ws)
    out = torch.full((M, n), float("nan"), device="cuda")
    ctx.set_wait_limit(0)
    tq.tq_scores(ctx, q, cs, out, ws)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_ERR_TIMEOUT
    assert ctx.poll() == tq.TQ_OK
    ctx.set_wait_limit(DEFAULT_LIMIT)
    tq.tq_scores(ctx, q, cs, out, ws)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK and clean.poll() == tq.TQ_OK
    assert torch.equal(out, ref)
    assert math.isfinite(float(out.abs().max()))
