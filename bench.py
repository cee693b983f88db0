#!/usr/bin/env python
"""Benchmark of the TurboQuant decode hot path on one GB300 (or N replicas).

Workload (the decode-attention configuration): one layer, batch 1, 32 query
heads / 8 KV heads (GQA 4), head_dim 128, 16384 cached tokens, fp16 K/V drawn
N(0,1) with 4 outlier channels x10, K and V TurboQuant_MSE at b bits (default
4; --bits 2 for the other half of the configuration).

One decode step = append the new token (encode its K and V: 2 x 8 vectors into
the caches, norm -> rotation -> bucketize -> pack) and attend over the 16384
tokens (query pre-rotation, attention over the packed cache, merge + inverse
rotation), all in one fused kernel launch (tq_decode_step).  A benchmark step runs one decode step on each of R
independent replica caches (distinct HBM regions together larger than 4x L2),
so every step streams its caches from HBM; the R caches are one batch-1 layer
each.  Timed steps replay a CUDA graph of one benchmark step.

value    = algorithmic decode bytes / s (codes + norms of K and V for all cached
           tokens, query, output, and the appended token) over the timed steps.
e2e      = the same metric with the step inputs (query, new K/V token: one
           pinned host block, one copy) copied from pinned host memory and the
           output copied back every decode step; the replicas alternate between
           two streams with their own buffers, so one replica's copies overlap
           another's decode, and a benchmark step (copies included) replays as
           one CUDA graph.
roofline = one decode-attention call alone (the same kernel without the
           append: query rotation, tiles and merge in one launch) against the
           measured HBM copy peak; traffic = its DRAM bytes per launch from the
           ncu capture recorded in profiles/traffic.json, while the kernel's
           source still matches that capture (else null).
"""

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D, B, HQ, HKV, SEQ = 128, 1, 32, 8, 16384
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--bits", type=int, default=4, choices=[1, 2, 3, 4])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="decode: skip the other configurations' measurements in the same run")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "encode", "scores", "longctx", "keys", "prefill", "mixed"],
                    help="decode (the headline) or a secondary workload (see bench_workloads.py)")
    ap.add_argument("--dim", type=int, default=3072, help="encode: vector dimension")
    ap.add_argument("--rows", type=int, default=100_000, help="encode: number of vectors")
    ap.add_argument("--rotation", default="dense", choices=["dense", "hadamard"], help="encode: rotation")
    ap.add_argument("--layers", type=int, default=80, help="longctx: layers run in sequence")
    return ap.parse_args()


def decode_bytes(bits):
    """Algorithmic bytes of one decode step (see module docstring)."""
    per_tok = 2 * (D * bits // 8 + 4)           # K + V codes and norms
    cache = B * HKV * SEQ * per_tok
    q_out = B * HQ * D * 2 + B * HQ * D * 4      # fp16 query in, fp32 output
    append = 2 * B * HKV * (D * 2 + D * bits // 8 + 4)  # fp16 K/V token in, codes out
    return cache + q_out + append, cache + q_out


def load_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampler running across the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except Exception:
            pass
        os.unlink(self.path)
        return self.summary(rows)

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max((float(r[2]) for r in rows if r[2].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


def dist_init(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- tq arm
def build_replicas(tq, synth, bits, R):
    import numpy as np
    import torch
    G = synth.gaussian_matrix(0, D)
    ctx = tq.Context(D, bits, tq.TQ_MSE, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(G))
    cap = SEQ
    Kh, Vh = synth.kv_layer(0, 0, B, HKV, SEQ, D)
    kx = torch.from_numpy(np.ascontiguousarray(Kh[:, :, :SEQ - 1].reshape(-1, D))).cuda()
    vx = torch.from_numpy(np.ascontiguousarray(Vh[:, :, :SEQ - 1].reshape(-1, D))).cuda()
    K0 = tq.CodeSet(ctx, B * HKV * cap, tq.TQ_LAYOUT_TOKEN)
    V0 = tq.CodeSet(ctx, B * HKV * cap, tq.TQ_LAYOUT_PAIR)
    tq.tq_encode(ctx, kx, K0, 0, SEQ - 1, cap)   # prefill all but the last token
    tq.tq_encode(ctx, vx, V0, 0, SEQ - 1, cap)
    torch.cuda.synchronize()
    reps = [(K0, V0)]
    for _ in range(R - 1):
        Kr = tq.CodeSet(ctx, B * HKV * cap, tq.TQ_LAYOUT_TOKEN)
        Vr = tq.CodeSet(ctx, B * HKV * cap, tq.TQ_LAYOUT_PAIR)
        Kr.codes.copy_(K0.codes), Kr.norm.copy_(K0.norm)
        Vr.codes.copy_(V0.codes), Vr.norm.copy_(V0.norm)
        reps.append((Kr, Vr))
    # the step's inputs (query, new K, new V; fp16) as views of one buffer, so
    # that an end-to-end step moves them from the host in one copy
    nq, nk = B * HQ * D, B * HKV * D
    inputs = torch.empty(nq + 2 * nk, dtype=torch.float16, device="cuda")
    q = inputs[:nq].view(B, HQ, D)
    knew = inputs[nq:nq + nk].view(-1, D)
    vnew = inputs[nq + nk:].view(-1, D)
    q.copy_(torch.from_numpy(synth.queries(0, B * HQ, D).reshape(B, HQ, D)).to(torch.float16))
    knew.copy_(torch.from_numpy(np.ascontiguousarray(Kh[:, :, SEQ - 1].reshape(-1, D))))
    vnew.copy_(torch.from_numpy(np.ascontiguousarray(Vh[:, :, SEQ - 1].reshape(-1, D))))
    return ctx, reps, cap, knew, vnew, q, inputs


def run_tq(args, world, rank, local):
    import numpy as np
    import torch

    import kv_cache_vector_tq_gb300 as tq
    from bench_workloads import traffic
    from kv_cache_vector_tq_gb300 import synth

    torch.cuda.set_device(local)
    bits = args.bits
    step_bytes, attn_bytes = decode_bytes(bits)
    cache_bytes = B * HKV * SEQ * 2 * (D * bits // 8 + 4)
    R = max(2, int(math.ceil(4 * L2_BYTES / cache_bytes)))
    ctx, reps, cap, knew, vnew, q, inputs = build_replicas(tq, synth, bits, R)
    scale = 1.0 / math.sqrt(D)
    ws = torch.zeros(tq.tq_decode_workspace_size(ctx, B, HQ, HKV, SEQ) // 4 + 64, dtype=torch.float32, device="cuda")
    out = torch.empty((B, HQ, D), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def decode_step(r, with_append=True, bufs=None):
        K, V = reps[r]
        qq, kk, vv, oo, ww = bufs or (q, knew, vnew, out, ws)
        if with_append:  # one launch: encode the new token's K/V into slot SEQ-1, then attend
            tq.tq_decode_step(ctx, ctx, qq, kk, vv, K, V, B, HQ, HKV, SEQ, cap, scale, oo, ww)
        else:
            tq.tq_decode_attention(ctx, ctx, qq, K, V, B, HQ, HKV, SEQ, cap, scale, oo, ww)

    # eager warm-up (sets kernel attributes outside capture), then graphs
    with torch.cuda.stream(stream):
        for r in range(R):
            decode_step(r)
    torch.cuda.synchronize()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        for r in range(R):
            decode_step(r)
    g_attn = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_attn, stream=stream):
        for r in range(R):
            decode_step(r, with_append=False)
    # end to end: replicas alternate between two streams, each with its own
    # input block, output and workspace, so one replica's copies overlap
    # another's decode (the replicas are independent caches)
    inputs2 = torch.empty_like(inputs)
    nq, nk = q.numel(), knew.numel()
    sets = [(q, knew, vnew, out, ws, inputs),
            (inputs2[:nq].view_as(q), inputs2[nq:nq + nk].view_as(knew), inputs2[nq + nk:].view_as(vnew),
             torch.empty_like(out), torch.zeros_like(ws), inputs2)]
    in_h = inputs.cpu().pin_memory()  # q, k_new, v_new of a step, one pinned block
    out_h = [torch.empty((B, HQ, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    side = torch.cuda.Stream()
    # one benchmark step end to end, as one graph: per replica the copy of its
    # inputs from pinned host memory, the decode step and the copy of its
    # output back, the replicas alternating between two streams
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        fork = torch.cuda.Event()
        fork.record(stream)
        side.wait_event(fork)
        for r in range(R):
            st_r, bs = (stream, side)[r % 2], sets[r % 2]
            with torch.cuda.stream(st_r):
                bs[5].copy_(in_h, non_blocking=True)
                decode_step(r, bufs=bs[:5])
                out_h[r % 2].copy_(bs[3], non_blocking=True)
        join = torch.cuda.Event()
        join.record(side)
        stream.wait_event(join)
    torch.cuda.synchronize()
    assert ctx.poll() == tq.TQ_OK

    # ---------------- warm-up steps, then exactly K timed steps
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_step.replay()
    torch.cuda.synchronize()
    barrier(world)
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            g_step.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    total_bytes = world * args.steps * R * step_bytes
    value_gbs = total_bytes / (ms * 1e-3) / 1e9

    # ---------------- decode-attention call alone (roofline unit)
    reps_attn = max(5, min(200, args.steps))
    with torch.cuda.stream(stream):
        g_attn.replay()
        e0.record(stream)
        for _ in range(reps_attn):
            g_attn.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    attn_us = e0.elapsed_time(e1) * 1e3 / (reps_attn * R)
    peak, peak_kind = load_peak()
    achieved = attn_bytes / (attn_us * 1e-6) / 1e9

    # ---------------- end to end through the C ABI with host buffers
    e2e_steps = max(3, min(args.steps, 100))
    with torch.cuda.stream(stream):
        g_e2e.replay()  # untimed
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            g_e2e.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_gbs = world * e2e_steps * R * step_bytes / (e2e_ms * 1e-3) / 1e9
    h2d = R * (q.numel() * 2 + knew.numel() * 2 + vnew.numel() * 2)
    d2h = R * out.numel() * 4
    assert ctx.poll() == tq.TQ_OK

    launches_per_decode = 1  # the fused decode-step kernel
    line = {
        "metric": "decode-attn HBM GB/s",
        "value": round(value_gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": f"u{bits} codes, f16 operands, f32 accumulate",
        "data": "synthetic (seeded N(0,1) fp16 K/V with 4 outlier channels x10)",
        "config": {
            "workload": f"decode attention, 1 layer, batch 1, 32 q / 8 kv heads, head_dim 128, seq 16384, "
                        f"K/V TurboQuant_MSE b={bits}; step = append 1 token + attend, on each of {R} replica caches",
            "bits": bits, "replicas": R, "seq": SEQ, "heads_q": HQ, "heads_kv": HKV, "head_dim": D,
            "l2": f"inputs larger than L2: {R} distinct caches x {cache_bytes / 1e6:.1f} MB per step",
            "bytes_per_decode": step_bytes, "parallelism": f"replicas x{world}",
            "decode_steps_per_s": round(world * args.steps * R / (ms * 1e-3), 1),
            "tokens_scored_per_s": round(world * args.steps * R * SEQ * HQ / (ms * 1e-3), 1),
        },
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic(os.path.dirname(os.path.abspath(__file__)), f"decode_b{bits}"),
            "kernel": "decode_step_kernel without the append (one launch per call)", "peak_kind": peak_kind,
            "us_per_call": round(attn_us, 3), "bytes_per_call": attn_bytes,
        },
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * R * launches_per_decode,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(tq, ctx, reps[0], bits, cap, q)
    if rank == 0 and not args.no_extras:
        del reps
        torch.cuda.empty_cache()
        line["configs"] = other_configs(args, world, rank, local)
    return line if rank == 0 else None


def _summary(sub_line, keep=()):
    """The figures of a secondary workload's line that the headline line carries."""
    r = sub_line.get("roofline") or {}
    out = {"workload": sub_line["config"]["workload"], "metric": sub_line["metric"], "value": sub_line["value"],
           "unit": sub_line["unit"], "ms_per_step": sub_line["ms_per_step"], "steps": sub_line["steps"],
           "roofline": {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "kernel",
                                          "peak_kind") if k in r},
           "clocks": sub_line.get("clocks")}
    for k in keep:
        if k in sub_line["config"]:
            out[k] = sub_line["config"][k]
    return out


def other_configs(args, world, rank, local):
    """Every other configuration of the metric, measured in this run with its own
    warm-up and timed steps (the same runners as --workload ...): decode at
    b = 2, the d = 128 encoder (long-context prefill and the Prod keys), Prod
    scores over 1M keys, the 4096-key encode + score, the 80-layer long-context
    decode, and bulk encode of fp32 rows (d = 128 at N = 1M, d = 1536 / 3072 at
    N = 100K; dense and Hadamard rotations)."""
    import types

    import torch

    import bench_workloads as bw

    def ns(**kw):
        base = dict(steps=20, warmup=3, no_cpu_baseline=True, no_extras=True, bits=4, dim=3072, rows=100_000,
                    rotation="dense", layers=80, gpus=args.gpus)
        base.update(kw)
        return types.SimpleNamespace(**base)

    out = {}
    b2 = run_tq(ns(steps=max(20, min(args.steps, 400)), bits=2), world, rank, local)
    out["decode_b2"] = _summary(b2, ("bits", "replicas")) | {"us_per_call": b2["roofline"]["us_per_call"]}
    torch.cuda.empty_cache()
    pf = bw.run_prefill(ns(steps=10), world, rank, local, ROOT, Clocks, {})
    out["encode_d128"] = _summary(pf, ("vectors", "prod_encode"))
    out["scores_prod_1m"] = _summary(bw.run_scores(ns(steps=20), world, rank, local, ROOT, Clocks, {}))
    out["keys_4096"] = _summary(bw.run_keys(ns(steps=50), world, rank, local, ROOT, Clocks, {}),
                                ("us_per_encode_plus_score",))
    torch.cuda.empty_cache()
    lc = bw.run_longctx(ns(steps=5), world, rank, local, ROOT, Clocks, {})
    out["longctx_80_layers"] = _summary(lc, ("prefill_encode_mvec_s", "ms_per_layer", "layers"))
    torch.cuda.empty_cache()
    mx = bw.run_mixed(ns(steps=20, bits=2), world, rank, local, ROOT, Clocks, {})
    out["decode_2p5bit"] = _summary(mx, ("encode_mvec_s", "encode_roofline")) | {
        "us_per_call": mx["roofline"]["us_per_call"]}
    torch.cuda.empty_cache()
    for rot in ("dense", "hadamard"):
        ln = bw.run_encode(ns(steps=5, dim=128, rows=1_000_000, rotation=rot), world, rank, local, ROOT, Clocks, {})
        out[f"bulk_encode_d128_{rot}_1m"] = _summary(ln)
        torch.cuda.empty_cache()
    for d in (1536, 3072):
        for rot in ("dense", "hadamard"):
            ln = bw.run_encode(ns(steps=5, dim=d, rows=100_000, rotation=rot), world, rank, local, ROOT, Clocks, {})
            out[f"bulk_encode_d{d}_{rot}_100k"] = _summary(ln)
            torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- oracle timing
def oracle_decode_sample(bits, idx_k, idx_v, kn, vn, q_np, heads, tokens):
    """Oracle decode attention (explicit dequantization, fp64) on `heads` KV
    heads x `tokens` tokens of the cache; returns seconds."""
    import numpy as np

    from kv_cache_vector_tq_gb300 import synth
    from oracle import attention as oatt
    from oracle import codebook as ocb
    from oracle import rotation as orot
    Pi = orot.haar_rotation(synth.gaussian_matrix(0, D))
    cb = ocb.build_codebook(D, bits)
    t0 = time.perf_counter()
    Khat = oatt.dequantize_cache(idx_k[:heads, :tokens].reshape(-1, D), kn[:heads, :tokens].reshape(-1), Pi,
                                 cb["centroids"], math.sqrt(D), 1, heads, tokens)
    Vhat = oatt.dequantize_cache(idx_v[:heads, :tokens].reshape(-1, D), vn[:heads, :tokens].reshape(-1), Pi,
                                 cb["centroids"], math.sqrt(D), 1, heads, tokens)
    oatt.decode_attention(q_np[:, :heads * (HQ // HKV)], Khat, Vhat, 1 / math.sqrt(D))
    return time.perf_counter() - t0


def cache_for_oracle(tq, reps0, cap):
    import numpy as np
    K, V = reps0
    idx_k = np.stack([tq.tq_unpack_indices(K, h * cap, SEQ) for h in range(HKV)])
    idx_v = np.stack([tq.tq_unpack_indices(V, h * cap, SEQ) for h in range(HKV)])
    kn = K.norm.cpu().numpy().reshape(HKV, cap)[:, :SEQ].astype(np.float64)
    vn = V.norm.cpu().numpy().reshape(HKV, cap)[:, :SEQ].astype(np.float64)
    return idx_k, idx_v, kn, vn


def oracle_band_check(tq, reps0, bits, cap):
    """The oracle's encoder on a sample of the cache's source rows (first KV
    head, 4096 tokens): the share of coordinates inside the 1e-6 band around a
    threshold, and how many GPU codes differ from the oracle's outside it."""
    import numpy as np

    from kv_cache_vector_tq_gb300 import synth
    from oracle import codebook as ocb
    from oracle import quantizer as oq
    from oracle import rotation as orot
    Pi = orot.haar_rotation(synth.gaussian_matrix(0, D))
    cb = ocb.build_codebook(D, bits)
    Kh, _ = synth.kv_layer(0, 0, B, HKV, SEQ, D)
    n = 4096
    X = Kh[0, 0, :n].astype(np.float64)
    ref, _, v = oq.mse_quantize(X, Pi, cb["centroids"], math.sqrt(D))
    band = oq.near_threshold(v, cb["centroids"])
    got = tq.tq_unpack_indices(reps0[0], 0, n).astype(np.int64)
    return {"band_frac": float(band.mean()), "coordinates": int(band.size),
            "index_mismatch_outside_band": int(((got != ref) & ~band).sum()),
            "sample": f"K rows 0-{n - 1} of KV head 0 (fp16 N(0,1), outlier channels), b={bits}"}


def cpu_baseline(tq, ctx, reps0, bits, cap, q):
    import numpy as np
    idx_k, idx_v, kn, vn = cache_for_oracle(tq, reps0, cap)
    q_np = q.float().cpu().numpy().astype(np.float64)
    total, done_bytes, runs = 0.0, 0, 0
    per_kv_head = SEQ * 2 * (D * bits // 8 + 4)
    while total < 10.0 and runs < 8:
        total += oracle_decode_sample(bits, idx_k, idx_v, kn, vn, q_np, HKV, SEQ)
        done_bytes += HKV * per_kv_head
        runs += 1
    return {"value": round(done_bytes / total / 1e9, 6), "unit": "GB/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{runs} full decode steps (8 KV heads x 16384 tokens, fp64 explicit dequantization)",
            "parity": oracle_band_check(tq, reps0, bits, cap)}


# ---------------------------------------------------------------- oracle timing, secondary workloads
def cpu_encode_baseline(d, bits, rot, rotm):
    """The oracle encoder timed on the host cores on a bounded sample of rows."""
    import numpy as np

    from kv_cache_vector_tq_gb300 import synth
    from oracle import codebook as ocb
    from oracle import quantizer as oq
    from oracle import rotation as orot
    Pi = orot.hadamard_rotation(d, rotm) if rot == "hadamard" else np.asarray(rotm)
    cb = ocb.build_codebook(d, bits)
    n = 256 if d >= 3072 else 512
    X = synth.bulk_rows(0, n, d).astype(np.float64)
    total, done = 0.0, 0
    while total < 10.0 and done < 64 * n:
        t0 = time.perf_counter()
        oq.mse_quantize(X, Pi, cb["centroids"], math.sqrt(d))
        total += time.perf_counter() - t0
        done += n
    return {"value": round(done / total / 1e6, 6), "unit": "Mvec/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "sample": f"{done} rows of d={d} (fp64 dense rotation, exhaustive nearest centroid)"}


def cpu_scores_baseline(tq, cs, q, G, S):
    """Oracle Prod scores (explicit dequantization) on a 64 x 65536-key sample."""
    import numpy as np

    from oracle import attention as oatt
    from oracle import codebook as ocb
    from oracle import rotation as orot
    n = 65536
    ids, bits = tq.tq_unpack_indices(cs, 0, n, with_bits=True)
    Pi = orot.haar_rotation(G)
    cb = ocb.build_codebook(128, 2)
    s = cs.norm[:n].cpu().numpy().astype(np.float64)
    g = cs.rnorm[:n].cpu().numpy().astype(np.float64)
    Q = q.cpu().numpy().astype(np.float64)
    t0 = time.perf_counter()
    oatt.prod_scores(Q, ids.astype(np.int64), s, bits, g, Pi, S, cb["centroids"], math.sqrt(128))
    t = time.perf_counter() - t0
    return {"value": round(Q.shape[0] * n / t, 1), "unit": "tokens scored/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "sample": f"64 queries x {n} keys (fp64 explicit dequantization)"}


def cpu_mixed_baseline(tq, rep, b, cap, q):
    """Oracle decode at b + 1/2 bits (explicit dequantization, fp64) on one KV
    head x 4096 tokens of the GPU's cache, as decode-attn GB/s of its bytes."""
    import numpy as np

    from kv_cache_vector_tq_gb300 import synth
    from oracle import attention as oatt
    from oracle import codebook as ocb
    from oracle import quantizer as oq
    from oracle import rotation as orot
    K, V = rep
    n = 4096
    lo, hi = ocb.build_codebook(D, b)["centroids"], ocb.build_codebook(D, b + 1)["centroids"]
    Pk = orot.haar_rotation(synth.gaussian_matrix(0, D))
    Pv = orot.haar_rotation(synth.gaussian_matrix(1, D))
    ik, iv = tq.tq_unpack_indices(K, 0, n).astype(np.int64), tq.tq_unpack_indices(V, 0, n).astype(np.int64)
    kn = K.norm[:n].cpu().numpy().astype(np.float64)
    vn = V.norm[:n].cpu().numpy().astype(np.float64)
    qs = q[:, :HQ // HKV].float().cpu().numpy().astype(np.float64)
    t0 = time.perf_counter()
    Kh = oq.mixed_dequantize(ik, kn, Pk, lo, hi, b, math.sqrt(D)).reshape(1, 1, n, D)
    Vh = oq.mixed_dequantize(iv, vn, Pv, lo, hi, b, math.sqrt(D)).reshape(1, 1, n, D)
    oatt.decode_attention(qs, Kh, Vh, 1 / math.sqrt(D))
    t = time.perf_counter() - t0
    nbytes = n * 2 * (K.words_per_vec * 4 + 4)
    return {"value": round(nbytes / t / 1e9, 6), "unit": "GB/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "sample": f"1 KV head x {n} tokens, {HQ // HKV} query heads (fp64 explicit dequantization)"}


# ---------------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    """The oracle as it stands, timed on the host cores, same metric/config."""
    if rank != 0:
        return None
    import numpy as np

    from kv_cache_vector_tq_gb300 import synth
    from oracle import codebook as ocb
    from oracle import quantizer as oq
    from oracle import rotation as orot
    bits = args.bits
    Pi = orot.haar_rotation(synth.gaussian_matrix(0, D))
    cb = ocb.build_codebook(D, bits)
    Kh, Vh = synth.kv_layer(0, 0, B, HKV, SEQ, D)
    # codes of the cache by the oracle's own encoder (untimed setup)
    idx_k = np.empty((HKV, SEQ, D), dtype=np.int64)
    idx_v = np.empty((HKV, SEQ, D), dtype=np.int64)
    kn = np.empty((HKV, SEQ))
    vn = np.empty((HKV, SEQ))
    for h in range(HKV):
        idx_k[h], kn[h], _ = oq.mse_quantize(Kh[0, h].astype(np.float64), Pi, cb["centroids"], math.sqrt(D))
        idx_v[h], vn[h], _ = oq.mse_quantize(Vh[0, h].astype(np.float64), Pi, cb["centroids"], math.sqrt(D))
    q_np = synth.queries(0, B * HQ, D).reshape(B, HQ, D).astype(np.float16).astype(np.float64)
    # bounded sample per step: heads x tokens chosen so W + K steps take ~2 minutes
    t_one = oracle_decode_sample(bits, idx_k, idx_v, kn, vn, q_np, 1, 2048)
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(min(SEQ, max(256, 2048 * per_step_budget / max(t_one, 1e-6))))
    heads = 1
    for _ in range(args.warmup):
        oracle_decode_sample(bits, idx_k, idx_v, kn, vn, q_np, heads, tokens)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_decode_sample(bits, idx_k, idx_v, kn, vn, q_np, heads, tokens)
    per_tok = 2 * (D * bits // 8 + 4)
    gbs = args.steps * heads * tokens * per_tok / t / 1e9
    sample = f"1 KV head (4 query heads) x {tokens} tokens per step, fp64 explicit dequantization"
    return {
        "impl": "reference", "metric": "decode-attn HBM GB/s", "value": round(gbs, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeds as the tq arm)",
        "config": {"workload": f"decode attention, 1 layer, batch 1, 32 q / 8 kv heads, head_dim 128, seq 16384, "
                               f"K/V TurboQuant_MSE b={bits}",
                   "bits": bits, "seq": SEQ, "heads_q": HQ, "heads_kv": HKV, "head_dim": D,
                   "sampled": sample},
        "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": len(os.sched_getaffinity(0)),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_init(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    elif args.workload != "decode":
        import bench_workloads as bw
        run = {"encode": bw.run_encode, "scores": bw.run_scores, "longctx": bw.run_longctx,
               "keys": bw.run_keys, "prefill": bw.run_prefill, "mixed": bw.run_mixed}[args.workload]
        line = run(args, world, rank, local, ROOT, Clocks,
                   {"encode": cpu_encode_baseline, "scores": cpu_scores_baseline, "mixed": cpu_mixed_baseline})
    else:
        line = run_tq(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
