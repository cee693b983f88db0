"""Secondary workloads of bench.py (--workload encode | scores | longctx | keys | prefill | mixed).

Each prints one JSON line in the same shape as the decode headline:
  encode   bulk indexing: b = 4, d = --dim (1536 / 3072), N = --rows fp32 rows
           N(0, 1) with a seeded 1 % of the rows x50, dense Haar or randomized
           Hadamard rotation (--rotation); metric encode Mvec/s.
  scores   TurboQuant_Prod b = 3 (2-bit MSE + 1-bit QJL), d = 128, 1M unit-norm
           keys, 64 queries; metric tokens (query-key pairs) scored/s.
  longctx  decode at a 70B-like shape: 64 q / 8 kv heads, head_dim 128,
           seq 131072, batch 1, b = 3 K/V, --layers layers run in sequence
           (80 by default); per layer the cache is prefilled by tq_encode
           (timed separately), then one decode step (append + attend) runs
           over all layers; metric decode-attn HBM GB/s.
  keys     d = 128, b = 3: encode 4096 fp32 keys (channels 0-3 x20), then score
           one query against them; metric encode Mvec/s (scores in config).
  mixed    the decode layer of the headline at b + 1/2 bits per coordinate
           (--bits 1..3, 2.5 bits by default): append with tq_encode, then
           attend; metric decode-attn HBM GB/s, the encoder at that width on
           1M fp16 rows in config.
Inputs of the large workloads are generated on the device (torch's seeded
generator) with the same distributions as the seeded host recipes the parity
tests use; the parity tests cover the same kernels on host-generated rows.
The host baselines (the oracle timed on the host cores) are passed in by
bench.py as `cpu`.
"""

import math
import os
import time


def _peaks(root, sustained=False):
    """HBM GB/s, dense bf16 TFLOP/s and where they come from.  `sustained`:
    the bf16 figure of a seconds-long loop under the power cap (for a timed
    region that long), else the burst figure."""
    import json
    try:
        with open(os.path.join(root, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        if sustained and "bf16_tflops_sustained" in j:
            return float(j["hbm_gbs"]), float(j["bf16_tflops_sustained"]), "measured (sustained bf16)"
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1700.0 if sustained else 1900.0, "fallback"


def code_digest(text):
    """SHA-256 of C/C++/CUDA source with its comments and whitespace removed,
    so that an edit of comments alone keeps the digest (string literals kept)."""
    import hashlib
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":  # a literal, copied up to its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return hashlib.sha256(" ".join("".join(out).split()).encode()).hexdigest()


def traffic(root, key):
    """DRAM bytes (read + written) of one launch of the kernel recorded under
    `key` in profiles/traffic.json, or None when no row matches or the code of
    the kernel's source file has changed since that capture (its digest by
    code_digest differs)."""
    import json
    try:
        with open(os.path.join(root, "profiles", "traffic.json")) as f:
            rows = json.load(f)["rows"]
    except (OSError, ValueError, KeyError):
        return None
    for r in rows:
        if r.get("key") != key:
            continue
        try:
            with open(os.path.join(root, r["source"]), encoding="utf-8") as f:
                digest = code_digest(f.read())
        except (OSError, KeyError):
            return None
        return int(r["read_bytes"]) + int(r["write_bytes"]) if digest == r.get("code_digest") else None
    return None


def _timed(fn, steps, warmup, stream, clocks_cls, local, flush=None, graph=False):
    """W warm-up calls, then K timed calls bracketed by events on `stream`.
    With `flush`, L2 is flushed between calls and only the calls are timed.
    With `graph`, one call is captured as a CUDA graph after the warm-up and
    the timed calls replay it (no host launch gaps between calls)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        fn = g.replay
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
    clocks = clocks_cls(local)
    clocks.start()
    time.sleep(0.2)
    total = 0.0
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        total = e0.elapsed_time(e1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                flush()
                a.record(stream)
                fn()
                b.record(stream)
        torch.cuda.synchronize()
        total = sum(a.elapsed_time(b) for a, b in evs)
    clk = clocks.stop()
    return total, clk


def _line(args, world, metric, value, unit, ms_per_step, dtype, data, config, roofline, e2e, launches, clk):
    return {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": data, "config": config,
        "roofline": roofline, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
    }


# ---------------------------------------------------------------- bulk encode
def run_encode(args, world, rank, local, root, clocks_cls, cpu):
    import numpy as np
    import torch

    import kv_cache_vector_tq_gb300 as tq
    from kv_cache_vector_tq_gb300 import synth
    torch.cuda.set_device(local)
    d, N, bits, rot = args.dim, args.rows, 4, args.rotation
    if rot == "hadamard":
        rotm = synth.hadamard_signs(0, d)
        ctx = tq.Context(d, bits, tq.TQ_MSE, tq.TQ_ROT_HADAMARD, rotm)
    else:
        rotm = tq.tq_rotation_haar(synth.gaussian_matrix(0, d))
        ctx = tq.Context(d, bits, tq.TQ_MSE, tq.TQ_ROT_DENSE, rotm)
    gen = torch.Generator(device="cuda").manual_seed(1234 + rank)
    x = torch.randn((N, d), generator=gen, device="cuda", dtype=torch.float32)
    k = max(1, N // 100)
    rows = torch.randperm(N, generator=gen, device="cuda")[:k]
    x[rows] *= 50.0
    cs = tq.CodeSet(ctx, N, tq.TQ_LAYOUT_TOKEN)
    stream = torch.cuda.Stream()
    total_ms, clk = _timed(lambda: tq.tq_encode(ctx, x, cs, stream=stream), args.steps, args.warmup, stream,
                           clocks_cls, local, graph=True)
    assert ctx.poll() == tq.TQ_OK
    sec = total_ms * 1e-3
    mvec = world * args.steps * N / sec / 1e6
    hbm, bf16, kind = _peaks(root, sustained=total_ms > 1000.0)  # a timed region of seconds runs at the power cap
    bytes_per_vec = 4 * d + d * bits // 8 + 4
    if rot == "hadamard" or d == 128:
        # the Hadamard kernel, and the d = 128 tensor-memory kernel on fp32 rows
        # (three 32.8 KFLOP products per 580 B: the bytes bind first; it also
        # serves d = 128 Hadamard contexts, with H·D/√d as its matrix), are HBM-bound
        kern = "encode128_kernel" if d == 128 else "encode_wht_kernel"
        key = f"encode128_f32_n{N // 1000}k" if d == 128 else f"encode_wht_d{d}_n{N // 1000}k"
        ach = args.steps * N * bytes_per_vec / sec / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                "traffic": traffic(root, key), "kernel": kern, "peak_kind": kind,
                "bytes_per_vector": bytes_per_vec}
    else:
        ach = args.steps * 2.0 * N * d * d / sec / 1e12  # useful flops of Y = X·Πᵀ
        peak = bf16 / 3.0  # fp32-accurate products: three fp16 tensor passes (hi·hi, lo·hi, hi·lo)
        roof = {"bound": "tensor", "achieved": round(ach, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": traffic(root, f"encode_dense_d{d}_n{N // 1000}k"),
                "kernel": "encode_umma_kernel",
                "peak_kind": f"{kind} bf16 dense / 3 split passes (fp16 hi/lo, same tensor rate as bf16)",
                "passes": 3, "flops_per_vector": 2 * d * d,
                "timed": "whole tq_encode call (row_norm_kernel + encode_umma_kernel)",
                "traffic_of": "encode_umma_kernel alone"}
    # kernels per tq_encode call: the Hadamard kernel alone, or the norm pass and
    # the tensor-core kernel (d > 128, a multiple of 128), or one dense kernel
    launches = 2 if rot == "dense" and d > 128 and d % 128 == 0 else 1
    # end to end: rows from pinned host memory, codes and norms back, per call
    e2e = None
    if N * d * 4 <= (2 << 30):
        xh = x.cpu().pin_memory()
        ch = torch.empty_like(cs.codes, device="cpu").pin_memory()
        nh = torch.empty_like(cs.norm, device="cpu").pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, min(args.steps, 10))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                x.copy_(xh, non_blocking=True)
                tq.tq_encode(ctx, x, cs, stream=stream)
                ch.copy_(cs.codes, non_blocking=True)
                nh.copy_(cs.norm, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        e2e = {"value": round(world * reps * N / (e0.elapsed_time(e1) * 1e-3) / 1e6, 3), "unit": "Mvec/s",
               "h2d_bytes_per_step": N * d * 4, "d2h_bytes_per_step": cs.codes.numel() * 4 + cs.norm.numel() * 4}
    line = _line(args, world, "encode Mvec/s", round(mvec, 3), "Mvec/s", total_ms / args.steps,
                 "f32 in, u4 codes, f16 hi/lo tensor products, f32 accumulate",
                 "synthetic (device-generated N(0,1) fp32 rows, a seeded 1% x50)",
                 {"workload": f"bulk indexing encode, TurboQuant_MSE b=4, d={d}, N={N}, {rot} rotation",
                  "d": d, "rows": N, "bits": bits, "rotation": rot,
                  "timing": "CUDA graph of one call, replayed per step", "l2": f"inputs larger than L2: {N * d * 4 / 1e9:.2f} GB of rows per step"},
                 roof, e2e, args.steps * launches, clk)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu["encode"](d, bits, rot, rotm)
    return line if rank == 0 else None


# ---------------------------------------------------------------- d = 128 encode (prefill, Prod keys)
def run_prefill(args, world, rank, local, root, clocks_cls, cpu):
    """The d = 128 encoder on its two large workloads: one layer's prefill at
    the long-context shape (K and V of 8 KV heads x 131072 tokens, fp16, b = 3,
    K in TOKEN and V in PAIR layout) and the Prod encode of 1M unit-norm fp32
    keys (b = 3: 2-bit MSE + 1-bit QJL).  value = the prefill's Mvec/s."""
    import torch

    import kv_cache_vector_tq_gb300 as tq
    from kv_cache_vector_tq_gb300 import synth
    torch.cuda.set_device(local)
    d, HKV, SEQ = 128, 8, 131072
    hbm, bf16, kind = _peaks(root)
    stream = torch.cuda.Stream()
    gen = torch.Generator(device="cuda").manual_seed(77 + rank)
    # ---- prefill: K (TOKEN) and V (PAIR), fp16 rows
    ctx = tq.Context(d, 3, tq.TQ_MSE, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(synth.gaussian_matrix(0, d)))
    kv = torch.randn((2, HKV * SEQ, d), generator=gen, device="cuda")
    kv[:, :, :4] *= 10.0
    kv = kv.half()
    K = tq.CodeSet(ctx, HKV * SEQ, tq.TQ_LAYOUT_TOKEN)
    V = tq.CodeSet(ctx, HKV * SEQ, tq.TQ_LAYOUT_PAIR)

    def prefill():
        tq.tq_encode(ctx, kv[0], K, 0, SEQ, SEQ, stream=stream)
        tq.tq_encode(ctx, kv[1], V, 0, SEQ, SEQ, stream=stream)

    total_ms, clk = _timed(prefill, args.steps, args.warmup, stream, clocks_cls, local, graph=True)
    assert ctx.poll() == tq.TQ_OK
    nvec = 2 * HKV * SEQ
    sec = total_ms * 1e-3
    mvec = world * args.steps * nvec / sec / 1e6
    bpv = 2 * d + 3 * d // 8 + 4                 # fp16 row in, 3-bit codes and the norm out
    fpv = 2 * 2 * d * d                          # two fp16 passes (x exact, Π hi + lo)
    t_hbm, t_tc = bpv / (hbm * 1e9), fpv / (bf16 * 1e12)
    ach_gbs = args.steps * nvec * bpv / sec / 1e9
    roof = {"bound": "hbm" if t_hbm >= t_tc else "tensor", "achieved": round(ach_gbs, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(max(t_hbm, t_tc) * nvec * args.steps / sec, 4),
            "traffic": traffic(root, "encode128_prefill_b3"), "kernel": "encode128_kernel<3,0,1> (K then V)",
            "peak_kind": kind, "bytes_per_vector": bpv, "tensor_flops_per_vector": fpv, "passes": 2,
            "roofline_rule": "max(bytes / HBM peak, issued fp16 flops / bf16 dense peak)"}
    del kv
    # ---- Prod encode of 1M unit-norm fp32 keys (the Prod-scores workload's setup)
    pctx = tq.Context(d, 3, tq.TQ_PROD, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(synth.gaussian_matrix(0, d)),
                      synth.qjl_matrix(0, d))
    NK = 1 << 20
    keys = torch.randn((NK, d), generator=gen, device="cuda")
    keys /= keys.norm(dim=1, keepdim=True)
    cs = tq.CodeSet(pctx, NK, tq.TQ_LAYOUT_TOKEN)
    pms, _ = _timed(lambda: tq.tq_encode(pctx, keys, cs, stream=stream), args.steps, args.warmup, stream,
                    clocks_cls, local, graph=True)
    assert pctx.poll() == tq.TQ_OK
    psec = pms * 1e-3
    pbpv = 4 * d + 2 * d // 8 + d // 8 + 8       # fp32 row in; 2-bit codes, sign words, s and γ out
    pfpv = 6 * 2 * d * d                         # three split passes for Π·u and three for (S·Πᵀ)·r
    pt_hbm, pt_tc = pbpv / (hbm * 1e9), pfpv / (bf16 * 1e12)
    prod = {"workload": "TurboQuant_Prod b=3 encode, d=128, 1M unit-norm fp32 keys",
            "value": round(world * args.steps * NK / psec / 1e6, 2), "unit": "Mvec/s",
            "ms_per_call": round(pms / args.steps, 4),
            "roofline": {"bound": "hbm" if pt_hbm >= pt_tc else "tensor",
                         "frac": round(max(pt_hbm, pt_tc) * NK * args.steps / psec, 4),
                         "achieved_tflops": round(args.steps * NK * pfpv / psec / 1e12, 1), "peak_tflops": bf16,
                         "kernel": "encode128_kernel<2,1,0>", "passes": 6, "tensor_flops_per_vector": pfpv,
                         "bytes_per_vector": pbpv}}
    line = _line(args, world, "encode Mvec/s", round(mvec, 2), "Mvec/s", total_ms / args.steps,
                 "f16 in, u3 codes, f16 tensor products (x exact, Π hi + lo), f32 accumulate",
                 "synthetic (device-generated N(0,1) fp16 K/V, channels 0-3 x10; unit-norm Gaussian keys)",
                 {"workload": "prefill encode of one long-context layer: K and V of 8 KV heads x 131072 tokens, "
                              "d=128, TurboQuant_MSE b=3 (K TOKEN, V PAIR layout)",
                  "vectors": nvec, "timing": "CUDA graph of one call, replayed per step", "l2": f"inputs larger than L2: {nvec * 2 * d / 1e9:.2f} GB of rows per call",
                  "prod_encode": prod},
                 roof, None, args.steps * 2, clk)
    return line if rank == 0 else None


# ---------------------------------------------------------------- Prod scores
def run_scores(args, world, rank, local, root, clocks_cls, cpu):
    import numpy as np
    import torch

    import kv_cache_vector_tq_gb300 as tq
    from kv_cache_vector_tq_gb300 import synth
    torch.cuda.set_device(local)
    d, N, M = 128, 1 << 20, 64
    G, S = synth.gaussian_matrix(0, d), synth.qjl_matrix(0, d)
    ctx = tq.Context(d, 3, tq.TQ_PROD, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(G), S)
    gen = torch.Generator(device="cuda").manual_seed(99 + rank)
    keys = torch.randn((N, d), generator=gen, device="cuda")
    keys /= keys.norm(dim=1, keepdim=True)
    cs = tq.CodeSet(ctx, N, tq.TQ_LAYOUT_TOKEN)
    tq.tq_encode(ctx, keys, cs)
    torch.cuda.synchronize()
    del keys
    q = torch.from_numpy(synth.queries(0, M, d)).cuda()
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(tq.tq_scores_workspace_size(ctx, M) // 4, 4), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    total_ms, clk = _timed(lambda: tq.tq_scores(ctx, q, cs, out, ws, stream=stream), args.steps, args.warmup,
                           stream, clocks_cls, local, graph=True)
    assert ctx.poll() == tq.TQ_OK
    sec = total_ms * 1e-3
    pairs = world * args.steps * M * N / sec
    hbm, _, kind = _peaks(root)
    bytes_call = N * (32 + 16 + 4 + 4) + M * N * 4
    ach = args.steps * bytes_call / sec / 1e9
    roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
            "traffic": traffic(root, "scores_prod_b3"), "kernel": "scores_kernel (Prod)", "peak_kind": kind, "bytes_per_call": bytes_call}
    qh = q.cpu().pin_memory()
    oh = torch.empty((M, N), dtype=torch.float32).pin_memory()
    reps = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            q.copy_(qh, non_blocking=True)
            tq.tq_scores(ctx, q, cs, out, ws, stream=stream)
            oh.copy_(out, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e = {"value": round(world * reps * M * N / (e0.elapsed_time(e1) * 1e-3), 1), "unit": "tokens scored/s",
           "h2d_bytes_per_step": M * d * 4, "d2h_bytes_per_step": M * N * 4}
    line = _line(args, world, "tokens scored/s", round(pairs, 1), "tokens scored/s", total_ms / args.steps,
                 "u2 codes + 1-bit QJL, f16 operands, f32 accumulate",
                 "synthetic (device-generated unit-norm Gaussian keys; seeded N(0,1) queries and S)",
                 {"workload": "TurboQuant_Prod b=3 scores, d=128, 1M keys x 64 queries", "keys": N, "queries": M,
                  "timing": "CUDA graph of one call, replayed per step", "l2": f"inputs larger than L2: {bytes_call / 1e6:.0f} MB moved per call"},
                 roof, e2e, args.steps, clk)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu["scores"](tq, cs, q, G, S)
    return line if rank == 0 else None


# ---------------------------------------------------------------- long context
def run_longctx(args, world, rank, local, root, clocks_cls, cpu):
    import numpy as np
    import torch

    import kv_cache_vector_tq_gb300 as tq
    from kv_cache_vector_tq_gb300 import synth
    torch.cuda.set_device(local)
    D, B, HQ, HKV, SEQ, L, bits = 128, 1, 64, 8, 131072, args.layers, 3
    ctx = tq.Context(D, bits, tq.TQ_MSE, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(synth.gaussian_matrix(0, D)))
    cap = SEQ
    gen = torch.Generator(device="cuda").manual_seed(4321 + rank)
    layers = []
    stream = torch.cuda.Stream()
    enc_ms = 0.0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for layer in range(L):
        K = tq.CodeSet(ctx, B * HKV * cap, tq.TQ_LAYOUT_TOKEN)
        V = tq.CodeSet(ctx, B * HKV * cap, tq.TQ_LAYOUT_PAIR)
        kv = torch.randn((2, B * HKV * SEQ, D), generator=gen, device="cuda", dtype=torch.float32)
        kv[:, :, :4] *= 10.0
        kv = kv.half()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):  # prefill: all but the last token of every (batch, KV head)
            e0.record(stream)
            tq.tq_encode(ctx, kv[0], K, 0, SEQ, cap, stream=stream)
            tq.tq_encode(ctx, kv[1], V, 0, SEQ, cap, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        enc_ms += e0.elapsed_time(e1)
        knew = kv[0].view(B * HKV, SEQ, D)[:, SEQ - 1].contiguous()
        vnew = kv[1].view(B * HKV, SEQ, D)[:, SEQ - 1].contiguous()
        del kv
        layers.append((K, V, knew, vnew))
    q = torch.randn((L, B, HQ, D), generator=gen, device="cuda").half()
    out = torch.empty((L, B, HQ, D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(ctx, B, HQ, HKV, SEQ) // 4 + 64, dtype=torch.float32,
                     device="cuda")
    scale = 1.0 / math.sqrt(D)

    def step():
        for i, (K, V, knew, vnew) in enumerate(layers):
            tq.tq_decode_step(ctx, ctx, q[i], knew, vnew, K, V, B, HQ, HKV, SEQ, cap, scale, out[i], ws,
                              stream=stream)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    total_ms, clk = _timed(g.replay, args.steps, args.warmup, stream, clocks_cls, local)
    assert ctx.poll() == tq.TQ_OK
    sec = total_ms * 1e-3
    per_layer = B * HKV * SEQ * 2 * (D * bits // 8 + 4)
    step_bytes = L * (per_layer + B * HQ * D * 6 + 2 * B * HKV * (D * 2 + D * bits // 8 + 4))
    gbs = world * args.steps * step_bytes / sec / 1e9
    hbm, _, kind = _peaks(root)
    enc_vecs = L * 2 * B * HKV * SEQ
    line = _line(args, world, "decode-attn HBM GB/s", round(gbs, 2), "GB/s", total_ms / args.steps,
                 "u3 codes, f16 operands, f32 accumulate",
                 "synthetic (device-generated N(0,1) fp16 K/V, channels 0-3 x10; N(0,1) queries)",
                 {"workload": f"long-context decode, {L} layers in sequence, batch 1, 64 q / 8 kv heads, "
                              f"head_dim 128, seq 131072, K/V TurboQuant_MSE b=3; step = append + attend per layer",
                  "layers": L, "seq": SEQ, "heads_q": HQ, "heads_kv": HKV, "bits": bits,
                  "resident_cache_gb": round(L * per_layer / 1e9, 2),
                  "l2": f"inputs larger than L2: {L * per_layer / 1e9:.1f} GB of caches per step",
                  "prefill_encode_mvec_s": round(enc_vecs / (enc_ms * 1e-3) / 1e6, 2),
                  "prefill_encode_gbs": round(enc_vecs * (D * 2 + D * bits // 8 + 4) / (enc_ms * 1e-3) / 1e9, 1),
                  "ms_per_layer": round(total_ms / args.steps / L, 4)},
                 {"bound": "hbm", "achieved": round(gbs / world, 1), "peak": hbm, "unit": "GB/s",
                  "frac": round(gbs / world / hbm, 4), "traffic": traffic(root, "longctx_b3"),
                  "kernel": "decode_step_kernel<3,3,8,8>",
                  "peak_kind": kind, "bytes_per_step": step_bytes},
                 None, args.steps * L, clk)
    return line if rank == 0 else None


# ---------------------------------------------------------------- keys (encode + one query)
def run_keys(args, world, rank, local, root, clocks_cls, cpu):
    import numpy as np
    import torch

    import kv_cache_vector_tq_gb300 as tq
    from kv_cache_vector_tq_gb300 import synth
    torch.cuda.set_device(local)
    d, N, b = 128, 4096, 3
    ctx = tq.Context(d, b, tq.TQ_MSE, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(synth.gaussian_matrix(0, d)))
    x = torch.from_numpy(synth.gaussian_rows(0, N, d, outlier_cols=4, outlier_scale=20.0)).cuda()
    q = torch.from_numpy(synth.queries(0, 1, d)).cuda()
    cs = tq.CodeSet(ctx, N, tq.TQ_LAYOUT_TOKEN)
    out = torch.empty((1, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(tq.tq_scores_workspace_size(ctx, 1) // 4, 4), dtype=torch.float32, device="cuda")
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def call():
        tq.tq_encode(ctx, x, cs, stream=stream)
        tq.tq_scores(ctx, q, cs, out, ws, stream=stream)

    total_ms, clk = _timed(call, args.steps, args.warmup, stream, clocks_cls, local, flush=flush_buf.zero_,
                           graph=True)
    assert ctx.poll() == tq.TQ_OK
    sec = total_ms * 1e-3
    mvec = world * args.steps * N / sec / 1e6
    hbm, _, kind = _peaks(root)
    byts = N * (4 * d + 48 + 4) + N * (48 + 4) + N * 4
    ach = args.steps * byts / sec / 1e9
    line = _line(args, world, "encode Mvec/s", round(mvec, 3), "Mvec/s", total_ms / args.steps,
                 "f32 in, u3 codes, f16 hi/lo tensor products, f32 accumulate",
                 "synthetic (seeded N(0,1) fp32 keys, channels 0-3 x20; N(0,1) query)",
                 {"workload": "TurboQuant_MSE b=3, d=128: encode 4096 keys, then score 1 query against them",
                  "keys": N, "timing": "CUDA graph of one encode + score, replayed per step",
                  "l2": "L2 flushed (256 MB write) before every timed call",
                  "us_per_encode_plus_score": round(total_ms / args.steps * 1e3, 2)},
                 {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                  "traffic": None, "kernel": "encode128_kernel + scores_kernel (latency-bound at this size)",
                  "peak_kind": kind},
                 None, 2 * args.steps, clk)
    return line if rank == 0 else None


# ---------------------------------------------------------------- b + 1/2 bits per coordinate
def run_mixed(args, world, rank, local, root, clocks_cls, cpu):
    """One decode layer (batch 1, 32 q / 8 kv heads, head_dim 128, seq 16384)
    with K and V at b + 1/2 bits per coordinate (b = --bits when 1..3, else 2:
    2.5 bits).  A step appends the new token's K and V with tq_encode and
    attends with tq_decode_attention (three launches), on each of R replica
    caches larger than L2 together.  The roofline unit is the attention call;
    the same line reports the encoder at that width on 1M fp16 rows."""
    import numpy as np
    import torch

    import kv_cache_vector_tq_gb300 as tq
    from kv_cache_vector_tq_gb300 import synth
    torch.cuda.set_device(local)
    b = args.bits if args.bits in (1, 2, 3) else 2
    D, B, HQ, HKV, SEQ = 128, 1, 32, 8, 16384
    kctx = tq.Context(D, b, tq.TQ_MIXED, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(synth.gaussian_matrix(0, D)))
    vctx = tq.Context(D, b, tq.TQ_MIXED, tq.TQ_ROT_DENSE, tq.tq_rotation_haar(synth.gaussian_matrix(1, D)))
    cap = SEQ
    Kh, Vh = synth.kv_layer(0, 0, B, HKV, SEQ, D)
    K0 = tq.CodeSet(kctx, B * HKV * cap, tq.TQ_LAYOUT_TOKEN)
    V0 = tq.CodeSet(vctx, B * HKV * cap, tq.TQ_LAYOUT_PAIR)
    tq.tq_encode(kctx, torch.from_numpy(np.ascontiguousarray(Kh[:, :, :SEQ - 1].reshape(-1, D))).cuda(), K0, 0,
                 SEQ - 1, cap)
    tq.tq_encode(vctx, torch.from_numpy(np.ascontiguousarray(Vh[:, :, :SEQ - 1].reshape(-1, D))).cuda(), V0, 0,
                 SEQ - 1, cap)
    vec_bytes = K0.words_per_vec * 4 + 4  # codes + fp32 norm
    cache_bytes = B * HKV * SEQ * 2 * vec_bytes
    R = max(2, int(math.ceil(4 * 129 * 1024 * 1024 / cache_bytes)))
    reps = [(K0, V0)]
    for _ in range(R - 1):
        Kr, Vr = tq.CodeSet(kctx, B * HKV * cap, tq.TQ_LAYOUT_TOKEN), tq.CodeSet(vctx, B * HKV * cap, tq.TQ_LAYOUT_PAIR)
        Kr.codes.copy_(K0.codes), Kr.norm.copy_(K0.norm), Vr.codes.copy_(V0.codes), Vr.norm.copy_(V0.norm)
        reps.append((Kr, Vr))
    knew = torch.from_numpy(np.ascontiguousarray(Kh[:, :, SEQ - 1].reshape(-1, D))).cuda()
    vnew = torch.from_numpy(np.ascontiguousarray(Vh[:, :, SEQ - 1].reshape(-1, D))).cuda()
    q = torch.from_numpy(synth.queries(0, B * HQ, D).reshape(B, HQ, D)).to(torch.float16).cuda()
    out = torch.empty((B, HQ, D), dtype=torch.float32, device="cuda")
    ws = torch.zeros(tq.tq_decode_workspace_size(kctx, B, HQ, HKV, SEQ) // 4 + 64, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    stream = torch.cuda.Stream()

    def step(r, append=True):
        K, V = reps[r]
        if append:
            tq.tq_encode(kctx, knew, K, SEQ - 1, 1, cap)
            tq.tq_encode(vctx, vnew, V, SEQ - 1, 1, cap)
        tq.tq_decode_attention(kctx, vctx, q, K, V, B, HQ, HKV, SEQ, cap, scale, out, ws)

    with torch.cuda.stream(stream):
        for r in range(R):
            step(r)
    torch.cuda.synchronize()
    g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        for r in range(R):
            step(r)
    with torch.cuda.graph(g_attn, stream=stream):
        for r in range(R):
            step(r, append=False)
    torch.cuda.synchronize()
    total_ms, clk = _timed(g_step.replay, args.steps, args.warmup, stream, clocks_cls, local)
    assert kctx.poll() == tq.TQ_OK and vctx.poll() == tq.TQ_OK
    attn_bytes = cache_bytes + q.numel() * 2 + out.numel() * 4
    step_bytes = attn_bytes + 2 * B * HKV * (D * 2 + vec_bytes)  # + the appended rows in, their codes out
    value = world * args.steps * R * step_bytes / (total_ms * 1e-3) / 1e9
    reps_attn = max(5, min(200, args.steps))
    attn_ms, _ = _timed(g_attn.replay, reps_attn, 1, stream, clocks_cls, local)
    attn_us = attn_ms * 1e3 / (reps_attn * R)
    hbm, _, kind = _peaks(root)
    ach = attn_bytes / (attn_us * 1e-6) / 1e9
    # end to end: q and the new K/V rows from pinned host memory, the output back, per step
    q_h, kn_h, vn_h = q.cpu().pin_memory(), knew.cpu().pin_memory(), vnew.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 50))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            for r in range(R):
                q.copy_(q_h, non_blocking=True)
                knew.copy_(kn_h, non_blocking=True)
                vnew.copy_(vn_h, non_blocking=True)
                step(r)
                out_h.copy_(out, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e = {"value": round(world * e2e_steps * R * step_bytes / (e0.elapsed_time(e1) * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": R * (q.numel() + knew.numel() + vnew.numel()) * 2,
           "d2h_bytes_per_step": R * out.numel() * 4}
    # the encoder at this width: 1M fp16 rows (2 KV heads' worth of the same recipe, tiled)
    N = 1 << 20
    X = torch.from_numpy(np.ascontiguousarray(Kh.reshape(-1, D))).cuda().repeat(N // (HKV * SEQ), 1)
    cs = tq.CodeSet(kctx, N, tq.TQ_LAYOUT_TOKEN)
    enc_ms, _ = _timed(lambda: tq.tq_encode(kctx, X, cs), 10, 3, stream, clocks_cls, local)
    enc_mvec = 10 * N / (enc_ms * 1e-3) / 1e6
    enc_bpv = D * 2 + vec_bytes
    assert kctx.poll() == tq.TQ_OK
    line = _line(args, world, "decode-attn HBM GB/s", round(value, 2), "GB/s", total_ms / args.steps,
                 f"u{b}/u{b + 1} codes (b + 1/2 bits), f16 operands, f32 accumulate",
                 "synthetic (seeded N(0,1) fp16 K/V with 4 outlier channels x10)",
                 {"workload": f"decode attention at {b}.5 bits per coordinate (TurboQuant_mse, coordinates j mod 16 < 8 "
                              f"at {b + 1} bits), 1 layer, batch 1, 32 q / 8 kv heads, head_dim 128, seq 16384; step = "
                              f"append 1 token (tq_encode K and V) + attend, on each of {R} replica caches",
                  "bits": b + 0.5, "replicas": R, "bytes_per_vector": vec_bytes, "bytes_per_step": step_bytes,
                  "l2": f"inputs larger than L2: {R} distinct caches x {cache_bytes / 1e6:.1f} MB per step",
                  "encode_mvec_s": round(enc_mvec, 1),
                  "encode_roofline": {"bound": "hbm", "achieved": round(enc_mvec * 1e6 * enc_bpv / 1e9, 1),
                                      "peak": hbm, "unit": "GB/s",
                                      "frac": round(enc_mvec * 1e6 * enc_bpv / 1e9 / hbm, 4),
                                      "kernel": "encode128_kernel", "bytes_per_vector": enc_bpv,
                                      "rows": f"{N} fp16 rows"}},
                 {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                  "traffic": traffic(root, f"decode_mixed_b{b}"), "kernel": "decode_step_kernel (b + 1/2 bits)",
                  "peak_kind": kind, "us_per_call": round(attn_us, 3), "bytes_per_call": attn_bytes},
                 e2e, args.steps * R * 3, clk)
    if rank == 0 and not args.no_cpu_baseline and "mixed" in cpu:
        line["cpu_baseline"] = cpu["mixed"](tq, reps[0], b, cap, q)
    return line if rank == 0 else None
