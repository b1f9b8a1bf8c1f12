#!/usr/bin/env python
"""Benchmark of the Dual-AR frame decode on one GB300 (or N replicas).

One step = one pass of the whole hot path over the workload's synthetic
input: radix cache cleared, every sequence released and prefilled again, then
n greedy frames decoded for the batch.  Default workload: the full-size S2
model (random-init bf16 weights, 36 + 4 layers, d = 2560), batch 1, 41-token
prompt, 60 frames.  Metric: frames/s (whole job) and ms/frame.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the machine's host cores instead (bounded sample, same metric).

Multi-GPU: sequences are independent, so N GPUs run N replicas of the
workload (weak scaling, no collective on the data path); the barrier and the
max-over-ranks time use torch.distributed.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

NCORES = len(os.sched_getaffinity(0))
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(NCORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "frames/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def bytes_per_frame(cfg, ctx_tokens_avg, batch, kv_bytes=4):
    """Algorithmic HBM bytes of one decode frame for the whole batch: every
    weight of the slow stack, the semantic head slice and 9 Fast AR passes
    (4 layers + one head slice each) read once, plus each sequence's KV
    (``kv_bytes`` per element: 4 for the default fp32 cache, 2 for bf16)."""
    from s2_inputs import param_counts
    c = param_counts(cfg)
    w = 2 * (c["slow_layers"] + c["sem_head_slice"] + 9 * (c["fast_layers"] + c["fast_head_slice"]))
    kv_per_tok = cfg.n_slow * 2 * cfg.n_kv * cfg.head_dim * kv_bytes
    return w + batch * kv_per_tok * ctx_tokens_avg, w


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- ranks

def max_over_ranks(x, world, device):
    """Max of a per-rank scalar over all ranks (the slowest rank's time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64 if device == "cpu" else torch.float32,
                     device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, max_seconds):
    """Throughput of the whole job: every rank's units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from s2_inputs import ensure_weights, make_workload, param_counts
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            dist.barrier()

    wl = make_workload(args.workload, n_frames=args.frames)
    if rank == 0:
        from serving_dual_ar_gb300 import buildlib
        buildlib.build()
        path = ensure_weights(wl.model)
    barrier()
    path = ensure_weights(wl.model) if rank != 0 else path
    from serving_dual_ar_gb300 import binding as b

    cfg = wl.model
    B, n = wl.batch, wl.n_frames
    T_max = max(p.T for p in wl.prompts)
    stream = torch.cuda.Stream()          # the library enqueues all work on this stream
    torch.cuda.set_stream(stream)
    ctx = b.s2_create(path, max_seqs=B, max_batch=B, kv_pool_pages=wl.pool_pages,
                      max_ctx=T_max + n + 16, max_prompt=T_max,
                      page_perm_seed=wl.page_perm_seed or 0, stream=stream,
                      flags=(b.S2_FLAG_INT8 if args.int8 else 0) |
                            (b.S2_FLAG_KV_BF16 if args.kv_bf16 else 0) |
                            (b.S2_FLAG_PERSIST if args.persist else 0))
    radix = wl.shared_prefix > 0
    dev_in = [(torch.from_numpy(p.tokens).cuda(), torch.from_numpy(p.codes).cuda(),
               torch.from_numpy(p.mask).cuda()) for p in wl.prompts]
    pin_in = [(torch.from_numpy(p.tokens).pin_memory(), torch.from_numpy(p.codes).pin_memory(),
               torch.from_numpy(p.mask).pin_memory()) for p in wl.prompts]
    seqs = np.arange(B, dtype=np.int32)
    out_dev = torch.zeros((B, n, 10), dtype=torch.int32, device="cuda")
    out_pin = torch.zeros((B, n, 10), dtype=torch.int32).pin_memory()
    live = [False]

    def step(inputs, out):
        b.s2_radix_clear(ctx)
        if live[0]:
            for i in range(B):
                b.s2_release(ctx, i)
        cached = 0
        for i, (t, c, m) in enumerate(inputs):
            masked = bool(wl.prompts[i].mask.any())
            cached += b.s2_prefill(ctx, i, t, c if masked else None, m if masked else None)
        live[0] = True
        b.s2_decode_frames(ctx, seqs, n, out=out)
        return cached

    for _ in range(args.warmup):
        step(dev_in, out_dev)
    torch.cuda.synchronize()
    clocks = Clocks(local_rank)
    barrier()
    torch.cuda.synchronize()
    l0 = b.s2_stats(ctx)["kernel_launches"]
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    cached = 0
    for _ in range(args.steps):
        cached = step(dev_in, out_dev)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    launches = b.s2_stats(ctx)["kernel_launches"] - l0
    ms_max = max_over_ranks(ms, world, "cuda")
    frames = B * n * args.steps * world
    value = whole_job_rate(B * n * args.steps, world, ms_max / 1000.0)

    # decode-only and prefill-only timing of one extra step (not the headline)
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    b.s2_radix_clear(ctx)
    for i in range(B):
        b.s2_release(ctx, i)
    e[0].record(stream)
    for i, (tk, c, m) in enumerate(dev_in):
        masked = bool(wl.prompts[i].mask.any())
        b.s2_prefill(ctx, i, tk, c if masked else None, m if masked else None)
    e[1].record(stream)
    b.s2_decode_frames(ctx, seqs, n, out=out_dev)
    e[2].record(stream)
    torch.cuda.synchronize()
    prefill_ms = e[0].elapsed_time(e[1])
    decode_ms = e[1].elapsed_time(e[2])

    # end to end through the public API with host (pinned) buffers
    torch.cuda.synchronize()
    barrier()
    h0 = time.perf_counter()
    for _ in range(args.steps):
        step(pin_in, out_pin.numpy())
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - h0
    e2e_value = whole_job_rate(B * n * args.steps, world, max_over_ranks(e2e_s, world, "cuda"))
    h2d = sum(p.tokens.nbytes + (p.codes.nbytes + p.mask.nbytes if p.mask.any() else 0)
              for p in wl.prompts)
    d2h = B * n * 10 * 4
    stats = b.s2_stats(ctx)
    b.s2_destroy(ctx)
    del dev_in, pin_in

    pk, pk_kind = peaks()
    ctx_avg = T_max + n / 2
    bpf, wbytes = bytes_per_frame(cfg, ctx_avg, B, kv_bytes=2 if args.kv_bf16 else 4)
    if args.int8:   # one byte per streamed weight (+ a 4-byte scale per row)
        bpf, wbytes = bpf - wbytes / 2, wbytes / 2
    decode_frames_s = n / (decode_ms / 1000.0)
    hbm_step = {
        "bytes_per_frame": bpf, "weight_bytes_per_frame": wbytes,
        "achieved_gbs": bpf * decode_frames_s / 1e9,
        "peak_gbs": pk["hbm_gbs"], "frac": bpf * decode_frames_s / 1e9 / pk["hbm_gbs"],
        "peak_kind": pk_kind, "nominal_frac_8tbs": bpf * decode_frames_s / 1e9 / 8000.0,
    }
    roof = gemv_roofline(b, torch, cfg, pk, pk_kind) if rank == 0 else None

    res = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "ms_per_frame": ms_max / (args.steps * n),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("int8-weights/fp32-accumulate" if args.int8 else
                  ("bf16" if cfg.wdtype == "bf16" else "f32")),
        "data": "synthetic (seeded random-init weights N(0,0.02), seeded random prompts)",
        "config": {"workload": wl.name, "batch": B, "prompt_tokens": T_max, "frames": n,
                   "model": f"dual-ar d={cfg.d} slow={cfg.n_slow} fast={cfg.n_fast}",
                   "radix_shared_prefix": wl.shared_prefix, "parallelism": f"replicas x{world}",
                   "kv_cache": "bf16" if args.kv_bf16 else "fp32",
                   "decode": "persistent" if args.persist else "cuda-graphs",
                   "l2": "weights (9.5 GB) >> L2 (129 MB): every step streams from HBM, no flush"},
        "decode_ms_per_frame": decode_ms / n, "prefill_ms": prefill_ms,
        "cached_prefix_tokens_per_step": cached,
        "hbm_step": hbm_step,
        "roofline": roof,
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "frames/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "device_error": stats["device_error"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, path)
    if world > 1:
        dist.destroy_process_group()
    return res


# DRAM bytes per launch of this version of the weight-stream kernel, the mean
# over the four projection shapes of one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), summarised in the profiles folder.  Set it to None
# whenever the kernel changes, until it has been captured again.
GEMV_TRAFFIC_PER_LAUNCH = 51.24e6


def gemv_roofline(b, torch, cfg, pk, pk_kind):
    """Dominant kernel: the weight-streaming GEMV.  Times it, with CUDA events
    on the stream it launches on, over the four projection shapes of all the
    slow layers (7.3 GB of weights, far beyond L2), and reports algorithmic
    bytes (weights + activations) per launch over the mean launch time."""
    d, F, qd, kvd = cfg.d, cfg.ffn, cfg.q_dim, cfg.kv_dim
    shapes = [(qd + 2 * kvd, d, 0, True), (d, qd, 1, False), (2 * F, d, 2, True), (d, F, 1, False)]
    L = cfg.n_slow
    mats = [[torch.randn((N, K), device="cuda", dtype=torch.bfloat16) * 0.02 for (N, K, _, _) in shapes]
            for _ in range(L)]
    xs = {K: torch.randn((1, K), device="cuda") for (_, K, _, _) in shapes}
    ys = {N: torch.zeros((1, N), device="cuda") for (N, _, _, _) in shapes}
    g = torch.ones(max(d, F), device="cuda")
    st = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def one_pass():
        for l in range(L):
            for (N, K, mode, norm), W in zip(shapes, mats[l]):
                out_cols = N // 2 if mode == 2 else N
                b.s2op_gemv(W, N, K, xs[K], K, 1, ys[N], out_cols, mode=mode,
                            gain=g if norm else None, stream=st)

    one_pass()
    torch.cuda.synchronize()
    reps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        one_pass()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    launches = reps * L * len(shapes)
    per_launch = sum(2 * N * K + 4 * K + 4 * N for (N, K, _, _) in shapes) * L / (L * len(shapes))
    achieved = per_launch * launches / (ms / 1000.0) / 1e9
    del mats
    torch.cuda.empty_cache()
    return {"kernel": "gemv_kernel<bf16,1> (K1 weight stream, batch 1)", "bound": "hbm",
            "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "peak_kind": f"{pk_kind} burst copy",
            "bytes_per_launch": per_launch, "us_per_launch": ms * 1000.0 / launches,
            "traffic": GEMV_TRAFFIC_PER_LAUNCH}


# ---------------------------------------------------------------- the oracle

def oracle_sample(wl, path, frames=2, w=None):
    """Time the oracle on one sequence: prefill, then ``frames`` frames.
    Returns (weights, prefill_s, per_frame_s)."""
    import oracle
    if w is None:
        w = oracle.OracleWeights(path, dtype=np.float32)
    p = wl.prompts[0]
    o = oracle.DualAROracle(w, paged=True, pool_pages=-(-(p.T + frames + 16) // 16) + 4, radix=False)
    t0 = time.perf_counter()
    o.prefill(0, p.tokens, p.codes, p.mask)
    t1 = time.perf_counter()
    o.decode_frames([0], frames)
    t2 = time.perf_counter()
    return w, t1 - t0, (t2 - t1) / frames


def cpu_baseline(wl, path):
    w, tp, tf = oracle_sample(wl, path, frames=2)
    n = wl.n_frames
    # one sequence's prefill + n frames, projected from the sample; batch
    # members are independent, so the batch costs B times that on the oracle
    per_seq = tp + n * tf
    value = wl.batch * n / (wl.batch * per_seq)
    return {"value": value, "unit": "frames/s", "cores": NCORES, "kind": "oracle",
            "sample": f"sequence 0: prefill ({wl.prompts[0].T} tokens, {tp:.2f} s) + 2 of {n} frames "
                      f"({tf:.2f} s/frame), fp32 NumPy; projected to the workload"}


def run_reference(args):
    """The oracle as the reference arm: same workload, metric and unit, each
    step a bounded sample (prefill + 1 frame of sequence 0) projected to the
    workload's frames."""
    from s2_inputs import ensure_weights, make_workload
    wl = make_workload(args.workload)
    path = ensure_weights(wl.model)
    w = None
    for _ in range(args.warmup):
        w, _, _ = oracle_sample(wl, path, frames=1, w=w)
    tps, tfs = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        w, tp, tf = oracle_sample(wl, path, frames=1, w=w)
        tps.append(tp)
        tfs.append(tf)
    wall = time.perf_counter() - t0
    n = wl.n_frames
    per_seq = statistics.mean(tps) + n * statistics.mean(tfs)
    value = n / per_seq
    return {"metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * wall / args.steps,
            "ms_per_frame": 1000.0 / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "frames": n},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "frames/s", "cores": NCORES, "kind": "oracle",
                             "sample": f"per step: prefill of sequence 0 + 1 frame; projected to "
                                       f"{n} frames per sequence"},
            "e2e": {"value": value, "unit": "frames/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_attn_kernel(args, b, torch, cfg):
    """Decode attention (K3+K4) on the S2 heads: ``--rows`` sequences, each
    with ``--ctx`` cached keys plus the new one, fp32 pages (``--kv-bf16``:
    bf16), one pool per layer of ``--layers``; the split count is the
    runtime's (CTAs for twice the SMs, at most 16 splits)."""
    B, ctx, L = args.rows, args.ctx, args.layers
    H, Hkv, hd = cfg.n_heads, cfg.n_kv, cfg.head_dim
    qd, kvd = H * hd, Hkv * hd
    P = 16
    ppseq = (ctx + 1 + P - 1) // P
    n_pages = B * ppseq
    kvsz = 2 if args.kv_bf16 else 4
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nsplit = max(1, min(16, (2 * sms + B * Hkv - 1) // (B * Hkv)))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    dt = torch.bfloat16 if args.kv_bf16 else torch.float32
    pools = [torch.randn((n_pages, 2, Hkv, P, hd), device="cuda", generator=gen).to(dt) for _ in range(L)]
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(7)).to(torch.int32)
    table = perm.reshape(B, ppseq).contiguous().cuda()
    pos = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
    qkv = torch.randn((B, qd + 2 * kvd), device="cuda", generator=gen)
    gain = torch.ones(hd, device="cuda")
    cs, sn = b.s2op_rope_table(ctx + 1, hd, cfg.rope_theta)
    cs, sn = torch.from_numpy(cs).cuda(), torch.from_numpy(sn).cuda()
    o = torch.zeros((B, qd), device="cuda")
    ws = torch.zeros(b.s2op_attn_decode_workspace_bytes(B, 1, H, Hkv, hd, nsplit), dtype=torch.uint8,
                     device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()

    def one():
        for l in range(L):
            b.s2op_attn_decode(qkv, qd + 2 * kvd, B, 1, H, Hkv, hd, gain, gain, cfg.eps, cs, sn, pos,
                               pools[l], int(args.kv_bf16), table, ppseq, o, qd, nsplit=nsplit,
                               workspace=ws, stream=st)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(args.steps):
        one()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    launches = args.steps * L
    # algorithmic bytes of one launch: the cached keys and values, the new row's
    # q/k/v in and its k/v appended, the output out
    per = B * ((ctx * 2 * kvd) * kvsz + (qd + 2 * kvd) * 4 + 2 * kvd * kvsz + qd * 4)
    pk, kind = peaks()
    gbs = per * launches / ms / 1e6
    print(json.dumps({"kernel": "attn", "rows": B, "ctx": ctx, "layers": L, "nsplit": nsplit,
                      "kv": "bf16" if args.kv_bf16 else "fp32", "launches": launches,
                      "us_per_launch": 1000 * ms / launches, "bytes_per_launch": per,
                      "gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"], "peak_kind": kind}), flush=True)


def run_kernel(args):
    """Microbenchmark of one kernel on the S2 shapes (for ncu captures and
    tuning): ``gemv`` streams the four projections of ``--layers`` layers at
    batch ``--rows``; ``tc`` runs the tcgen05 GEMM on the same matrices with
    ``--rows`` activation rows; ``attn`` runs the decode attention.  Weights
    total > L2; a few GB at most."""
    import torch
    from s2_inputs import S2
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding as b
    cfg = S2
    if args.kernel == "attn":
        run_attn_kernel(args, b, torch, cfg)
        return
    d, F, qd, kvd = cfg.d, cfg.ffn, cfg.q_dim, cfg.kv_dim
    shapes = [(qd + 2 * kvd, d, 0, True), (d, qd, 1, False), (2 * F, d, 2, True), (d, F, 1, False)]
    L, R = args.layers, args.rows
    mats = [[torch.randn((N, K), device="cuda", dtype=torch.bfloat16) * 0.02 for (N, K, _, _) in shapes]
            for _ in range(L)]
    st = torch.cuda.current_stream()
    xs = {K: torch.randn((R, K), device="cuda") for (_, K, _, _) in shapes}
    x16 = {K: torch.randn((R, K), device="cuda").to(torch.bfloat16) for (_, K, _, _) in shapes}
    ys = {N: torch.zeros((R, N), device="cuda") for (N, _, _, _) in shapes}
    y16 = torch.zeros((R, F), device="cuda", dtype=torch.bfloat16)
    g = torch.ones(max(d, F), device="cuda")
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    tk = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()

    def one():
        for l in range(L):
            for (N, K, mode, norm), W in zip(shapes, mats[l]):
                oc = N // 2 if mode == 2 else N
                if args.kernel == "gemv":
                    b.s2op_gemv(W, N, K, xs[K], K, R, ys[N], oc, mode=mode, gain=g if norm else None,
                                stream=st)
                else:
                    if mode == 2:
                        b.s2op_tc_gemm(W, N, K, x16[K], R, K, Y16=y16, ldy16=F, epi=2, workspace=ws,
                                       tickets=tk, stream=st)
                    else:
                        b.s2op_tc_gemm(W, N, K, x16[K], R, K, Y=ys[N], ldy=N, epi=mode, workspace=ws,
                                       tickets=tk, stream=st)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(args.steps):
        one()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    launches = args.steps * L * len(shapes)
    wbytes = sum(2 * N * K for (N, K, _, _) in shapes) * L * args.steps
    flops = sum(2 * N * K * R for (N, K, _, _) in shapes) * L * args.steps
    pk, kind = peaks()
    print(json.dumps({"kernel": args.kernel, "rows": R, "layers": L, "launches": launches,
                      "us_per_launch": 1000 * ms / launches, "weight_gbs": wbytes / ms / 1e6,
                      "frac_hbm": wbytes / ms / 1e6 / pk["hbm_gbs"], "tflops": flops / ms / 1e9,
                      "peak_kind": kind}), flush=True)


def run_calibration(args):
    """Read-bandwidth calibration on this GPU: torch reductions over the S2
    projection matrices and over one large tensor, and the GEMV on one large
    matrix (no per-launch ramp).  Prints one JSON line."""
    import torch
    from s2_inputs import S2
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding as b
    cfg = S2
    d, F, qd, kvd = cfg.d, cfg.ffn, cfg.q_dim, cfg.kv_dim
    shapes = [(qd + 2 * kvd, d), (d, qd), (2 * F, d), (d, F)]
    L = args.layers
    mats = [torch.randn((N, K), device="cuda", dtype=torch.bfloat16) for _ in range(L) for (N, K) in shapes]
    big = torch.randn((1 << 30,), device="cuda", dtype=torch.bfloat16)        # 2 GiB
    huge = torch.randn((131072, d), device="cuda", dtype=torch.bfloat16)      # 671 MB GEMV
    x = torch.randn((1, d), device="cuda")
    y = torch.zeros((1, 131072), device="cuda")
    out = {}

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps / 1000.0

    nbytes = sum(m.numel() * 2 for m in mats)
    t = timed(lambda: [m.sum(dtype=torch.float32) for m in mats])
    out["torch_sum_projections_gbs"] = nbytes / t / 1e9
    t = timed(lambda: big.sum(dtype=torch.float32))
    out["torch_sum_2GiB_gbs"] = big.numel() * 2 / t / 1e9
    t = timed(lambda: big.clone())
    out["torch_copy_2GiB_rw_gbs"] = 2 * big.numel() * 2 / t / 1e9
    t = timed(lambda: b.s2op_gemv(huge, 131072, d, x, d, 1, y, 131072))
    out["gemv_671MB_gbs"] = huge.numel() * 2 / t / 1e9
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=1, help="workload index 1..4 (default 1)")
    ap.add_argument("--frames", type=int, default=None,
                    help="frames per step instead of the workload's (for short profiling captures; "
                         "not a bench line of the workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--int8", action="store_true",
                    help="per-channel INT8 weights (reported separately; not the bf16 headline)")
    ap.add_argument("--kv-bf16", action="store_true",
                    help="bf16 Slow AR KV cache (default fp32)")
    ap.add_argument("--persist", action="store_true",
                    help="decode full frames in the persistent kernel instead of per-frame CUDA graphs")
    ap.add_argument("--kernel", choices=["gemv", "tc", "attn", "calib"], default=None,
                    help="microbenchmark one kernel on the S2 shapes instead of the workload")
    ap.add_argument("--rows", type=int, default=1)
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--ctx", type=int, default=100, help="--kernel attn: cached keys per sequence")
    args = ap.parse_args()
    if args.kernel == "calib":
        run_calibration(args)
        return
    if args.kernel:
        run_kernel(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
