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


def kv_bytes_per_token(cfg, kv_bytes=2):
    """KV of one context token of one sequence across the Slow AR layers."""
    return cfg.n_slow * 2 * cfg.n_kv * cfg.head_dim * kv_bytes


def bytes_per_frame(cfg, ctx_tokens_avg, batch, shared_prefix=0, kv_bytes=2):
    """Algorithmic HBM bytes of one steady decode step for the whole batch:
    every weight of the slow stack, the semantic head slice and 9 Fast AR
    passes (4 layers + one head slice each) read once; the KV of each
    sequence's context read once (a radix-shared prefix of ``shared_prefix``
    tokens is one set of pages, read once per step, not once per sequence)
    and one new token's KV written per sequence.  ``kv_bytes`` per element:
    2, the bf16 KV the method needs (the build's fp32 cache is a storage
    choice, not algorithmic bytes).  Returns (total, weight bytes)."""
    from s2_inputs import param_counts
    c = param_counts(cfg)
    w = 2 * (c["slow_layers"] + c["sem_head_slice"] + 9 * (c["fast_layers"] + c["fast_head_slice"]))
    if ctx_tokens_avg <= 0:
        return w, w
    per_tok = kv_bytes_per_token(cfg, kv_bytes)
    shared = min(shared_prefix, ctx_tokens_avg)
    kv_tokens = shared + batch * (ctx_tokens_avg - shared) + batch
    return w + per_tok * kv_tokens, w


def decode_call_bytes(cfg, T, n, batch, shared_prefix=0, kv_bytes=2):
    """Algorithmic bytes of one decode call of n frames after a T-token
    prompt: frame 0 comes from the prefill's last hidden (no slow step), so
    n - 1 slow steps, each reading the weights of the slow stack and the KV
    of T + f - 1 cached tokens per sequence (f = 1 .. n-1; the shared prefix
    once) and writing one token per sequence, plus n semantic heads and Fast
    AR loops.  Returns (total, weight bytes)."""
    from s2_inputs import param_counts
    c = param_counts(cfg)
    slow = 2 * c["slow_layers"]
    head_fast = 2 * (c["sem_head_slice"] + 9 * (c["fast_layers"] + c["fast_head_slice"]))
    per_tok = kv_bytes_per_token(cfg, kv_bytes)
    kv_tokens = 0
    for f in range(1, n):
        ctx = T + f - 1
        sh = min(shared_prefix, ctx)
        kv_tokens += sh + batch * (ctx - sh) + batch
    w = (n - 1) * slow + n * head_fast
    return w + per_tok * kv_tokens, w


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

def _flags(b, args):
    return ((b.S2_FLAG_INT8 if args.int8 else 0) | (b.S2_FLAG_KV_BF16 if args.kv_bf16 else 0) |
            (b.S2_FLAG_PERSIST if args.persist else 0) | (b.S2_FLAG_STREAM if args.stream else 0) |
            (b.S2_FLAG_NO_PREFIX_TC if args.no_prefix_tc else 0))


class WorkloadRunner:
    """One workload on one library context: the step (radix cleared, every
    sequence released and prefilled again, n frames decoded for the batch)
    with device-resident or pinned-host inputs."""

    def __init__(self, b, torch, path, wl, flags, stream):
        self.b, self.torch, self.wl, self.stream = b, torch, wl, stream
        B, n = wl.batch, wl.n_frames
        T_max = max(p.T for p in wl.prompts)
        # a batched prefill pass may hold every prompt's rows (at most 32,768)
        rows = min(sum(p.T for p in wl.prompts), 32768) if B > 1 else 0
        self.ctx = b.s2_create(path, max_seqs=B, max_batch=B, kv_pool_pages=wl.pool_pages,
                               max_ctx=T_max + n + 16, max_prompt=T_max,
                               page_perm_seed=wl.page_perm_seed or 0, stream=stream, flags=flags,
                               prefill_rows=max(rows, T_max))
        self.dev_in = [(torch.from_numpy(p.tokens).cuda(), torch.from_numpy(p.codes).cuda(),
                        torch.from_numpy(p.mask).cuda()) for p in wl.prompts]
        self.pin_in = [(torch.from_numpy(p.tokens).pin_memory(), torch.from_numpy(p.codes).pin_memory(),
                        torch.from_numpy(p.mask).pin_memory()) for p in wl.prompts]
        self.seqs = np.arange(B, dtype=np.int32)
        # several prompts: one s2_prefill_batch call over the concatenated prompts
        self.batched = B > 1
        if self.batched:
            masked = any(p.mask.any() for p in wl.prompts)
            cat = [np.concatenate([p.tokens for p in wl.prompts]).astype(np.int32),
                   np.concatenate([p.codes.reshape(-1) for p in wl.prompts]).astype(np.int32) if masked else None,
                   np.concatenate([p.mask for p in wl.prompts]).astype(np.uint8) if masked else None]
            self.lens = np.array([p.T for p in wl.prompts], np.int32)
            self.cached_out = np.zeros(B, np.int32)
            self.cat_dev = [torch.from_numpy(x).cuda() if x is not None else None for x in cat]
            self.cat_pin = [torch.from_numpy(x).pin_memory() if x is not None else None for x in cat]
        self.out_dev = torch.zeros((B, n, 10), dtype=torch.int32, device="cuda")
        self.out_pin = torch.zeros((B, n, 10), dtype=torch.int32).pin_memory()
        self.live = False

    def prefill_all(self, inputs):
        if self.batched:
            cat = self.cat_pin if inputs is self.pin_in else self.cat_dev
            b = self.b
            b._check(b.LIB.s2_prefill_batch(self.ctx, len(self.lens), b.ptr(self.seqs), b.ptr(cat[0]),
                                            b.ptr(self.lens), b.ptr(cat[1]), b.ptr(cat[2]),
                                            b.ptr(self.cached_out)), "s2_prefill_batch")
            return int(self.cached_out.sum())
        cached = 0
        for i, (t, c, m) in enumerate(inputs):
            masked = bool(self.wl.prompts[i].mask.any())
            cached += self.b.s2_prefill(self.ctx, i, t, c if masked else None, m if masked else None)
        return cached

    def reset(self):
        self.b.s2_radix_clear(self.ctx)
        if self.live:
            for i in range(self.wl.batch):
                self.b.s2_release(self.ctx, i)
        self.live = False

    def step(self, host=False):
        self.reset()
        cached = self.prefill_all(self.pin_in if host else self.dev_in)
        self.live = True
        self.b.s2_decode_frames(self.ctx, self.seqs, self.wl.n_frames,
                                out=self.out_pin.numpy() if host else self.out_dev)
        return cached

    def timed_steps(self, steps):
        """(ms over ``steps`` device-resident steps on the library's stream,
        launches, cached prefix tokens per step)."""
        torch, st = self.torch, self.stream
        l0 = self.b.s2_stats(self.ctx)["kernel_launches"]
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(st)
        cached = 0
        for _ in range(steps):
            cached = self.step()
        ev1.record(st)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1), self.b.s2_stats(self.ctx)["kernel_launches"] - l0, cached

    def split_step(self):
        """Prefill-only and decode-only times (ms) of one more step."""
        torch, st = self.torch, self.stream
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        self.reset()
        e[0].record(st)
        self.prefill_all(self.dev_in)
        self.live = True
        e[1].record(st)
        self.b.s2_decode_frames(self.ctx, self.seqs, self.wl.n_frames, out=self.out_dev)
        e[2].record(st)
        torch.cuda.synchronize()
        return e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])

    def close(self):
        self.b.s2_destroy(self.ctx)
        self.dev_in = self.pin_in = None


def hbm_record(cfg, wl, decode_ms, kv_storage_bytes, pk, pk_kind, int8=False):
    """The decode call against the HBM roofline: algorithmic bytes of the
    call (bf16 weights and KV, the shared prefix once) over its time."""
    T_max = max(p.T for p in wl.prompts)
    n = wl.n_frames
    shared = wl.shared_prefix // 16 * 16     # whole 16-token pages are shared
    total, wbytes = decode_call_bytes(cfg, T_max, n, wl.batch, shared, kv_bytes=2)
    if int8:   # one byte per streamed weight (the row scales are negligible)
        total, wbytes = total - wbytes / 2, wbytes / 2
    gbs = total / (decode_ms / 1000.0) / 1e9
    return {"bytes_per_call": total, "bytes_per_frame": total / n, "weight_bytes_per_call": wbytes,
            "kv_bytes_per_element": 2, "kv_cache_storage_bytes_per_element": kv_storage_bytes,
            "shared_prefix_tokens_counted_once": shared,
            "achieved_gbs": gbs, "peak_gbs": pk["hbm_gbs"], "frac": gbs / pk["hbm_gbs"],
            "peak_kind": pk_kind, "nominal_frac_8tbs": gbs / 8000.0}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from s2_inputs import ensure_weights, make_workload
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
    trace_file = None
    if args.frame_trace and rank == 0:
        import tempfile
        trace_file = os.path.join(tempfile.mkdtemp(), "frame_trace.txt")
        os.environ["S2_FRAME_TRACE"] = trace_file   # read by s2_create
    run = WorkloadRunner(b, torch, path, wl, _flags(b, args), stream)
    if trace_file:
        del os.environ["S2_FRAME_TRACE"]

    for _ in range(args.warmup):
        run.step()
    torch.cuda.synchronize()
    clocks = Clocks(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    ms, launches, cached = run.timed_steps(args.steps)
    barrier()
    clk = clocks.stop()
    ms_max = max_over_ranks(ms, world, "cuda")
    value = whole_job_rate(B * n * args.steps, world, ms_max / 1000.0)
    prefill_ms, decode_ms = run.split_step()

    # end to end through the public API with host (pinned) buffers
    torch.cuda.synchronize()
    barrier()
    h0 = time.perf_counter()
    for _ in range(args.steps):
        run.step(host=True)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - h0
    e2e_value = whole_job_rate(B * n * args.steps, world, max_over_ranks(e2e_s, world, "cuda"))
    h2d = sum(p.tokens.nbytes + (p.codes.nbytes + p.mask.nbytes if p.mask.any() else 0)
              for p in wl.prompts)
    d2h = B * n * 10 * 4
    stats = b.s2_stats(run.ctx)
    run.close()

    pk, pk_kind = peaks()
    hbm_step = hbm_record(cfg, wl, decode_ms, 2 if args.kv_bf16 else 4, pk, pk_kind, int8=args.int8)
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
                   "decode": ("persistent" if args.persist else
                              "streaming-kernel" if args.stream else "cuda-graphs"),
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
    if (rank == 0 and world == 1 and args.workload == 1 and args.frames is None
            and not args.no_batch32):
        res["batch32"] = run_batch32(args, b, torch, path, stream, local_rank, pk, pk_kind)
    if (rank == 0 and world == 1 and args.workload == 1 and args.frames is None
            and not args.no_vocoder):
        # the codec stage on the batch-32 workload's output volume (32 x 300 frames)
        voc = vocoder_record(b, torch, 32, 300, 3, 2, pk)
        voc.pop("launches")
        res["vocoder"] = voc
    if trace_file:
        res["frame_trace"] = frame_trace_summary(trace_file)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, path)
    if world > 1:
        dist.destroy_process_group()
    return res


def run_profile_decode(args):
    """One step of the workload for a profiler's launch list: every prompt
    prefilled, then one decode call inside an NVTX range named s2_decode
    (``ncu --nvtx --nvtx-include s2_decode/`` captures exactly its launches)."""
    import torch
    from s2_inputs import ensure_weights, make_workload
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding as b
    wl = make_workload(args.workload, n_frames=args.frames)
    path = ensure_weights(wl.model)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    run = WorkloadRunner(b, torch, path, wl, _flags(b, args), stream)
    run.step()                      # graphs captured, caches warm
    torch.cuda.synchronize()
    run.reset()
    run.prefill_all(run.dev_in)
    run.live = True
    torch.cuda.synchronize()
    l0 = b.s2_stats(run.ctx)["kernel_launches"]
    torch.cuda.nvtx.range_push("s2_decode")
    b.s2_decode_frames(run.ctx, run.seqs, wl.n_frames, out=run.out_dev)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    print(json.dumps({"workload": wl.name, "frames": wl.n_frames,
                      "decode_launches": b.s2_stats(run.ctx)["kernel_launches"] - l0}), flush=True)
    run.close()


def run_batch32(args, b, torch, path, stream, local_rank, pk, pk_kind):
    """The batch-32 workload (32 sequences sharing a radix-cached 900-position
    VQ prefix, 40-token private suffixes, 300 frames each) on the same
    model: 1 warm-up step and ``BATCH32_STEPS`` timed steps with CUDA events
    on the library's stream and clocks sampled during them."""
    from s2_inputs import make_workload
    wl = make_workload(3)
    run = WorkloadRunner(b, torch, path, wl, _flags(b, args), stream)
    run.step()
    torch.cuda.synchronize()
    clocks = Clocks(local_rank)
    clocks.start()
    ms, launches, cached = run.timed_steps(BATCH32_STEPS)
    clk = clocks.stop()
    prefill_ms, decode_ms = run.split_step()
    stats = b.s2_stats(run.ctx)
    run.close()
    frames = wl.batch * wl.n_frames
    return {"workload": wl.name, "batch": wl.batch, "frames_per_sequence": wl.n_frames,
            "steps": BATCH32_STEPS, "warmup": 1,
            "value": frames * BATCH32_STEPS / (ms / 1000.0), "unit": "frames/s",
            "ms_per_step": ms / BATCH32_STEPS, "ms_per_frame": ms / (BATCH32_STEPS * frames),
            "decode_ms_per_batch_frame": decode_ms / wl.n_frames,
            "decode_frames_per_s": frames / (decode_ms / 1000.0), "prefill_ms": prefill_ms,
            "cached_prefix_tokens_per_step": cached,
            "hbm_step": hbm_record(wl.model, wl, decode_ms, 2 if args.kv_bf16 else 4, pk, pk_kind,
                                   int8=args.int8),
            "clocks": clk, "gpu_launches": launches, "device_error": stats["device_error"]}


BATCH32_STEPS = 2


# DRAM bytes per launch of this version of the weight-stream kernel, the mean
# over the four projection shapes of one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), summarised in the profiles folder.  Set it to None
# whenever the kernel changes, until it has been captured again.
GEMV_TRAFFIC_PER_LAUNCH = 51.25e6


def gemv_roofline(b, torch, cfg, pk, pk_kind):
    """Dominant kernel: the weight-streaming GEMV.  Times it, with CUDA events
    on the stream it launches on, over the four projection shapes of all the
    slow layers (7.3 GB of weights, far beyond L2; the 144 launches captured
    once as a CUDA graph and replayed), and reports algorithmic bytes
    (weights + activations) per launch over the mean launch time."""
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
    # the 144 launches replayed as one CUDA graph (as the decode replays its
    # frame), so the host's per-call overhead does not sit between launches
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(st)
    with torch.cuda.stream(cap):
        st = cap
        with torch.cuda.graph(graph, stream=cap):
            one_pass()
    torch.cuda.synchronize()
    reps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        graph.replay()   # warm
        e0.record(cap)
        for _ in range(reps):
            graph.replay()
        e1.record(cap)
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

ORACLE_SAMPLE_FRAMES = 4


def oracle_sample(wl, path, w=None):
    """Time the oracle on sequence 0 of the workload: its prefill, its first
    frame (made from the prefill's last hidden: heads and Fast AR only) and
    ``ORACLE_SAMPLE_FRAMES`` - 1 steady frames (one slow step each).
    Returns (weights, prefill_s, first_frame_s, steady_frame_s)."""
    import oracle
    if w is None:
        w = oracle.OracleWeights(path, dtype=np.float32)
    p = wl.prompts[0]
    frames = ORACLE_SAMPLE_FRAMES
    o = oracle.DualAROracle(w, paged=True, pool_pages=-(-(p.T + frames + 16) // 16) + 4, radix=False)
    t0 = time.perf_counter()
    o.prefill(0, p.tokens, p.codes, p.mask)
    t1 = time.perf_counter()
    o.decode_frames([0], 1)
    t2 = time.perf_counter()
    o.decode_frames([0], frames - 1)
    t3 = time.perf_counter()
    return w, t1 - t0, t2 - t1, (t3 - t2) / (frames - 1)


def oracle_rate(wl, samples):
    """frames/s of the oracle on the workload, projected from the medians of
    the samples: each sequence costs its prefill + the first frame + n - 1
    steady frames, and the oracle runs the batch's sequences one after
    another (they are independent)."""
    tp = statistics.median(x[0] for x in samples)
    t0 = statistics.median(x[1] for x in samples)
    ts = statistics.median(x[2] for x in samples)
    n = wl.n_frames
    per_seq = tp + t0 + (n - 1) * ts
    return n / per_seq, tp, t0, ts


def oracle_sample_text(wl, tp, t0, ts, k):
    return (f"sequence 0, median of {k} samples: prefill ({wl.prompts[0].T} tokens, {tp:.2f} s), "
            f"first frame ({t0:.3f} s), {ORACLE_SAMPLE_FRAMES - 1} steady frames ({ts:.3f} s each); "
            f"fp32 NumPy, projected to {wl.n_frames} frames per sequence, sequences one after another")


CPU_BASELINE_SAMPLES = 3


def cpu_baseline(wl, path):
    w, samples = None, []
    for _ in range(CPU_BASELINE_SAMPLES):
        w, tp, t0, ts = oracle_sample(wl, path, w)
        samples.append((tp, t0, ts))
    value, tp, t0, ts = oracle_rate(wl, samples)
    return {"value": value, "unit": "frames/s", "cores": NCORES, "kind": "oracle",
            "sample": oracle_sample_text(wl, tp, t0, ts, len(samples))}


def run_reference(args):
    """The oracle as the reference arm: same workload, metric and unit; each
    step one sample (prefill + first frame + steady frames of sequence 0),
    the same rule the cpu_baseline of our arm uses."""
    from s2_inputs import ensure_weights, make_workload
    wl = make_workload(args.workload)
    path = ensure_weights(wl.model)
    w = None
    for _ in range(args.warmup):
        w, _, _, _ = oracle_sample(wl, path, w)
    samples = []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        w, tp, t0, ts = oracle_sample(wl, path, w)
        samples.append((tp, t0, ts))
    wall = time.perf_counter() - t_start
    value, tp, t0, ts = oracle_rate(wl, samples)
    n = wl.n_frames
    return {"metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * wall / args.steps,
            "ms_per_frame": 1000.0 / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "frames": n},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "frames/s", "cores": NCORES, "kind": "oracle",
                             "sample": oracle_sample_text(wl, tp, t0, ts, len(samples))},
            "e2e": {"value": value, "unit": "frames/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_attn_kernel(args, b, torch, cfg):
    """Decode attention (K3+K4) on the S2 heads: ``--rows`` sequences, each
    with ``--ctx`` cached keys plus the new one, fp32 pages (``--kv-bf16``:
    bf16), one pool per layer of ``--layers``; the split count is the
    runtime's (s2op_attn_decode_pick_split)."""
    B, ctx, L = args.rows, args.ctx, args.layers
    H, Hkv, hd = cfg.n_heads, cfg.n_kv, cfg.head_dim
    qd, kvd = H * hd, Hkv * hd
    P = 16
    ppseq = (ctx + 1 + P - 1) // P
    n_pages = B * ppseq
    kvsz = 2 if args.kv_bf16 else 4
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nsplit = b.s2op_attn_decode_pick_split(B, cfg.n_heads, Hkv, cfg.head_dim, args.kv_bf16)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    dt = torch.bfloat16 if args.kv_bf16 else torch.float32
    pools = [torch.randn((n_pages, 2, Hkv, P, hd), device="cuda", generator=gen).to(dt) for _ in range(L)]
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(7)).to(torch.int32)
    table = perm.reshape(B, ppseq).contiguous()
    shared = args.shared_prefix // P * P
    if shared:   # every sequence's table starts with sequence 0's first pages
        table[:, : shared // P] = table[0, : shared // P]
    table = table.cuda()
    pos = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
    qkv = torch.randn((B, qd + 2 * kvd), device="cuda", generator=gen)
    gain = torch.ones(hd, device="cuda")
    cs, sn = b.s2op_rope_table(ctx + 1, hd, cfg.rope_theta)
    cs, sn = torch.from_numpy(cs).cuda(), torch.from_numpy(sn).cuda()
    o = torch.zeros((B, qd), device="cuda")
    st = torch.cuda.Stream()
    if shared:   # per layer: the shared keys' operand images, written once (as per decode call)
        wss = [torch.zeros(b.s2op_attn_decode_prefix_workspace_bytes(B, H, Hkv, hd, nsplit, ctx + 1),
                           dtype=torch.uint8, device="cuda") for _ in range(L)]
        for l in range(L):
            b.s2op_attn_prefix_planes(pools[l], int(args.kv_bf16), table, Hkv, hd, shared, ctx + 1, wss[l],
                                      stream=st)
    else:
        ws = torch.zeros(b.s2op_attn_decode_workspace_bytes(B, 1, H, Hkv, hd, nsplit), dtype=torch.uint8,
                         device="cuda")
    torch.cuda.synchronize()

    def one():
        for l in range(L):
            if shared:
                b.s2op_attn_decode_shared_prefix(qkv, qd + 2 * kvd, B, H, Hkv, hd, gain, gain, cfg.eps, cs,
                                                 sn, pos, pools[l], int(args.kv_bf16), table, ppseq, shared,
                                                 ctx + 1, o, qd, nsplit=nsplit, workspace=wss[l], stream=st)
            else:
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
    # algorithmic bytes of one launch: the cached keys and values (a shared
    # prefix once), the new row's q/k/v in and its k/v appended, the output out
    kv_tokens = shared + B * (ctx - shared)
    per = kv_tokens * 2 * kvd * kvsz + B * ((qd + 2 * kvd) * 4 + 2 * kvd * kvsz + qd * 4)
    pk, kind = peaks()
    gbs = per * launches / ms / 1e6
    phases = prefix_phase_trace(b, torch, one, B, Hkv) if (shared and args.trace) else None
    print(json.dumps({"kernel": "attn", "rows": B, "ctx": ctx, "shared_prefix": shared, "layers": L,
                      "prefix_phases_us": phases, "nsplit": nsplit,
                      "kv": "bf16" if args.kv_bf16 else "fp32", "launches": launches,
                      "us_per_launch": 1000 * ms / launches, "bytes_per_launch": per,
                      "gbs": gbs, "frac_hbm": gbs / pk["hbm_gbs"], "peak_kind": kind}), flush=True)


def frame_trace_summary(path):
    """The last decoded frame's timeline (S2_FRAME_TRACE): per launch kind, in
    us, the medians over its launches of: step = its last CTA's exit after the
    previous launch's last exit; wait = when its CTAs pass the wait on the
    previous kernel, after that kernel's last exit (median over CTAs);
    prologue = wait to end of the activation prologue; body = prologue end to
    exit (median over CTAs); tail = last exit after the median exit."""
    kinds, rows = {}, {}
    for line in open(path):
        f = line.split()
        if f[0] == "launch":
            kinds[int(f[1])] = " ".join(f[2:])
        else:
            rows.setdefault(int(f[0]), []).append([int(x) for x in f[2:6]])
    ids = sorted(rows)
    per = {}
    prev_exit = None
    for i in ids:
        t = np.array(rows[i], dtype=np.int64)
        # rows left over from an earlier graph's launch in the same slot (more
        # CTAs than this launch) lie far from this launch's entries: drop them
        t = t[np.abs(t[:, 0] - np.median(t[:, 0])) < 1_000_000]
        last_exit = int(t[:, 3].max())
        rec = {"prologue": float(np.median(t[:, 2] - t[:, 1])), "body": float(np.median(t[:, 3] - t[:, 2])),
               "tail": float(last_exit - np.median(t[:, 3]))}
        if prev_exit is not None:
            rec["step"] = float(last_exit - prev_exit)
            rec["wait"] = float(np.median(t[:, 1]) - prev_exit)
        prev_exit = last_exit
        per.setdefault(kinds.get(i, "?"), []).append(rec)
    out = {}
    for k, recs in per.items():
        out[k] = {"launches": len(recs)}
        for key in ("step", "wait", "prologue", "body", "tail"):
            v = [r[key] for r in recs if key in r]
            if v:
                out[k][key] = round(float(np.median(v)) / 1000, 2)
    def kept(i):
        t = np.array(rows[i], dtype=np.int64)
        return t[np.abs(t[:, 0] - np.median(t[:, 0])) < 1_000_000]
    span = max(int(kept(i)[:, 3].max()) for i in ids) - min(int(kept(i)[:, 0].min()) for i in ids)
    return {"launches": len(ids), "span_us": span / 1000, "by_kind": out}


def prefix_phase_trace(b, torch, one, B, Hkv):
    """One more call with the shared-prefix kernel's phase trace on (the
    last layer's launch is kept): per phase the median over the CTAs that
    ran it (us), and the launch's span from the first entry to the last
    exit."""
    n = 8 * Hkv * ((4 * B + 127) // 128)
    buf = torch.zeros((n, 16), dtype=torch.int64, device="cuda")
    b.s2op_attn_prefix_set_trace(buf, n)
    one()
    torch.cuda.synchronize()
    b.s2op_attn_prefix_set_trace(None, 0)
    t = buf.cpu().numpy().astype(np.int64)
    names = ["setup", "dependency_wait", "query_copy_issue", "operands_landed", "s_mma", "softmax", "pv_mma",
             "o_readback", "cluster_barrier_1", "merge", "cluster_barrier_2"]
    out = {}
    for i, nm in enumerate(names, start=1):
        prev = i - 1
        if i == 8:   # after the last chunk: from P V of the first chunk, or the query issue (no chunk)
            ok = t[:, 7] > 0
            d = np.where(ok, t[:, 8] - t[:, 7], t[:, 8] - t[:, 3])
            out[nm] = float(np.median(d)) / 1000
            continue
        if i == 9:
            prev = 8
        ok = (t[:, i] > 0) & (t[:, prev] > 0)
        out[nm] = float(np.median(t[ok, i] - t[ok, prev])) / 1000 if ok.any() else None
    out["span"] = float(t[:, 11].max() - t[:, 0].min()) / 1000
    return out


def tc_phase_trace(b, torch, shapes, mats, x16, x16lo, ys, y16, F, R, ws, tk, st, two_plane):
    """One launch of each projection shape with the K2 phase trace on: per
    shape the launch ramp (spread of CTA entry), the median per-CTA phase
    durations (us) and the whole span, from globaltimer stamps."""
    buf = torch.zeros((1024, 6), dtype=torch.int64, device="cuda")
    out = []
    names = ["qkv", "o", "gate_up", "down"]
    for (N, K, mode, _), W, nm in zip(shapes, mats, names):
        b.s2op_tc_set_trace(buf, 1024)
        buf.zero_()
        kw = dict(Y16=y16, ldy16=F, epi=2) if mode == 2 else dict(Y=ys[N], ldy=N, epi=mode)
        if two_plane:
            b.s2op_tc_gemm2(W, N, K, x16[K], x16lo[K], R, K, workspace=ws, tickets=tk, stream=st, **kw)
        else:
            kw.pop("Y16lo", None)
            b.s2op_tc_gemm(W, N, K, x16[K], R, K, workspace=ws, tickets=tk, stream=st, **kw)
        torch.cuda.synchronize()
        b.s2op_tc_set_trace(None, 0)
        t = buf.cpu().numpy()
        t = t[t[:, 0] > 0].astype(np.float64)
        t0 = t[:, 0].min()
        d = np.diff(t, axis=1) / 1e3
        out.append({"shape": nm, "ctas": int(len(t)), "ramp_us": float((t[:, 0].max() - t0) / 1e3),
                    "span_us": float((t[:, 5].max() - t0) / 1e3),
                    "median_us": {k: float(np.median(d[:, i])) for i, k in
                                  enumerate(["setup", "first_stage", "stream", "mma_tail", "epilogue"])},
                    "max_us": {k: float(np.max(d[:, i])) for i, k in
                               enumerate(["setup", "first_stage", "stream", "mma_tail", "epilogue"])}})
    return out


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
    xf = {K: torch.randn((R, K), device="cuda") for (_, K, _, _) in shapes}
    x16 = {K: xf[K].to(torch.bfloat16) for K in xf}
    x16lo = {K: (xf[K] - x16[K].float()).to(torch.bfloat16) for K in xf}
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
                elif args.two_plane:   # the decode path's operand: bf16 hi + lo planes
                    if mode == 2:
                        b.s2op_tc_gemm2(W, N, K, x16[K], x16lo[K], R, K, Y16=y16, ldy16=F, epi=2,
                                        workspace=ws, tickets=tk, stream=st)
                    else:
                        b.s2op_tc_gemm2(W, N, K, x16[K], x16lo[K], R, K, Y=ys[N], ldy=N, epi=mode,
                                        workspace=ws, tickets=tk, stream=st)
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
    phases = None
    if args.trace and args.kernel == "tc":
        phases = tc_phase_trace(b, torch, shapes, mats[0], x16, x16lo, ys, y16, F, R, ws, tk, st,
                                args.two_plane)
    print(json.dumps({"kernel": args.kernel, "rows": R, "layers": L, "launches": launches,
                      "phases": phases,
                      "us_per_launch": 1000 * ms / launches, "weight_gbs": wbytes / ms / 1e6,
                      "frac_hbm": wbytes / ms / 1e6 / pk["hbm_gbs"], "tflops": flops / ms / 1e9,
                      "peak_kind": kind}), flush=True)


def dac_plan(cfg, B, n):
    """The vocoder decode's launches in order with their algorithmic work for
    B sequences of n frames: (name, flops, bytes).  Flops count one
    multiply-add per weight tap and output (x2), unpadded channels; bytes are
    the layer-by-layer minimum: each convolution reads its input activation
    once and writes its output once at 4 bytes an element, a residual
    convolution also reads the residual stream, and the bf16 weights are read
    once per launch."""
    out = [("halo_clear", 0, 0)]
    T = B * n
    out.append(("codebook_lookup", 2 * T * cfg.n_codebooks * cfg.latent * cfg.cb_dim,
                T * cfg.n_codebooks * 4 + T * cfg.latent * 4))

    def conv(name, rows_out, cin, cout, taps, rows_in, resid=False):
        fl = 2 * rows_out * cout * cin * taps
        by = rows_in * cin * 4 + rows_out * cout * 4 + (rows_out * cout * 4 if resid else 0) + \
            2 * cout * cin * taps
        return (name, fl, by)

    out.append(conv("conv_in", T, cfg.latent, cfg.dim, 7, T))
    rows = T
    for i, s in enumerate(cfg.rates):
        ci, co = cfg.channels(i - 1), cfg.channels(i)
        name = f"block.{i}.up"
        fl = 2 * rows * s * co * ci * 2
        by = rows * ci * 4 + rows * s * co * 4 + 2 * ci * co * 2 * s
        out.append((name, fl, by))
        rows *= s
        for j in range(3):
            out.append(conv(f"block.{i}.res.{j}.conv1", rows, co, co, 7, rows))
            out.append(conv(f"block.{i}.res.{j}.conv2", rows, co, co, 1, rows, resid=True))
    cl = cfg.channels(len(cfg.rates) - 1)
    out.append(("out_conv", 2 * rows * cl * 7, rows * cl * 4 + rows * 4))
    return out


def vocoder_record(b, torch, B, n, steps, warmup, peak):
    """Time the full-size vocoder on B sequences of n frames (codes resident
    on the device, waveform written to the device): ``steps`` decodes after
    ``warmup``, then one decode with per-launch events for the breakdown and
    the dominant launch's roofline."""
    from s2_inputs.vocoder import DAC_S2, ensure_vocoder, random_codes
    path = ensure_vocoder(DAC_S2)
    v = b.s2_vocoder_create(path, B, n)
    try:
        codes = torch.from_numpy(random_codes(DAC_S2, B, n, 900)).cuda()
        audio = torch.zeros((B, n * DAC_S2.hop), dtype=torch.float32, device="cuda")
        for _ in range(max(1, warmup)):
            b.s2_vocoder_decode(v, codes, audio)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            b.s2_vocoder_decode(v, codes, audio)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        launches = b.s2_vocoder_last_launches(v)
        b.s2_vocoder_set_profile(v, True)
        b.s2_vocoder_decode(v, codes, audio)
        per = b.s2_vocoder_profile(v)
        b.s2_vocoder_set_profile(v, False)
    finally:
        b.s2_vocoder_destroy(v)
    return vocoder_summary(DAC_S2, B, n, ms, launches, per, peak)


def vocoder_summary(cfg, B, n, ms, launches, per, peak):
    """JSON record of a timed vocoder decode: ``ms`` per call, ``per`` the
    per-launch durations (ms) of one profiled call in launch order."""
    plan = dac_plan(cfg, B, n)
    per = [float(x) for x in per]
    ms = float(ms)
    assert len(plan) == len(per), (len(plan), len(per))
    P_f, P_b = peak["bf16_tflops"] * 1e12, peak["hbm_gbs"] * 1e9
    rows = []
    roof_s = 0.0
    for (name, fl, by), t in zip(plan, per):
        tr = max(fl / P_f, by / P_b)
        roof_s += tr
        rows.append({"launch": name, "us": round(1000 * float(t), 2), "tflops": fl / (t * 1e9) if t else 0,
                     "gbs": by / (t * 1e6) if t else 0, "frac_roofline": tr / (t * 1e-3) if t else 0})
    dom = max(range(len(rows)), key=lambda i: rows[i]["us"])
    name, fl, by = plan[dom]
    t = float(per[dom]) * 1e-3
    tensor = fl / P_f >= by / P_b
    frames = B * n
    return {
        "workload": f"{cfg.name}_b{B}_f{n}", "batch": B, "frames_per_sequence": n,
        "samples_per_frame": cfg.hop, "ms_per_call": ms, "frames_per_s": frames / ms * 1e3,
        "audio_seconds_per_s": frames * cfg.hop / 44100 / (ms * 1e-3),
        "gpu_launches_per_call": int(launches),
        "algorithmic_tflop_per_call": sum(p[1] for p in plan) / 1e12,
        "algorithmic_gb_per_call": sum(p[2] for p in plan) / 1e9,
        "roofline_ms_per_call": roof_s * 1e3, "frac_of_roofline": roof_s * 1e3 / ms,
        "roofline": {"kernel": f"dac_conv_kernel ({name})", "bound": "tensor" if tensor else "hbm",
                     "achieved": (fl / t / 1e12) if tensor else (by / t / 1e9),
                     "peak": peak["bf16_tflops"] if tensor else peak["hbm_gbs"],
                     "unit": "TFLOP/s" if tensor else "GB/s",
                     "frac": (fl / t / P_f) if tensor else (by / t / P_b),
                     "flops_per_launch": fl, "bytes_per_launch": by, "us_per_launch": t * 1e6,
                     "traffic": None},
        "launches": rows,
    }


def run_dac(args):
    """``--kernel dac``: the full-size DAC vocoder decode (one JSON line)."""
    import torch
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding as b
    pk, kind = peaks()
    B = args.rows if args.rows > 1 else 32
    n = args.frames or 300
    rec = vocoder_record(b, torch, B, n, args.steps, args.warmup, pk)
    rec["kernel"] = "dac"
    rec["peak_kind"] = kind
    print(json.dumps(rec), flush=True)


def run_calibration(args):
    """Read-bandwidth calibration on this GPU (one JSON line).

    The dedicated streaming-read kernels of the library (s2op_stream_read):
    one 4 GiB buffer read by plain 16-byte loads (one launch) and by the
    persistent bulk-copy ring at several chunk sizes; then ``--layers``
    layers of the four S2 projection matrices read as a chain of operations
    (one launch per matrix; the ring without and with a grid barrier between
    matrices); the weight-streaming GEMV on the same chain and on one large
    matrix; torch's own sum and copy for comparison.  All buffers are far
    beyond L2, so every read comes from HBM."""
    import torch
    from s2_inputs import S2
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding as b
    cfg = S2
    d, F, qd, kvd = cfg.d, cfg.ffn, cfg.q_dim, cfg.kv_dim
    shapes = [(qd + 2 * kvd, d), (d, qd), (2 * F, d), (d, F)]
    L = args.layers
    mats = [torch.empty((N, K), device="cuda", dtype=torch.bfloat16).normal_(0, 0.02)
            for _ in range(L) for (N, K) in shapes]
    big = torch.empty((1 << 31,), device="cuda", dtype=torch.bfloat16).normal_()   # 4 GiB
    st = torch.cuda.Stream()
    torch.cuda.set_stream(st)
    scratch = torch.zeros(b.s2op_stream_read_scratch_bytes(len(mats)), dtype=torch.uint8, device="cuda")
    out = {"layers": L, "chain_bytes": sum(m.numel() * 2 for m in mats)}

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) / 1000.0
            best = t if best is None else min(best, t)
        return best

    errs = []

    def ring(bufs, nbytes, reps, chunk, stages, barrier):
        errs.append(b.s2op_stream_read(bufs, nbytes, scratch, reps=reps, mode=1, chunk_bytes=chunk,
                                       stages=stages, barrier=barrier, stream=st))

    nb_big = big.numel() * 2
    t = timed(lambda: b.s2op_stream_read([big], [nb_big], scratch, reps=1, mode=0, stream=st))
    out["ldg_4GiB_gbs"] = nb_big / t / 1e9
    for chunk, stages in [(8192, 24), (16384, 12), (32768, 6), (16384, 6), (49152, 4)]:
        t = timed(lambda: ring([big], [nb_big], 1, chunk, stages, 0))
        out[f"ring_4GiB_{chunk // 1024}Kx{stages}_gbs"] = nb_big / t / 1e9
    chain = [m for m in mats]
    nbs = [m.numel() * 2 for m in mats]
    tot = sum(nbs)
    t = timed(lambda: b.s2op_stream_read(chain, nbs, scratch, reps=1, mode=0, stream=st))
    out["ldg_chain_launch_per_matrix_gbs"] = tot / t / 1e9
    for chunk, stages in [(16384, 12), (32768, 6)]:
        for bar in (0, 1):
            t = timed(lambda: ring(chain, nbs, 1, chunk, stages, bar))
            out[f"ring_chain_{chunk // 1024}Kx{stages}_barrier{bar}_gbs"] = tot / t / 1e9
    xs = {K: torch.randn((1, K), device="cuda") for (_, K) in shapes}
    ys = {N: torch.zeros((1, N), device="cuda") for (N, _) in shapes}

    def gemv_chain():
        for i, m in enumerate(mats):
            N, K = m.shape
            b.s2op_gemv(m, N, K, xs[K], K, 1, ys[N], N, stream=st)

    t = timed(gemv_chain)
    out["gemv_chain_gbs"] = tot / t / 1e9
    huge = big[: 131072 * d].view(131072, d)
    y = torch.zeros((1, 131072), device="cuda")
    t = timed(lambda: b.s2op_gemv(huge, 131072, d, xs[d], d, 1, y, 131072, stream=st))
    out["gemv_671MB_gbs"] = huge.numel() * 2 / t / 1e9
    t = timed(lambda: big.sum(dtype=torch.float32))
    out["torch_sum_4GiB_gbs"] = nb_big / t / 1e9
    half = big[: 1 << 30]
    t = timed(lambda: half.clone())
    out["torch_copy_2GiB_rw_gbs"] = 2 * half.numel() * 2 / t / 1e9
    out["ring_errors"] = sum(1 for e in errs if e)
    pk, kind = peaks()
    out["peak_gbs"] = pk["hbm_gbs"]
    out["peak_kind"] = kind
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
    ap.add_argument("--no-batch32", action="store_true",
                    help="skip the batch-32 record the default (workload 1) run adds")
    ap.add_argument("--no-vocoder", action="store_true",
                    help="skip the DAC vocoder record the default (workload 1) run adds")
    ap.add_argument("--int8", action="store_true",
                    help="per-channel INT8 weights (reported separately; not the bf16 headline)")
    ap.add_argument("--kv-bf16", action="store_true",
                    help="bf16 Slow AR KV cache (default fp32)")
    ap.add_argument("--persist", action="store_true",
                    help="decode full frames in the persistent kernel instead of per-frame CUDA graphs")
    ap.add_argument("--profile-decode", action="store_true",
                    help="one prefill + one decode call of --frames frames, the decode inside an NVTX "
                         "range s2_decode (for profiler launch lists; prints no bench line)")
    ap.add_argument("--no-prefix-tc", action="store_true",
                    help="attend to a batch's shared radix prefix on CUDA cores (default: tcgen05)")
    ap.add_argument("--frame-trace", action="store_true",
                    help="per-CTA timeline of the last decoded frame's GEMV and attention launches "
                         "(S2_FRAME_TRACE), summarised per launch kind")
    ap.add_argument("--stream", action="store_true",
                    help="decode full frames at batch 1-2 in the streaming kernel")
    ap.add_argument("--kernel", choices=["gemv", "tc", "attn", "calib", "dac"], default=None,
                    help="microbenchmark one kernel on the S2 shapes instead of the workload")
    ap.add_argument("--rows", type=int, default=1)
    ap.add_argument("--two-plane", action="store_true",
                    help="--kernel tc: activations as two bf16 planes (the decode path's operand)")
    ap.add_argument("--trace", action="store_true",
                    help="--kernel tc: one launch per shape with the K2 phase trace; --kernel attn with "
                         "--shared-prefix: the prefix kernel's phase trace (per-CTA timestamps)")
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--ctx", type=int, default=100, help="--kernel attn: cached keys per sequence")
    ap.add_argument("--shared-prefix", type=int, default=0,
                    help="--kernel attn: keys every sequence shares (radix pages; tcgen05 prefix attention)")
    args = ap.parse_args()
    if args.kernel == "calib":
        run_calibration(args)
        return
    if args.kernel == "dac":
        run_dac(args)
        return
    if args.profile_decode:
        run_profile_decode(args)
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
