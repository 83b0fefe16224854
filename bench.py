"""Benchmark: batch-1 MoE decode throughput on B300 through libmoe.

Default workload: the 80B-shaped (hidden 2048, 512 experts, top-10, inter 512, shared 512,
int4 group 64) 48-layer pre-norm residual stack with every expert blob resident in the HBM pool at
a fixed stride. One step = one decode token through all 48 layers = one cooperative kernel launch
(router, top-k, routed + shared experts, combine, residual for every layer). Each step streams
~1.04 GB of weights, far above the 126 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an independent replica on its
own GPU (the layer has no exchange step at batch 1); value = tokens of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CONFIGS = {
    # name: (shape factory, layers, description)
    "stack80": ("S80", 48, 4, "80B-shaped 48-layer resident MoE stack, batch-1 decode, int4"),
    "stack35": ("S35", 40, 4, "35B-shaped 40-layer resident MoE stack, batch-1 decode, int4"),
    "stack35_int8": ("S35", 40, 8, "35B-shaped 40-layer resident MoE stack, batch-1 decode, int8"),
    "stack80_pool2g": ("S80", 48, 4, "80B-shaped 48-layer MoE stack, batch-1 decode, bounded 2 GiB HBM expert pool "
                       "(LFU + recency) filled from pinned host memory, Zipf(1.1) routing popularity"),
}
for _t in (8, 64, 512, 4096):
    CONFIGS[f"prefill80_t{_t}"] = ("S80", 1, 4, f"80B-shaped single MoE layer, batched decode/prefill of {_t} tokens, "
                                   "int4, router top-10, tokens sorted per expert, grouped GEMMs on the tensor cores")
BATCHED = {f"prefill80_t{_t}": _t for _t in (8, 64, 512, 4096)}
# the hybrid stack's other per-layer steps: (step kind, layers, context)
CONFIGS["gdn80"] = ("GDN80", 36, 32, "80B-shaped Gated DeltaNet decode step through the 36 DeltaNet layers "
                    "(16 key / 32 value heads, 128 x 128 fp32 state per value head: 72 MiB in all)")
CONFIGS["gqa80_8k"] = ("GQA80", 12, 32, "80B-shaped gated GQA decode attention through the 12 attention layers "
                       "at an 8K context (16 query / 2 K/V heads of 256, fp32 K/V cache: 384 MiB in all)")
HYBRID = {"gdn80": ("gdn", 36, 0), "gqa80_8k": ("gqa", 12, 8192)}
BATCHED_LAYERS = 8  # resident layers rotated step by step, so consecutive steps read disjoint weights
POOL_SLOTS = {"stack80_pool2g": (2 << 30) // 1769472}  # 1213 slots of 1,769,472 bytes
METRIC = "MoE decode tokens/s (1 B300) and expert-byte HBM GB/s vs ~8 TB/s roofline"
SEED = 0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def _tensor_peak():
    """Dense fp16/bf16 tensor TFLOP/s (the same nominal rate for both types): the measured cuBLAS
    bf16 burst figure when present."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        for key in ("bf16_tflops", "bf16_tflops_burst"):
            if key in d:
                return float(d[key]), "measured (cuBLAS bf16 burst; fp16 has the same nominal rate)"
    return 1800.0, "fallback"


def _shape(name, bits):
    from int4_routed_expert_05_b300 import synth
    return getattr(synth, name).with_bits(bits)


def _bytes_per_layer(sh):
    """Algorithmic bytes of one layer for one token: routed + shared expert blobs, router, gate."""
    from int4_routed_expert_05_b300 import moe
    from int4_routed_expert_05_b300.resident import moe_shape
    ms = moe_shape(sh)
    blob = moe.expert_bytes(ms)
    blob_s = moe.expert_bytes(ms, shared=True)
    expert = sh.top_k * blob + blob_s
    router = sh.n_experts * sh.hidden * 2 + sh.hidden * 2
    return expert, router


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(ws, v):
    """The slowest rank's time (every rank gets it): the whole job's clock."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(sh, n_layers_sample, n_layers_model, seed=SEED, budget_s=20.0, threads=1):
    """The oracle as it stands on a bounded sample of the same workload: n_layers_sample layers of
    the stack for as many tokens as fit the budget (at least one), its row loops on `threads` host
    threads (1: serial). Returns tokens/s of the full n_layers_model stack (time scaled by the
    layer ratio)."""
    import oracle
    from int4_routed_expert_05_b300 import synth
    from oracle.layers import OracleLayers
    oracle.set_threads(threads)
    O = OracleLayers(oracle, sh, seed, n_layers_sample)
    for l in range(n_layers_sample):       # blobs of the layers are packed outside the timed region
        O.dense(l)
    t_total, tokens = 0.0, 0
    while tokens == 0 or t_total < budget_s:
        x = synth.activation_f32(sh, seed, 10_000 + tokens)[0].astype(np.float64)
        for l in range(n_layers_sample):
            u = oracle.rmsnorm_bf16(x)
            # the selected experts' blobs are written outside the timed region
            lg, _ = oracle.router_logits(O.dense(l)[0], u)
            for e in oracle.topk(lg, sh.top_k, sh.renorm)[0]:
                O.blob(l, int(e))
            t0 = time.perf_counter()
            r = O.layer(l, u)
            t_total += time.perf_counter() - t0
            x = x + r["y"]
        tokens += 1
        if tokens >= 64:
            break
    oracle.set_threads(1)
    per_token_full = t_total / tokens * (n_layers_model / n_layers_sample)
    return 1.0 / per_token_full, {"layers": n_layers_sample, "tokens": tokens, "seconds": t_total, "threads": threads}


def run_reference(args):
    """The oracle as it stands, on every host core (its row loops threaded; the results equal the
    serial ones bit for bit), on this arm's workload. A step is a bounded sample: one full oracle
    layer for one token when K + W of them fit in about two and a half minutes, else one expert FFN
    of a layer (the oracle's dominant cost), with tokens/s of the whole stack derived from the
    sampled time."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    if args.config in HYBRID:
        kind, L, ctx = HYBRID[args.config]
        times, vals = [], []
        for i in range(args.warmup + args.steps):
            v, info = cpu_oracle_hybrid(kind, L, ctx, budget_s=min(2.0, args.ref_budget))
            if i >= args.warmup:
                vals.append(v)
        value = statistics.median(vals)
        line = {"impl": "reference", "metric": f"{'Gated DeltaNet' if kind == 'gdn' else 'gated GQA'} decode "
                f"tokens/s through {L} layers (1 B300) and HBM GB/s vs the measured copy roofline",
                "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 / value, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic (seeded generator)",
                "config": {"workload": args.config, "description": CONFIGS[args.config][3], "batch": 1, "layers": L},
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": info},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    import oracle
    from int4_routed_expert_05_b300 import synth
    from oracle.layers import OracleLayers
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    oracle.set_threads(ncores)
    name, L, bits, desc = CONFIGS[args.config]
    sh = _shape(name, bits)
    if args.config in BATCHED:
        times = []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            v_i, info = cpu_oracle_batched(sh, BATCHED[args.config], budget_s=2.0)
            times.append(time.perf_counter() - t0)
        v = v_i
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times[args.warmup:] or times),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.config, "description": desc, "tokens": BATCHED[args.config]},
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": ncores, "kind": "oracle", "sample": info},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    O = OracleLayers(oracle, sh, SEED, 1)
    Wr, w_sg, shared = O.dense(0)
    x = synth.activation_f32(sh, SEED, 0)[0].astype(np.float64)
    u = oracle.rmsnorm_bf16(x)
    t0 = time.perf_counter()
    r = O.layer(0, u)
    t_layer = time.perf_counter() - t0
    n_steps = args.warmup + args.steps
    blob = O.blob(0, int(r["idx"][0]))
    t0 = time.perf_counter()
    oracle.expert_ffn(sh, blob, u)
    t_expert = time.perf_counter() - t0
    # the largest unit whose K + W repetitions fit in about two and a half minutes
    mode = "layer" if n_steps * t_layer <= 150.0 else ("expert" if n_steps * t_expert <= 150.0 else "router")
    if mode == "layer":  # every blob written before timing
        for e in range(sh.n_experts):
            O.blob(0, e)
    times = []
    for i in range(n_steps):
        t0 = time.perf_counter()
        if mode == "layer":
            O.layer(0, oracle.rmsnorm_bf16(x + i * 1e-3))
        elif mode == "expert":
            oracle.expert_ffn(sh, blob, u)
        else:
            oracle.router_logits(Wr, u)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times[args.warmup:]) if args.steps else times[-1]
    if mode == "layer":
        v = 1.0 / (t * L)
        sample = f"one oracle layer (router, top-{sh.top_k}, {sh.top_k + 1} expert FFNs, combine) per step, x{L} layers"
    elif mode == "expert":
        t0 = time.perf_counter()
        oracle.router_logits(Wr, u)
        t_router = time.perf_counter() - t0
        v = 1.0 / (L * ((sh.top_k + 1) * t + t_router))
        sample = f"one expert FFN per step, scaled by {sh.top_k + 1} experts and {L} layers plus the router"
    else:
        v = 1.0 / (L * ((sh.top_k + 1) * t_expert + t))
        sample = (f"the router GEMV per step (one expert FFN timed once: {1e3 * t_expert:.1f} ms), scaled by "
                  f"{sh.top_k + 1} experts and {L} layers")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.config, "description": desc, "batch": 1, "layers": L},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": ncores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _h2d_gbs(nbytes=1 << 30):
    """Pinned host -> device copy bandwidth (one large copy, best of 3)."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    return best


def run_streamed(args):
    """Bounded-pool decode: the per-layer host loop of moe_stack_forward_streamed over 48 layers."""
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from int4_routed_expert_05_b300 import _build, synth
    _build.build()
    from int4_routed_expert_05_b300 import moe
    from int4_routed_expert_05_b300.streamed import Streamed, calibrate_beta, simulated_hit_rate
    name, L, bits, desc = CONFIGS[args.config]
    if args.layers:
        L, desc = args.layers, desc + f" (first {args.layers} layers only)"
    sh = _shape(name, bits)
    n_slots = POOL_SLOTS[args.config]
    if args.pool_gib:
        n_slots = int(args.pool_gib * (1 << 30)) // 1769472
    S = Streamed(sh, L, SEED, n_slots, beta=0.0, prefetch=0, verbose=(rank == 0))
    H = sh.hidden
    xs = torch.from_numpy(np.stack([synth.activation_f32(sh, SEED, s)[0] for s in range(64)])).cuda()
    # Zipf(1.1) popularity always on: beta is bisected on the device, over the timed run's own
    # warm-up and length, so that the measured hit rate lands near 0.60, inside the 43-70% band
    # (random-init routing alone already reuses experts).
    sched = dict(warm=args.warmup, tokens=args.steps)  # the timed run's own warm-up and length
    hr0 = S.measure_hit_rate(xs, **sched)
    if args.zipf_beta is not None:  # a fixed strength (a pool-size sweep keeps the routing fixed)
        beta, hr_cal = args.zipf_beta, None
    else:
        beta, hr_cal = (0.0, hr0) if hr0 >= 0.60 else S.calibrate_beta(xs, target=0.60, **sched)
    # the pool's own hit rate is calibrated without speculation; the timed run uses --prefetch
    S.prefetch = args.prefetch
    if beta != S.beta:
        S.set_beta(beta)
    sim = simulated_hit_rate(sh, L, n_slots, beta, seed=SEED)
    S.reset_pool()  # a fresh, empty pool for the timed run
    out = torch.empty(H, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    step = S.step
    qinfo = None
    if args.qpack:
        # the misses come from an on-disk container instead of the pinned host store
        t_w = time.perf_counter()
        S.write_qpack(args.qpack)
        t_w = time.perf_counter() - t_w
        qp = S.qpack = moe.Qpack.open(args.qpack, direct=True, n_threads=8)
        n_staging = 2 * sh.top_k
        staging = S.pinned_staging(n_staging)
        step = lambda x, o, st: S.step_qpack(x, o, qp, staging, n_staging, st)  # noqa: E731
        qinfo = {"path": args.qpack, "direct": qp.info()[3], "reader_threads": 8, "staging_slots": n_staging,
                 "file_bytes": os.path.getsize(args.qpack), "write_s": t_w}
    for i in range(args.warmup):
        step(xs[i % 64], out, stream)
    torch.cuda.synchronize()
    h0, m0, b0 = S.pool.stats()
    clocks = ClockSampler(local)
    _barrier(ws)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(args.steps):
        step(xs[(args.warmup + i) % 64], out, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    _barrier(ws)
    clk = clocks.stop()
    ms = _max_over_ranks(ws, e0.elapsed_time(e1))
    h1, m1, b1 = S.pool.stats()
    if S.pool.device_status() != 0:
        raise RuntimeError("device status is not MOE_OK after the timed region")
    if rank != 0:
        return
    hits, misses, nbytes = h1 - h0, m1 - m0, b1 - b0
    link = _h2d_gbs()
    miss_gbs = nbytes / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": ws * args.steps / (ms / 1e3), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int4",
        "data": "synthetic (seeded generator, random-init weights of the stated shapes)",
        "config": {"workload": args.config, "description": desc, "batch": 1, "layers": L, "pool_slots": n_slots,
                   "pool_bytes": n_slots * S.stride, "zipf_s": 1.1, "zipf_beta": beta,
                   "hit_rate_uniform_routing": hr0, "hit_rate_calibration": hr_cal, "simulated_hit_rate": sim,
                   "prefetch": args.prefetch,
                   "host_store": f"{S.n_unique} unique blobs pinned, expert (l, e) -> blob maps[l][e]"},
        "qpack": None if qinfo is None else dict(qinfo, read_gbs=nbytes / wall / 1e9),
        "pool": {"hit_rate": hits / max(1, hits + misses), "misses_per_token": misses / args.steps,
                 "miss_bytes_per_token": nbytes / args.steps, "miss_gbs": miss_gbs, "pinned_h2d_gbs": link,
                 "wall_s": wall},
        "roofline": {"bound": "host-link", "achieved": miss_gbs, "peak": link, "unit": "GB/s", "frac": miss_gbs / link,
                     "traffic": None, "peak_kind": "measured pinned H2D copy in this run"},
        "gpu_launches": args.steps * L * 2,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from int4_routed_expert_05_b300 import _build, synth
    _build.build()
    from int4_routed_expert_05_b300 import moe
    from int4_routed_expert_05_b300.resident import Resident

    name, L, bits, desc = CONFIGS[args.config]
    if args.layers:
        L, desc = args.layers, desc + f" (first {args.layers} layers only)"
    sh = _shape(name, bits)
    flags = moe.RENORM | moe.PRENORM | moe.RESIDUAL
    R = Resident(sh, L, SEED, flags=flags, verbose=(rank == 0))
    H = sh.hidden
    n_in = args.warmup + args.steps
    xs = torch.from_numpy(np.stack([synth.activation_f32(sh, SEED, s)[0] for s in range(min(n_in, 64))])).cuda()
    out = torch.empty(H, dtype=torch.float32, device="cuda")
    idx = torch.empty((L, sh.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((L, sh.top_k), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        R.pool.stack_forward(0, L, xs[i % xs.shape[0]], out, None, idx, w, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if R.pool.device_status() != moe.OK:
        raise RuntimeError("device status after warm-up is not MOE_OK")

    clocks = ClockSampler(local)
    _barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    ms = _max_over_ranks(ws, ms)
    status = R.pool.device_status()
    if status != moe.OK:
        raise RuntimeError(f"device status {status} after the timed region")

    # end to end through the C ABI with host buffers: pinned x in, residual out, every step
    h_x = torch.empty((xs.shape[0], H), dtype=torch.float32, pin_memory=True)
    h_x.copy_(xs.cpu())
    h_out = torch.empty(H, dtype=torch.float32, pin_memory=True)
    d_x = torch.empty(H, dtype=torch.float32, device="cuda")
    n_e2e = max(1, min(args.steps, 2000))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        d_x.copy_(h_x[i % h_x.shape[0]], non_blocking=True)
        R.pool.stack_forward(0, L, d_x, out, None, None, None, stream)
        h_out.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = _max_over_ranks(ws, e2e_s)

    if rank != 0:
        return
    expert_b, router_b = _bytes_per_layer(sh)
    per_launch_expert = expert_b * L
    per_launch_all = (expert_b + router_b) * L
    ms_step = ms / args.steps
    tok_s = ws * args.steps / (ms / 1e3)
    peak, peak_kind = _peaks()
    achieved = per_launch_expert / (ms_step / 1e3) / 1e9
    cpu_v, cpu_info, cpu1_v, cpu1_info = None, None, None, None
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    if ws == 1 and not args.no_cpu_baseline:
        # the oracle on every host core, and serially (half the budget each)
        cpu_v, cpu_info = cpu_oracle_sample(sh, args.ref_layers, L, budget_s=args.ref_budget / 2, threads=ncores)
        cpu1_v, cpu1_info = cpu_oracle_sample(sh, args.ref_layers, L, budget_s=args.ref_budget / 2, threads=1)
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        t = json.load(open(tp)).get(args.config)
        traffic = t.get("bytes_per_launch") if t else None
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4" if bits == 4 else "int8",
        "data": "synthetic (seeded generator, random-init weights of the stated shapes)",
        "config": {"workload": args.config, "description": desc, "batch": 1, "layers": L,
                   "hidden": sh.hidden, "experts": sh.n_experts, "top_k": sh.top_k, "inter": sh.inter,
                   "shared_inter": sh.shared_inter, "bits": bits, "group": sh.group,
                   "l2": "inputs larger than L2 (%.2f GB of weights per step vs 126 MB L2)" % (per_launch_all / 1e9),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "layer_latency_us": ms_step * 1e3 / L,
        "expert_gbs": achieved,
        "all_weight_gbs": per_launch_all / (ms_step / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "moe_decode_kernel", "bytes_per_launch": per_launch_expert},
        "cpu_baseline": None if cpu_v is None else {
            "value": cpu_v, "unit": "tokens/s", "cores": ncores, "kind": "oracle",
            "sample": f"{cpu_info['tokens']} token(s) through {cpu_info['layers']} of {L} layers in "
                      f"{cpu_info['seconds']:.1f} s on {ncores} threads (row loops), time scaled to the full stack",
            "serial": {"value": cpu1_v, "unit": "tokens/s", "cores": 1,
                       "sample": f"{cpu1_info['tokens']} token(s) through {cpu1_info['layers']} of {L} layers in "
                                 f"{cpu1_info['seconds']:.1f} s, one thread"}},
        "e2e": {"value": ws * n_e2e / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * H, "d2h_bytes_per_step": 4 * H,
                "steps": n_e2e},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_batched(args):
    """Batched decode / prefill of T tokens through one 80B-shaped layer (the GEMM path).
    One step = one call of moe_layer_forward_batched on T fresh tokens; the steps rotate over
    8 resident layers so that consecutive steps read disjoint weights (6.6 GB, far above L2)."""
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from int4_routed_expert_05_b300 import _build, synth
    _build.build()
    from int4_routed_expert_05_b300 import moe
    from int4_routed_expert_05_b300.resident import Resident

    T = BATCHED[args.config]
    name, _, bits, desc = CONFIGS[args.config]
    sh = _shape(name, bits)
    L = args.layers or BATCHED_LAYERS
    R = Resident(sh, L, SEED, flags=moe.RENORM | (moe.GEMV if args.gemv else 0), verbose=(rank == 0))
    H, E, k = sh.hidden, sh.n_experts, sh.top_k
    n_x = 4
    xs = torch.from_numpy(np.ascontiguousarray(
        np.stack([synth.activation_bits(sh, SEED, 1000 + i, T) for i in range(n_x)])).view(np.int16)).cuda()
    work = torch.empty(moe.batched_workspace_bytes(R.mshape, T), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i, x=None):
        R.pool.layer_forward_batched(i % L, xs[i % n_x] if x is None else x, T, y, work, idx, w, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if R.pool.device_status() != moe.OK:
        raise RuntimeError("device status after warm-up is not MOE_OK")
    # distinct experts touched per step (for the algorithmic bytes), from the warm-up's selection
    touched = []
    for i in range(min(L, 4)):
        step(i)
        touched.append(len(np.unique(idx.cpu().numpy())))
    torch.cuda.synchronize()

    # The layer call does no host synchronisation, so each (layer, input) pair of the rotation is
    # captured once as a CUDA graph and replayed: the same seven launches, without per-launch host
    # overhead. Falls back to direct calls if capture is refused. (Events recorded inside a graph
    # cannot be waited on from the host, so with graphs the expert-GEMM time comes from a second,
    # direct-call pass below.)
    n_combo = int(np.lcm(L, n_x))
    graphs = []
    if not args.no_graphs:
        try:
            R.pool.time_batched(0)
            gs = torch.cuda.Stream()
            gs.wait_stream(stream)
            for c in range(n_combo):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=gs):
                    R.pool.layer_forward_batched(c % L, xs[c % n_x], T, y, work, idx, w, gs)
                graphs.append(g)
            stream.wait_stream(gs)
            torch.cuda.synchronize()
        except Exception as exc:  # noqa: BLE001 - any refusal means direct calls
            print(f"[bench] CUDA graph capture unavailable ({exc}); timing direct calls", file=sys.stderr)
            graphs = []
            torch.cuda.synchronize()
    if not graphs:
        R.pool.time_batched(args.steps)  # CUDA events around the expert GEMMs of every timed step

    def timed_step(i):
        if graphs:
            graphs[i % n_combo].replay()
        else:
            step(i)

    for i in range(3):  # replays warm up too
        timed_step(args.warmup + i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    _barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        timed_step(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    clk = clocks.stop()
    ms = _max_over_ranks(ws, e0.elapsed_time(e1))
    if graphs:  # the expert GEMMs' own time, from direct calls with the event hook
        R.pool.time_batched(args.steps)
        for i in range(args.steps):
            step(args.warmup + i)
        torch.cuda.synchronize()
    gemm_ms, gemm_calls = R.pool.batched_gemm_ms()
    R.pool.time_batched(0)
    if R.pool.device_status() != moe.OK:
        raise RuntimeError("device status after the timed region is not MOE_OK")

    # end to end: bf16 tokens from pinned host memory in, fp32 outputs back, every step
    h_x = torch.empty((n_x, T, H), dtype=torch.int16, pin_memory=True)
    h_x.copy_(xs.cpu())
    h_y = torch.empty((T, H), dtype=torch.float32, pin_memory=True)
    d_x = torch.empty((T, H), dtype=torch.int16, device="cuda")
    n_e2e = max(1, min(args.steps, 200))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        d_x.copy_(h_x[i % n_x], non_blocking=True)
        step(i, d_x)
        h_y.copy_(y, non_blocking=True)
        stream.synchronize()
    e2e_s = _max_over_ranks(ws, time.perf_counter() - t0)
    if rank != 0:
        return

    from int4_routed_expert_05_b300.resident import moe_shape
    ms_ = moe_shape(sh)
    blob, blob_s = moe.expert_bytes(ms_), moe.expert_bytes(ms_, shared=True)
    uniq = float(np.mean(touched))
    A = T * (k + 1)
    # the expert GEMMs (the dominant kernels, about 90 % of a step): weights of the touched experts
    # and the shared expert, input rows and h rows in assignment order (fp16), y reductions (fp32)
    gemm_bytes = uniq * blob + blob_s + 2 * A * H + 2 * 2 * A * sh.inter + 4 * T * H
    gemm_flops = 2.0 * T * (k * 3 * sh.inter + 3 * sh.shared_inter) * H
    bytes_step = uniq * blob + blob_s + E * H * 2 + H * 2 + T * H * 2 + T * H * 4
    flops_step = 2.0 * T * (E * H + (k * 3 * sh.inter + 3 * sh.shared_inter) * H)
    ms_step = ms / args.steps
    ms_gemm = gemm_ms / max(1, gemm_calls)
    hbm_peak, hbm_kind = _peaks()
    tc_peak, tc_kind = _tensor_peak()

    def roofline(nbytes, flops, ms_unit):
        if flops / (tc_peak * 1e12) >= nbytes / (hbm_peak * 1e9):
            ach = flops / (ms_unit / 1e3) / 1e12
            return {"bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s", "frac": ach / tc_peak,
                    "peak_kind": tc_kind, "flops_per_launch": flops}
        ach = nbytes / (ms_unit / 1e3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                "peak_kind": hbm_kind, "bytes_per_launch": nbytes}

    roof = roofline(gemm_bytes, gemm_flops, ms_gemm)
    roof.update({"traffic": None, "kernel": "expert_kernel<1> + expert_kernel<2> (gate/up and down expert GEMMs)",
                 "ms_per_launch": ms_gemm, "timed_launches": gemm_calls})
    step_roof = roofline(bytes_step, flops_step, ms_step)
    step_roof.update({"kernel": "moe_layer_forward_batched (all 7 launches of one step)"})
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        v, info = cpu_oracle_batched(sh, T, budget_s=args.ref_budget)
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": info}
    line = {
        "metric": METRIC, "value": ws * T * args.steps / (ms / 1e3), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int4 weights, fp16 tensor-core operands, fp32 accumulate",
        "data": "synthetic (seeded generator, random-init weights of the stated shapes)",
        "config": {"workload": args.config, "description": desc, "tokens": T, "layers_rotated": L,
                   "expert_path": "matrix-vector (MOE_GEMV)" if args.gemv else "tensor-core GEMMs",
                   "cuda_graphs": bool(graphs),
                   "hidden": H, "experts": E, "top_k": k, "inter": sh.inter, "shared_inter": sh.shared_inter,
                   "bits": bits, "group": sh.group,
                   "l2": "steps rotate over %d resident layers (%.1f GB of expert blobs), far above the 126 MB L2"
                         % (L, L * E * blob / 1e9),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "layer_latency_us": ms_step * 1e3,
        "experts_touched_per_step": uniq,
        "tflops": flops_step / (ms_step / 1e3) / 1e12,
        "roofline": roof,
        "step_roofline": step_roof,
        "cpu_baseline": cpu,
        "e2e": {"value": ws * T * n_e2e / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 2 * T * H,
                "d2h_bytes_per_step": 4 * T * H, "steps": n_e2e},
        "gpu_launches": 7 * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def _hybrid_setup(kind, L, batch, ctx, n_steps):
    """Device state of a hybrid-step workload: per-layer parameters and state (or caches) and
    per-step inputs, all from the seeded generator."""
    import torch
    from int4_routed_expert_05_b300 import moe
    from int4_routed_expert_05_b300 import synth_hybrid as SH

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    W = {"kind": kind, "L": L, "batch": batch}
    n_in = min(n_steps, 8)  # distinct input sets, cycled

    def packed(layers):
        """Input set 0: every layer's inputs as views of one flat device buffer (16-byte aligned
        pieces), so that the end-to-end run moves a step's inputs with one host-to-device copy."""
        pieces, off = [], 0
        for d in layers:
            for k, a in d.items():
                a = np.ascontiguousarray(a)
                pieces.append((k, a, off))
                off += (a.nbytes + 15) // 16 * 16
        flat = np.zeros(off, np.uint8)
        for _, a, o in pieces:
            flat[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
        W["flat"] = torch.from_numpy(flat).cuda()
        out, i = [], 0
        for d in layers:
            e = {}
            for k, a in d.items():
                _, _, o = pieces[i]
                i += 1
                tdt = torch.int16 if a.dtype == np.uint16 else torch.float32
                e[k] = W["flat"][o:o + a.nbytes].view(tdt).view(a.shape)
            out.append(e)
        return out
    if kind == "gdn":
        sh = SH.GDN80
        W["shape"] = moe.GdnShape(sh.n_key_heads, sh.n_value_heads, sh.key_dim, sh.value_dim)
        W["state"] = [dev(SH.gdn_state(sh, SEED, l, batch)) for l in range(L)]
        W["par"] = [{k: dev(v) for k, v in SH.gdn_params(sh, SEED, l).items()} for l in range(L)]
        W["inp"] = [packed([SH.gdn_inputs(sh, SEED, l, 0, batch) for l in range(L)])] + [
            [{k: dev(v) for k, v in SH.gdn_inputs(sh, SEED, l, s, batch).items()} for l in range(L)]
            for s in range(1, n_in)]
        W["y"] = torch.empty(batch, sh.n_value_heads, sh.value_dim, device="cuda")
        # algorithmic bytes of one layer launch: state read + written, inputs, parameters, y
        W["bytes_per_launch"] = batch * (2 * 4 * sh.state_floats() + 2 * 2 * sh.n_key_heads * sh.key_dim +
                                         2 * 2 * sh.n_value_heads * sh.value_dim + 2 * 4 * sh.n_value_heads +
                                         4 * sh.n_value_heads * sh.value_dim) + 4 * (2 * sh.n_value_heads + sh.value_dim)
    else:
        sh = SH.GQA80
        W["shape"] = moe.GqaShape(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, ctx)
        start = ctx - n_steps
        W["kc"] = [dev(SH.gqa_cache(sh, SEED, l, ctx, start, batch)) for l in range(L)]
        W["vc"] = [dev(SH.gqa_cache(sh, SEED + 1, l, ctx, start, batch)) for l in range(L)]
        W["pos"] = torch.full((batch,), start, dtype=torch.int32, device="cuda")
        W["start"] = start
        W["inp"] = [packed([SH.gqa_inputs(sh, SEED, l, 0, batch) for l in range(L)])] + [
            [{k: dev(v) for k, v in SH.gqa_inputs(sh, SEED, l, s, batch).items()} for l in range(L)]
            for s in range(1, n_in)]
        W["y"] = torch.empty(batch, sh.n_q_heads, sh.head_dim, device="cuda")
        W["wb"] = moe.gqa_workspace_bytes(W["shape"], batch, ctx)
        W["work"] = torch.empty(W["wb"] // 4 + 4, dtype=torch.float32, device="cuda")
        W["status"] = torch.zeros(4, dtype=torch.int32, device="cuda")
        # algorithmic bytes of one layer at position p: K and V rows 0..p read (the new row
        # written), inputs, y
        W["kv_row_bytes"] = 2 * 4 * sh.n_kv_heads * sh.head_dim * batch
        W["io_bytes"] = batch * (2 * 2 * sh.n_q_heads * sh.head_dim + 2 * 2 * sh.n_kv_heads * sh.head_dim +
                                 4 * sh.n_q_heads * sh.head_dim)
    W["sh"] = sh
    return W


def _hybrid_step(W, s, stream_ptr):
    """One decode token through the workload's L layers (one launch, or two for GQA, per layer)."""
    from int4_routed_expert_05_b300 import moe
    inp = W["inp"][s % len(W["inp"])]
    for l in range(W["L"]):
        d = inp[l]
        if W["kind"] == "gdn":
            p = W["par"][l]
            moe.gdn_step(W["shape"], W["batch"], W["state"][l], d["q"], d["k"], d["v"], d["z"], d["a"], d["b"],
                         p["A_log"], p["dt_bias"], p["norm_w"], W["sh"].key_dim ** -0.5, W["y"], stream=stream_ptr)
        else:
            moe.gqa_decode(W["shape"], W["batch"], W["shape"].max_len, W["kc"][l], W["vc"][l], W["pos"], d["q"],
                           d["k"], d["v"], d["gate"], W["sh"].head_dim ** -0.5, W["work"], W["wb"], W["y"],
                           W["status"], stream=stream_ptr)


def cpu_oracle_hybrid(kind, L, ctx, budget_s=15.0):
    """The hybrid-step oracle as it stands, on host data from the seeded generator: layer steps of
    one sequence (cycling over the first layers' data) for as long as the budget allows (at least
    one). Returns (tokens/s for L layers, description of the sample)."""
    from oracle import hybrid as OH
    from int4_routed_expert_05_b300 import synth_hybrid as SH
    from int4_routed_expert_05_b300.synth import bf16_value
    f = lambda a: bf16_value(a[0]).astype(np.float64)
    n, t_total = 0, 0.0
    while n == 0 or t_total < budget_s:
        l = n % 2
        if kind == "gdn":
            sh = SH.GDN80
            S = SH.gdn_state(sh, SEED, l, 1)[0].astype(np.float64)
            p = SH.gdn_params(sh, SEED, l)
            d = SH.gdn_inputs(sh, SEED, l, 0, 1)
            t0 = time.perf_counter()
            OH.gdn_step(S, f(d["q"]), f(d["k"]), f(d["v"]), f(d["z"]), d["a"][0], d["b"][0], p["A_log"], p["dt_bias"],
                        p["norm_w"], sh.key_dim ** -0.5)
        else:
            sh = SH.GQA80
            if n < 2:
                caches = (SH.gqa_cache(sh, SEED, l, ctx, ctx - 1, 1)[0].astype(np.float64),
                          SH.gqa_cache(sh, SEED + 1, l, ctx, ctx - 1, 1)[0].astype(np.float64))
                cache_l = {l: caches}
            Kc, Vc = cache_l.get(l, caches)
            d = SH.gqa_inputs(sh, SEED, l, 0, 1)
            t0 = time.perf_counter()
            OH.gqa_step(Kc, Vc, ctx - 1, f(d["q"]), f(d["k"]), f(d["v"]), f(d["gate"]), sh.head_dim ** -0.5)
        t_total += time.perf_counter() - t0
        n += 1
    what = "state update" if kind == "gdn" else f"attention step at position {ctx - 1}"
    return (n / L) / t_total, (f"{n} single-sequence layer {what}(s) through the oracle in {t_total:.1f} s on one "
                               f"thread, time scaled to {L} layers")


def run_hybrid(args):
    """A decode token through the hybrid stack's DeltaNet (gdn80) or attention (gqa80_8k) layers.
    Each step is one CUDA-graph replay of the L layer launches. DeltaNet: the 72 MiB of state fit
    in L2, so a 256 MiB buffer is written between timed steps (outside the timed events); the
    write-back of that buffer's dirty lines then competes with the step's reads, which makes the
    figure conservative. Attention: the 384 MiB of cache exceed L2; no flush."""
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from int4_routed_expert_05_b300 import _build
    _build.build()
    kind, L, ctx = HYBRID[args.config]
    _, _, _, desc = CONFIGS[args.config]
    batch = args.batch
    n_e2e = max(1, min(args.steps, 200))
    n_total = args.warmup + args.steps + 1 + n_e2e  # attention: one cache position per step
    if kind == "gqa" and n_total >= ctx:
        raise SystemExit(f"warmup + steps must stay below the {ctx}-position context")
    W = _hybrid_setup(kind, L, batch, ctx, n_total)
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")  # 256 MiB > 126 MB L2

    # one graph per distinct input set (the graph holds the pointers of its inputs)
    graphs = []
    with torch.cuda.stream(stream):
        _hybrid_step(W, 0, sp)  # first launch outside capture (sets kernel attributes)
        if kind == "gqa":
            W["pos"] += 1
    torch.cuda.synchronize()
    for s in range(len(W["inp"])):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            _hybrid_step(W, s, torch.cuda.current_stream().cuda_stream)
        graphs.append(g)
    torch.cuda.synchronize()

    def replay(i):
        graphs[i % len(graphs)].replay()
        if kind == "gqa":
            W["pos"] += 1  # on the same stream, after the step

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            replay(i)
    torch.cuda.synchronize()
    if kind == "gqa" and int(W["status"][0].item()) != 0:
        raise RuntimeError(f"device status {int(W['status'][0].item())} after warm-up")

    clocks = ClockSampler(local)
    _barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    pos_sum = 0
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            if kind == "gdn":
                flush.fill_(float(i))
            ev[i][0].record(stream)
            replay(args.warmup + i)
            ev[i][1].record(stream)
            pos_sum += (W["start"] + 1 + args.warmup + i) if kind == "gqa" else 0
    torch.cuda.synchronize()
    _barrier(ws)
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev)
    ms = _max_over_ranks(ws, ms)
    if kind == "gqa" and int(W["status"][0].item()) != 0:
        raise RuntimeError(f"device status {int(W['status'][0].item())} after the timed region")

    # end to end: every step's inputs (all layers, one packed buffer) from pinned host memory, the
    # last layer's y back
    h_flat = torch.empty_like(W["flat"], device="cpu").pin_memory()
    h_flat.copy_(W["flat"])
    h_y = torch.empty_like(W["y"], device="cpu").pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            W["flat"].copy_(h_flat, non_blocking=True)
            replay(0)
            h_y.copy_(W["y"], non_blocking=True)
            stream.synchronize()
    e2e_s = _max_over_ranks(ws, time.perf_counter() - t0)

    if rank != 0:
        return
    ms_step = ms / args.steps
    launches_per_step = L * (1 if kind == "gdn" else 2)
    if kind == "gdn":
        bytes_step = W["bytes_per_launch"] * L
        dom, per_launch = "gdn_step_kernel", W["bytes_per_launch"]
    else:
        # mean position over the timed steps: rows 0..p read per layer
        mean_rows = pos_sum / args.steps
        per_launch = W["kv_row_bytes"] * mean_rows + W["io_bytes"]
        bytes_step = per_launch * L
        dom = "gqa_split_kernel"
    peak, peak_kind = _peaks()
    achieved = bytes_step / (ms_step / 1e3) / 1e9
    traffic = None  # DRAM bytes of one launch of the dominant kernel, from an ncu capture (profiles/)
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp) and batch == 1:
        t = json.load(open(tp)).get(args.config)
        traffic = t.get("bytes_per_launch") if t else None
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    cpu_v, cpu_info = (None, None)
    if ws == 1 and not args.no_cpu_baseline:
        cpu_v, cpu_info = cpu_oracle_hybrid(kind, L, ctx, budget_s=args.ref_budget)
    line = {
        "metric": f"{'Gated DeltaNet' if kind == 'gdn' else 'gated GQA'} decode tokens/s through {L} layers "
                  "(1 B300) and HBM GB/s vs the measured copy roofline",
        "value": ws * batch * args.steps / (ms / 1e3), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (bf16 inputs)",
        "data": "synthetic (seeded generator, random-init parameters of the stated shapes)",
        "config": {"workload": args.config, "description": desc, "batch": batch, "layers": L,
                   "context": ctx if kind == "gqa" else None,
                   "l2": ("256 MiB written between timed steps, outside the timed events" if kind == "gdn" else
                          "inputs larger than L2 (%.0f MiB of K/V cache vs 126 MB L2)" % (
                              L * W["kv_row_bytes"] * ctx / 2 ** 20 if kind == "gqa" else 0)),
                   "graphs": "each step is one CUDA-graph replay of the layers' launches",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "layer_latency_us": ms_step * 1e3 / L,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_kind": peak_kind, "kernel": dom, "bytes_per_launch": per_launch,
                     "note": "launch duration = step time / layers (graph replay, gaps included)"},
        "cpu_baseline": None if cpu_v is None else {"value": cpu_v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                                    "sample": cpu_info},
        "e2e": {"value": ws * batch * n_e2e / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": W["flat"].numel(), "d2h_bytes_per_step": W["y"].numel() * 4,
                "steps": n_e2e},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def cpu_oracle_batched(sh, T, seed=SEED, budget_s=15.0):
    """The oracle, single-threaded, on a sample of the batch: whole layers token by token until the
    budget is spent (at most T tokens); tokens/s of one layer."""
    import oracle
    from int4_routed_expert_05_b300 import synth
    from oracle.layers import OracleLayers
    O = OracleLayers(oracle, sh, seed, 1)
    xb = synth.activation_bits(sh, seed, 1000, min(T, 64))
    t_total, n = 0.0, 0
    while n < min(T, 64) and (n == 0 or t_total < budget_s):
        lg, _ = oracle.router_logits(O.dense(0)[0], xb[n])
        for e in oracle.topk(lg, sh.top_k, sh.renorm)[0]:
            O.blob(0, int(e))
        t0 = time.perf_counter()
        O.layer(0, xb[n])
        t_total += time.perf_counter() - t0
        n += 1
    return n / t_total, f"{n} of the {T} tokens through the oracle layer in {t_total:.1f} s"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="stack80", choices=sorted(CONFIGS))
    ap.add_argument("--ref-layers", type=int, default=2)
    ap.add_argument("--ref-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graphs", action="store_true", help="batched workloads: time direct calls, not graph replays")
    ap.add_argument("--pool-gib", type=float, default=0.0, help="bounded pool: size in GiB (default: the config's)")
    ap.add_argument("--zipf-beta", type=float, default=None,
                    help="bounded pool: fixed routing-popularity strength instead of the calibrated one")
    ap.add_argument("--qpack", default="",
                    help="bounded pool: read the misses from an expert container written to this path "
                         "(instead of the pinned host store)")
    ap.add_argument("--prefetch", type=int, default=6,
                    help="bounded pool: copy ahead the next layer's N best predicted experts (0: off; default 6, the best of a 2 GiB sweep)")
    ap.add_argument("--batch", type=int, default=1, help="hybrid workloads: independent sequences per step")
    ap.add_argument("--gemv", action="store_true",
                    help="batched workloads with T <= 64: the matrix-vector expert path (MOE_GEMV)")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the stack (small cases for profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.config in POOL_SLOTS:
        run_streamed(args)
    elif args.config in BATCHED:
        run_batched(args)
    elif args.config in HYBRID:
        run_hybrid(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
