#!/usr/bin/env python3
"""Benchmark of the 4-bit MoE layer on GB300.

Headline workload (one JSON line on rank 0): batch-1 decode through 40
independent MoE layers of the Qwen3.6-35B-A3B-style shape (d_model 2048, 256
experts, top-8, d_ff 512, one shared expert, group-64 affine 4-bit weights;
distinct seeded weights per layer, ~18 GB resident so L2 cannot hold them),
a fresh token per layer per step. One step = one token through all 40 layers
(router GEMV + top-8, gate/up GEMV + SwiGLU, down GEMV + weighted combine for
the 8 routed and the shared expert). metric = tokens/s.

The same line carries the prefill configurations (T = 64, 512, 4096, 32768 with a
Zipf router bias) under "prefill", each with its own tensor-pipe roofline.

--impl reference times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (batch-1 decode, 40 layers) at 1 GB300 + % roofline"
N_LAYERS = 40
SELECTED_BYTES_PER_LAYER = 9 * 1_769_472      # 8 routed + shared expert: q + scale + bias
ROUTER_BYTES_PER_LAYER = 2048 * 256 * 4 + 2048 * 4  # fp32 router and shared-gate weights
DECODE_BYTES_PER_LAYER = SELECTED_BYTES_PER_LAYER + ROUTER_BYTES_PER_LAYER
FLOP_PER_TOKEN = 9 * 3 * 2 * 2048 * 512        # 56,623,104


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill configurations")
    ap.add_argument("--no-batch-decode", action="store_true",
                    help="skip the small-batch decode lines (T = 2, 4, 8 tokens per layer)")
    ap.add_argument("--prefill-iters", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gdn", action="store_true", help="skip the Gated DeltaNet scan lines")
    ap.add_argument("--no-attn", action="store_true", help="skip the decode-attention lines")
    ap.add_argument("--profile", choices=["decode", "prefill", "prefill-det", "prefill-fused",
                                          "decode-batch", "attn", "gdn"],
                    help="no measurement: run one layer repeatedly (decode: 20 + 200 calls; prefill: "
                         "3 forwards at --profile-T tokens; prefill-det / prefill-fused: the same "
                         "with MOE_FWD_DETERMINISTIC / MOE_FWD_FUSED; decode-batch: 8 calls at each "
                         "of T = 2, 4, 8; attn: 4 decode-attention calls over 32768 cached "
                         "positions; gdn: 4 Gated DeltaNet scans over 4096 tokens) for a profiler to attach to")
    ap.add_argument("--profile-T", type=int, default=4096)
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world):
    import torch
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            m = json.load(f)
        return dict(hbm_gbs=float(m["hbm_gbs"]), bf16=float(m["bf16_tflops"]),
                    bf16_sustained=float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                    sm_max_mhz=float(m.get("sm_max_mhz", 2070.0)), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, sm_max_mhz=2070.0,
                    source="fallback")


# ------------------------------------------------------------------ helpers
def gpu_graph(fn, stream):
    """Capture fn() (a sequence of library calls) into a CUDA graph on `stream`."""
    import torch
    with torch.cuda.stream(stream):
        fn()  # warm-up outside capture (sets kernel attributes, loads modules)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def timed_replays(g, stream, iters, flush):
    """Per-iteration device time of a graph replay, L2 flushed before each one.
    The flush is enqueued before the start event, so it also keeps the GPU busy
    while the replay is being issued."""
    import torch
    times = []
    with torch.cuda.stream(stream):
        for _ in range(iters):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            times.append((e0, e1))
    stream.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in times]


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ------------------------------------------------------------------ decode (headline)
def decode_layers(shape, seed, n_layers, keep_host):
    from bit_moe_expert_route_gb300 import ops, synth
    layers, decs, hosts = [], [], []
    for l in range(n_layers):
        host = synth.layer_weights(shape, seed=seed, layer=l)
        dl = ops.DeviceLayer(host, shape)
        layers.append(dl)
        decs.append(ops.Decode(dl))
        if l < keep_host:
            hosts.append(host)
    return layers, decs, hosts


def run_decode(args, world, peaks):
    import numpy as np
    import torch
    from bit_moe_expert_route_gb300 import synth
    shape = synth.LayerShape()
    d, L = shape.d_model, N_LAYERS
    keep = 0 if args.no_cpu_baseline or world > 1 else 2
    layers, decs, hosts = decode_layers(shape, seed=0, n_layers=L, keep_host=keep)
    nsteps = args.warmup + args.steps
    x_host = torch.empty(nsteps, L, d, dtype=torch.int16).pin_memory()
    for l in range(L):
        xs = synth.tokens(shape, nsteps, seed=0, layer=l, tensor=synth.X_DECODE)
        x_host[:, l].copy_(torch.from_numpy(xs.view(np.int16)))
    x_dev = x_host.cuda()
    x_stage = torch.empty(L, d, dtype=torch.int16, device="cuda")
    out_stage = torch.empty(L, d, dtype=torch.int16, device="cuda")
    out_host = torch.empty(nsteps, L, d, dtype=torch.int16).pin_memory()
    stream = torch.cuda.Stream()

    def step():
        for l in range(L):
            decs[l](x_stage[l], out_stage[l].view(torch.bfloat16))

    g = gpu_graph(step, stream)
    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            x_stage.copy_(x_dev[s], non_blocking=True)
            g.replay()
    stream.synchronize()

    # device-resident inputs: K steps between two events
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for s in range(args.warmup, nsteps):
            x_stage.copy_(x_dev[s], non_blocking=True)
            g.replay()
        e1.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    barrier(world)
    t_dev = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world)

    # end to end: pinned host input -> device, layers, device -> pinned host output
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for s in range(args.warmup, nsteps):
            x_stage.copy_(x_host[s], non_blocking=True)
            g.replay()
            out_host[s].copy_(out_stage, non_blocking=True)
        f1.record(stream)
    stream.synchronize()
    t_e2e = max_over_ranks(f0.elapsed_time(f1) * 1e-3, world)
    assert bool(torch.isfinite(out_stage.view(torch.bfloat16).float()).all())

    K = args.steps
    step_s = t_dev / K
    # algorithmic bytes: the 9 selected experts' codes, scales and biases per
    # layer; the fp32 router and shared-gate weights are reported beside it
    achieved = L * SELECTED_BYTES_PER_LAYER / step_s / 1e9
    achieved_all = L * DECODE_BYTES_PER_LAYER / step_s / 1e9
    res = dict(
        value=world * K / t_dev, ms_per_step=step_s * 1e3,
        e2e=dict(value=world * K / t_e2e, unit="tokens/s", h2d_bytes_per_step=L * d * 2,
                 d2h_bytes_per_step=L * d * 2),
        gpu_launches=L * K,  # one decode kernel per layer
        roofline=dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"],
                      unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4),
                      traffic=TRAFFIC.get("decode_layer"),
                      kernel="decode_layer_kernel: router GEMV + top-8 + gate/up GEMV + SwiGLU + "
                             "down GEMV + weighted combine, one launch per layer",
                      bytes_per_layer=SELECTED_BYTES_PER_LAYER,
                      router_bytes_per_layer=ROUTER_BYTES_PER_LAYER,
                      achieved_incl_router=round(achieved_all, 1),
                      us_per_layer=round(step_s / L * 1e6, 3),
                      peak_source=peaks["source"]),
        clocks=clk,
    )
    if keep:
        res["cpu_baseline"] = decode_cpu_baseline(hosts, shape)
    del decs, g
    if not args.no_batch_decode:
        res["decode_batch"] = [run_decode_batch(layers, shape, T, stream, peaks) for T in (2, 4, 8)]
    del layers
    torch.cuda.empty_cache()
    return res


# Gated DeltaNet layer shape (a reading: the pages give no sizes; 16 key/query heads
# and 32 value heads of 128, as in the public Qwen3-Next-style configuration with
# d_model 2048); the model has 30 such layers.
GDN_SHAPE = dict(Hk=16, Hv=32, dk=128, dv=128)
GDN_LAYERS = 30


def run_gdn(args, peaks):
    """moe_gdn_scan on seeded synthetic inputs (unit-norm bf16 q and k, N(0,1) bf16 v,
    alpha in [0.8, 1), beta in [0, 1), fp32 state): prefill, one scan over T = 4096
    tokens; decode, one token through each of 30 layers (distinct states) captured in one
    CUDA graph, each launch reading its layer's state before waiting for the previous
    layer (MOE_GDN_STATE_EARLY). L2 flushed before every timed replay."""
    import torch
    from bit_moe_expert_route_gb300 import ops
    Hk, Hv, dk, dv = (GDN_SHAPE[n] for n in ("Hk", "Hv", "dk", "dv"))
    gen = torch.Generator(device="cuda").manual_seed(0)
    stream = torch.cuda.Stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def make(T):
        def unit(*shape):
            a = torch.randn(*shape, device="cuda", generator=gen)
            return (a / a.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        q, k = unit(T, Hk, dk), unit(T, Hk, dk)
        v = torch.randn(T, Hv, dv, device="cuda", generator=gen).to(torch.bfloat16)
        al = 0.8 + 0.2 * torch.rand(T, Hv, device="cuda", generator=gen)
        be = torch.rand(T, Hv, device="cuda", generator=gen)
        S = 0.1 * torch.randn(Hv, dv, dk, device="cuda", generator=gen)
        return q, k, v, al, be, S, torch.empty(T, Hv, dv, device="cuda")

    T = 4096
    q, k, v, al, be, S, out = make(T)
    g = gpu_graph(lambda: ops.gdn_scan(q, k, v, al, be, S, out=out), stream)
    for _ in range(3):
        g.replay()
    t_pre = statistics.median(timed_replays(g, stream, args.prefill_iters, flush))
    flop = 6 * T * Hv * dv * dk  # three multiply-adds per state entry per token
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    fp32_peak = sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
    state_bytes = Hv * dv * dk * 4
    layers = [make(1) for _ in range(GDN_LAYERS)]

    def step():
        for lq, lk, lv, la, lb, lS, lo in layers:
            ops.gdn_scan(lq, lk, lv, la, lb, lS, out=lo, state_early=True)
    gd = gpu_graph(step, stream)
    for _ in range(3):
        gd.replay()
    t_dec = statistics.median(timed_replays(gd, stream, args.prefill_iters, flush)) / GDN_LAYERS
    dec_gbs = 2 * state_bytes / t_dec / 1e9
    del g, gd, layers, flush
    torch.cuda.empty_cache()
    return dict(
        shape=dict(GDN_SHAPE, layers=GDN_LAYERS),
        prefill=dict(T=T, ms=round(t_pre * 1e3, 4), tokens_per_s=round(T / t_pre, 1),
                     roofline=dict(bound="alu", achieved=round(flop / t_pre / 1e12, 2),
                                   peak=round(fp32_peak, 1), unit="TFLOP/s",
                                   frac=round(flop / t_pre / 1e12 / fp32_peak, 4),
                                   flop_per_token=6 * Hv * dv * dk,
                                   kernel="gdn_scan_kernel: each state row in the registers of 8 "
                                          "lanes (4 rows per warp) for all T tokens; one butterfly "
                                          "per token",
                                   peak_source="SM count x 128 fp32 lanes x 2 x max SM clock")),
        decode=dict(us_per_layer=round(t_dec * 1e6, 3),
                    tokens_per_s_30_layers=round(1 / (t_dec * GDN_LAYERS), 1),
                    roofline=dict(bound="hbm", achieved=round(dec_gbs, 1), peak=peaks["hbm_gbs"],
                                  unit="GB/s", frac=round(dec_gbs / peaks["hbm_gbs"], 4),
                                  bytes_per_layer=2 * state_bytes,
                                  kernel="gdn_scan_kernel at T = 1: the state read and written "
                                         "once per layer")),
        gpu_launches_per_decode_step=GDN_LAYERS,
        l2="flushed (512 MB write) before every timed replay",
    )


# Decode attention with grouped KV heads (a reading: the pages give no sizes;
# 16 query heads, 2 KV heads of 256, as in the public Qwen3-Next-style
# configuration); the model has 10 such layers.
ATTN_SHAPE = dict(Hq=16, Hkv=2, d=256)
ATTN_LAYERS = 10


def run_attn(args, peaks):
    """moe_decode_attention on seeded bf16 q, K, V ~ N(0, 1): one new token over a
    cache of L positions, L = 4096 and 32768; 10 layers (distinct caches) in one
    CUDA graph, L2 flushed before every replay. Bound: HBM, for the K and V bytes
    read once (2 * L * Hkv * d * 2 per layer)."""
    import torch
    from bit_moe_expert_route_gb300 import ops
    Hq, Hkv, d = ATTN_SHAPE["Hq"], ATTN_SHAPE["Hkv"], ATTN_SHAPE["d"]
    gen = torch.Generator(device="cuda").manual_seed(0)
    stream = torch.cuda.Stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    res = []
    for L in (4096, 32768):
        layers = []
        for _ in range(ATTN_LAYERS):
            q = torch.randn(Hq, d, device="cuda", generator=gen).to(torch.bfloat16)
            K = torch.randn(L, Hkv, d, device="cuda", generator=gen).to(torch.bfloat16)
            V = torch.randn(L, Hkv, d, device="cuda", generator=gen).to(torch.bfloat16)
            out = torch.empty(Hq, d, dtype=torch.float32, device="cuda")
            nbytes = ops.lib().moe_decode_attention_workspace_bytes(L, Hq, Hkv, d)
            ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            layers.append((q, K, V, out, ws))

        def step():
            for q, K, V, out, ws in layers:
                ops.decode_attention(q, K, V, out=out, ws=ws)
        g = gpu_graph(step, stream)
        for _ in range(3):
            g.replay()
        t = statistics.median(timed_replays(g, stream, args.prefill_iters, flush)) / ATTN_LAYERS
        kv = 2 * L * Hkv * d * 2
        gbs = kv / t / 1e9
        res.append(dict(L=L, us_per_layer=round(t * 1e6, 3),
                        roofline=dict(bound="hbm", achieved=round(gbs, 1), peak=peaks["hbm_gbs"],
                                      unit="GB/s", frac=round(gbs / peaks["hbm_gbs"], 4),
                                      bytes_per_layer=kv,
                                      kernel="attn_split_kernel + attn_combine_kernel: all query "
                                             "heads of a KV head per block, each K/V row read once")))
        del layers, g
    del flush
    torch.cuda.empty_cache()
    return dict(shape=dict(ATTN_SHAPE, layers=ATTN_LAYERS), configs=res,
                gpu_launches_per_step=2 * ATTN_LAYERS,
                l2="flushed (512 MB write) before every timed replay")


EXPERT_BYTES = 1_769_472       # one expert's packed codes, scales and biases (3 projections)
ROUTER_BYTES = 2_105_344       # fp32 router [2048][256] and w_sg


def run_decode_batch(layers, shape, T, stream, peaks, steps=50, warmup=5):
    """T tokens per layer through the same 40 layers (moe_decode_batch_w4,
    PDL-chained in one CUDA graph), fresh tokens each step; bytes per layer
    count every distinct selected expert once, plus the shared expert and
    the router."""
    import numpy as np
    import torch
    from bit_moe_expert_route_gb300 import ops, synth
    d, L = shape.d_model, len(layers)
    decs = [ops.DecodeBatch(dl, T) for dl in layers]
    n = warmup + steps
    xs = torch.empty(n, L, T, d, dtype=torch.int16)
    for l in range(L):
        v = synth.tokens(shape, n * T, seed=1, layer=l, tensor=synth.X_DECODE)
        xs[:, l].copy_(torch.from_numpy(v.view(np.int16)).view(n, T, d))
    x_dev = xs.cuda()
    x_stage = torch.empty(L, T, d, dtype=torch.int16, device="cuda")
    out = torch.empty(L, T, d, dtype=torch.bfloat16, device="cuda")

    def step():
        for l in range(L):
            decs[l](x_stage[l], out[l])

    g = gpu_graph(step, stream)
    with torch.cuda.stream(stream):
        for s in range(warmup):
            x_stage.copy_(x_dev[s], non_blocking=True)
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for s in range(warmup, n):
            x_stage.copy_(x_dev[s], non_blocking=True)
            g.replay()
        e1.record(stream)
    stream.synchronize()
    t = e0.elapsed_time(e1) * 1e-3
    ids = [torch.unique(dec.view("topk_ids", (T, shape.top_k), torch.int32)).numel() for dec in decs]
    bytes_layer = float(np.mean(ids)) * EXPERT_BYTES + EXPERT_BYTES + ROUTER_BYTES
    step_s = t / steps
    achieved = L * bytes_layer / step_s / 1e9
    del decs, g
    return dict(T=T, tokens_per_s=round(T * steps / t, 1), ms_per_step=round(step_s * 1e3, 4),
                us_per_layer=round(step_s / L * 1e6, 2), distinct_experts_per_layer=round(float(np.mean(ids)), 2),
                roofline=dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                              frac=round(achieved / peaks["hbm_gbs"], 4), bytes_per_layer=int(bytes_layer),
                              kernel="moe_decode_batch_w4: router, top-k + gate/up, down: 3 PDL-chained "
                                     "launches per layer"),
                gpu_launches=3 * L * steps)


def oracle_decode_steps(hosts, shape, steps, first_step=0):
    """The oracle on `steps` decode steps: each step is one token through 40
    layers, every one of the 40 layer evaluations really computed, the layers'
    weights cycled over the `hosts` sample (a sample of weights, not of work).
    The evaluations that share a layer's weights go to the oracle as one batch
    (OpenMP over tokens, all host cores). Returns (wall seconds, evaluations)."""
    import numpy as np
    from bit_moe_expert_route_gb300 import synth
    from oracle import Oracle
    orc = Oracle()
    n_host = len(hosts)
    evals = steps * N_LAYERS
    per_host = [[] for _ in range(n_host)]
    for i in range(evals):
        s, l = divmod(i, N_LAYERS)
        per_host[l % n_host].append((first_step + s, l))
    xs = []
    for h in range(n_host):
        if not per_host[h]:
            xs.append(None)
            continue
        rows = [synth.tokens(shape, 1, seed=0, layer=l, off=s, tensor=synth.X_DECODE)
                for s, l in per_host[h]]
        xs.append(np.ascontiguousarray(np.concatenate(rows)))
    t0 = time.perf_counter()
    for h in range(n_host):
        if xs[h] is not None:
            orc.moe_forward(xs[h], hosts[h], shape)
    return time.perf_counter() - t0, evals


def omp_threads():
    return int(os.environ.get("OMP_NUM_THREADS", "0")) or (os.cpu_count() or 1)


def decode_cpu_baseline(hosts, shape, steps=10):
    """The oracle on a bounded sample of the decode workload (the same method as
    the reference arm): `steps` steps of one token through 40 layers."""
    wall, evals = oracle_decode_steps(hosts, shape, steps)
    return dict(value=round(steps / wall, 4), unit="tokens/s", cores=omp_threads(), kind="oracle",
                cpu=cpu_model(),
                sample=f"{steps} decode steps x {N_LAYERS} layer evaluations ({evals}, all computed), "
                       f"layer weights cycled over {len(hosts)} seeded layers; oracle fp64, OpenMP "
                       f"over tokens; {wall:.1f} s")


def prefill_cpu_baseline(host, shape, T, zipf, n_sample):
    """The oracle on `n_sample` of the T tokens (the first ones; tokens are
    independent, so the rate scales): tokens/s."""
    from bit_moe_expert_route_gb300 import synth
    from oracle import Oracle
    orc = Oracle()
    n = min(T, n_sample)
    x = synth.tokens(shape, T, seed=0)[:n]
    h = dict(host, router_bias=synth.zipf_router_bias(shape.n_experts) if zipf else None)
    t0 = time.perf_counter()
    orc.moe_forward(x, h, shape)
    wall = time.perf_counter() - t0
    return dict(value=round(n / wall, 2), unit="tokens/s", cores=omp_threads(), kind="oracle",
                cpu=cpu_model(),
                sample=f"{n} of the {T} tokens (router, top-8, 8 routed + shared experts per token), "
                       f"oracle fp64, OpenMP over tokens; {wall:.1f} s")


# ------------------------------------------------------------------ prefill configurations
def run_prefill(T, zipf, host0, args, peaks):
    import numpy as np
    import torch
    from bit_moe_expert_route_gb300 import ops, synth
    shape = synth.LayerShape()
    E, k, d, f = shape.n_experts, shape.top_k, shape.d_model, shape.d_ff
    host = dict(host0, router_bias=synth.zipf_router_bias(E) if zipf else None)
    dl = ops.DeviceLayer(host, shape)
    fwd = ops.Forward(dl, T)
    x = torch.from_numpy(synth.tokens(shape, T, seed=0).view(np.int16)).cuda()
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")  # > L2 (129 MB)
    g = gpu_graph(lambda: fwd(x, out), stream)
    for _ in range(3):
        g.replay()
    t_layer = statistics.median(timed_replays(g, stream, args.prefill_iters, flush))

    rows = T * k + T
    mt, bn = fwd.views.max_tiles, fwd.block_n
    bm = fwd.view("block_map", (mt, 4), torch.int32)
    nt = fwd.view("num_tiles", (1,), torch.int32)
    rt = fwd.view("row_token", (rows,), torch.int32)
    # the layer's own operands: x as f16 (written by the router kernel) and f16 h
    x16 = fwd.view("x16", (T, d), torch.float16)
    h = fwd.view("h", (rows, f), torch.float16)
    rw = fwd.view("row_weight", (rows,), torch.float32)
    acc = fwd.view("out_acc", (T, d), torch.float32)
    t = dl.t
    # the down projection runs on its own (taller) tile map at large T, and
    # gate/up joins it from 512 rows per expert (as the forward does)
    mt2, bn2 = fwd.views.down_max_tiles, fwd.views.down_block_n
    bm2 = fwd.view("down_block_map", (mt2, 4), torch.int32)
    nt2 = fwd.view("down_num_tiles", (1,), torch.int32)
    tall = bn2 == 256 and T * k >= 512 * E
    gu = (bm2, nt2, mt2, bn2) if tall else (bm, nt, mt, bn)
    g1 = gpu_graph(lambda: ops.grouped_gemm_w4a16(
        x16, [t["gate"], t["up"]], E, f, gu[0], gu[1], gu[2], gu[3], ops.EPI_SWIGLU, row_index=rt,
        n_rows=rows, W_extra=[t["sh_gate"], t["sh_up"]], C=h), stream)
    g2 = gpu_graph(lambda: ops.grouped_gemm_w4a16(
        h, [t["down"]], E, d, bm2, nt2, mt2, bn2, ops.EPI_COMBINE, n_rows=rows,
        W_extra=[t["sh_down"]], row_scale=rw, out_row=rt, C=acc), stream)
    t1 = statistics.median(timed_replays(g1, stream, args.prefill_iters, flush))
    t2 = statistics.median(timed_replays(g2, stream, args.prefill_iters, flush))
    # the same layer with MOE_FWD_DETERMINISTIC (fixed-order combine)
    fwd_det = ops.Forward(dl, T, deterministic=True)
    gd = gpu_graph(lambda: fwd_det(x, out), stream)
    for _ in range(3):
        gd.replay()
    t_det = statistics.median(timed_replays(gd, stream, args.prefill_iters, flush))
    del gd, fwd_det
    # the fused chain (MOE_FWD_FUSED: gate/up, SwiGLU and down per 64-row tile, h on chip)
    fwd_fused = ops.Forward(dl, T, fused=True)
    gf = gpu_graph(lambda: fwd_fused(x, out), stream)
    for _ in range(3):
        gf.replay()
    t_fused = statistics.median(timed_replays(gf, stream, args.prefill_iters, flush))
    del gf, fwd_fused
    f1 = 2 * 2 * d * f * rows
    f2 = 2 * f * d * rows
    achieved = (f1 + f2) / (t1 + t2) / 1e12
    counts = fwd.view("counts", (E,), torch.int32).cpu().numpy()
    weight_bytes = 257 * 1_769_472
    res = dict(
        T=T, router_bias="zipf 1.5*ln(1/rank)" if zipf else None, block_n=bn, gateup_block_n=gu[3],
        down_block_n=bn2,
        tokens_per_s=round(T / t_layer, 1), ms=round(t_layer * 1e3, 4),
        deterministic_ms=round(t_det * 1e3, 4),
        fused_chain_ms=round(t_fused * 1e3, 4),
        fused_chain_frac_of_bf16_peak=round(FLOP_PER_TOKEN * T / t_fused / 1e12 / peaks["bf16"], 4),
        layer_tflops=round(FLOP_PER_TOKEN * T / t_layer / 1e12, 2),
        layer_frac_of_bf16_peak=round(FLOP_PER_TOKEN * T / t_layer / 1e12 / peaks["bf16"], 4),
        weights_hbm_frac=round(weight_bytes / t_layer / 1e9 / peaks["hbm_gbs"], 4),
        gpu_launches=7,
        roofline=dict(bound="tensor", achieved=round(achieved, 1), peak=peaks["bf16"],
                      unit="TFLOP/s", frac=round(achieved / peaks["bf16"], 4),
                      traffic=TRAFFIC.get(f"gemm_T{T}"),
                      kernel="grouped W4A16 GEMMs (gate/up+SwiGLU, down+combine)",
                      gateup_ms=round(t1 * 1e3, 4), down_ms=round(t2 * 1e3, 4),
                      flop_per_token=FLOP_PER_TOKEN, peak_source=peaks["source"]),
        expert_counts=dict(min=int(counts.min()), max=int(counts.max()),
                           zero=int((counts == 0).sum()), mean=float(counts.mean())),
        l2="flushed (512 MB write) before every timed iteration",
    )
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = prefill_cpu_baseline(host0, shape, T, zipf, 256)
    del g, g1, g2, fwd, dl
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ reference arm (CPU oracle)
def reference_arm(args):
    """The oracle, as it stands, on the host cores, on the headline workload: each
    step is one decode token through 40 layers, every layer evaluation computed
    (the weights cycled over 4 seeded layers); the evaluations sharing a layer's
    weights run as one OpenMP batch over tokens. The same method as the GPU
    arm's cpu_baseline. Above 100 steps, each step evaluates a fixed sample of
    its 40 layers and the time is scaled to 40 (stated in `sample`)."""
    from bit_moe_expert_route_gb300 import synth
    shape = synth.LayerShape()
    n_host = 4
    hosts = [synth.layer_weights(shape, seed=0, layer=l) for l in range(n_host)]
    per_step = N_LAYERS if args.steps * N_LAYERS <= 4000 else max(1, 4000 // args.steps)
    scale = N_LAYERS / per_step

    def run(steps, first):
        if per_step == N_LAYERS:
            return oracle_decode_steps(hosts, shape, steps, first_step=first)
        # a fixed sample of each step's layers: evaluations 0..per_step-1 of every step
        import numpy as np
        from oracle import Oracle
        orc = Oracle()
        xs = [[] for _ in range(n_host)]
        for s_ in range(steps):
            for l in range(per_step):
                xs[l % n_host].append(synth.tokens(shape, 1, seed=0, layer=l, off=first + s_,
                                                   tensor=synth.X_DECODE))
        t0 = time.perf_counter()
        for h in range(n_host):
            if xs[h]:
                orc.moe_forward(np.ascontiguousarray(np.concatenate(xs[h])), hosts[h], shape)
        return time.perf_counter() - t0, steps * per_step

    run(args.warmup, 0)
    wall, evals = run(args.steps, args.warmup)
    wall_step = wall * scale / args.steps
    value = 1.0 / wall_step
    sample = (f"{args.steps} decode steps x {per_step} of {N_LAYERS} layer evaluations ({evals}, all "
              f"computed{'' if scale == 1 else f'; time scaled x{scale:g} to 40 layers'}), layer "
              f"weights cycled over {n_host} seeded layers; oracle fp64, OpenMP over tokens")
    return {
        "impl": "reference", "metric": BASELINE_METRIC, "value": round(value, 4),
        "unit": "tokens/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall_step * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": CONFIG,
        "cpu_baseline": dict(value=round(value, 4), unit="tokens/s", cores=omp_threads(),
                             kind="oracle", cpu=cpu_model(), sample=sample),
        "e2e": dict(value=round(value, 4), unit="tokens/s", h2d_bytes_per_step=0,
                    d2h_bytes_per_step=0),
    }


BASELINE_METRIC = "MoE-layer tokens/s (prefill T=512/4096/32768; batch-1 decode) at 1 GB300 + % roofline"
CONFIG = {
    "workload": "batch-1 decode: T=1 through 40 independent MoE layers (d_model 2048, 256 experts, "
                "top-8, d_ff 512, shared expert 512, group-64 affine 4-bit weights; distinct seeded "
                "weights per layer, ~18 GB resident), fresh token per layer per step",
    "layers": N_LAYERS, "tokens_per_step": 1, "l2": "weights (18 GB) larger than L2",
    "parallelism": "replicas",
}

# dram__bytes_read.sum + dram__bytes_write.sum per launch unit, from ncu captures of the
# current kernels summarised under profiles/: the decode kernel on one layer (cold
# cache: all of its weights come from HBM), and both grouped GEMMs of the third forward
# at T = 512, 4096 and 32768 (gate/up read + write, then down read + write). None where
# no capture of the current kernel exists.
TRAFFIC: dict = {
    "decode_layer": 18_125_824,
    "gemm_T512": 307_554_560 + 5_821_696 + 160_693_248 + 445_440,
    "gemm_T4096": 346_443_520 + 28_443_648 + 230_775_296 + 15_150_336,
    "gemm_T32768": 1_172_207_360 + 287_205_376 + 2_235_480_320 + 1_945_010_176,
}


def profile_run(args):
    """One layer of the seeded workload, run repeatedly with no timing: the target of the
    ncu commands recorded under profiles/."""
    import numpy as np
    import torch
    from bit_moe_expert_route_gb300 import ops, synth
    shape = synth.LayerShape()
    dl = ops.DeviceLayer(synth.layer_weights(shape, seed=0, layer=0), shape)
    if args.profile == "decode":
        dec = ops.Decode(dl)
        x = torch.from_numpy(synth.tokens(shape, 1, seed=1).view(np.int16)).cuda().view(-1)
        out = torch.empty(shape.d_model, dtype=torch.bfloat16, device="cuda")
        for _ in range(220):
            dec(x, out)
    elif args.profile == "attn":
        Hq, Hkv, d = ATTN_SHAPE["Hq"], ATTN_SHAPE["Hkv"], ATTN_SHAPE["d"]
        gen = torch.Generator(device="cuda").manual_seed(0)
        L = 32768
        q = torch.randn(Hq, d, device="cuda", generator=gen).to(torch.bfloat16)
        K = torch.randn(L, Hkv, d, device="cuda", generator=gen).to(torch.bfloat16)
        V = torch.randn(L, Hkv, d, device="cuda", generator=gen).to(torch.bfloat16)
        for _ in range(4):
            ops.decode_attention(q, K, V)
    elif args.profile == "gdn":
        Hk, Hv, dk, dv = (GDN_SHAPE[n] for n in ("Hk", "Hv", "dk", "dv"))
        gen = torch.Generator(device="cuda").manual_seed(0)
        T = 4096

        def unit(*shp):
            a = torch.randn(*shp, device="cuda", generator=gen)
            return (a / a.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        q, k = unit(T, Hk, dk), unit(T, Hk, dk)
        v = torch.randn(T, Hv, dv, device="cuda", generator=gen).to(torch.bfloat16)
        al = 0.8 + 0.2 * torch.rand(T, Hv, device="cuda", generator=gen)
        be = torch.rand(T, Hv, device="cuda", generator=gen)
        S = 0.1 * torch.randn(Hv, dv, dk, device="cuda", generator=gen)
        for _ in range(4):
            ops.gdn_scan(q, k, v, al, be, S)
    elif args.profile == "decode-batch":
        for T in (2, 4, 8):
            dec = ops.DecodeBatch(dl, T)
            x = torch.from_numpy(synth.tokens(shape, T, seed=1, tensor=synth.X_DECODE).view(np.int16)).cuda()
            for _ in range(8):
                dec(x)
    else:
        T = args.profile_T
        fwd = ops.Forward(dl, T, deterministic=args.profile == "prefill-det",
                          fused=args.profile == "prefill-fused")
        x = torch.from_numpy(synth.tokens(shape, T, seed=0).view(np.int16)).cuda()
        for _ in range(3):
            fwd(x)
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "ok": True}), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return 0
    import torch
    torch.cuda.set_device(local)
    dist_init(world)
    from bit_moe_expert_route_gb300 import build as B
    if rank == 0 and not B.up_to_date():
        B.build()
    barrier(world)
    if args.profile:
        profile_run(args)
        return 0
    peaks = measured_peaks()
    res = run_decode(args, world, peaks)
    prefill = []
    if not args.no_prefill:
        from bit_moe_expert_route_gb300 import synth
        host0 = synth.layer_weights(synth.LayerShape(), seed=0, layer=0)
        for T, zipf in ((64, False), (512, False), (4096, False), (32768, True)):
            prefill.append(run_prefill(T, zipf, host0, args, peaks))
    gdn = None if args.no_gdn else run_gdn(args, peaks)
    attn = None if args.no_attn else run_attn(args, peaks)
    line = {
        "metric": BASELINE_METRIC, "value": round(res["value"], 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(res["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "w4a16 (fp32 accumulate)",
        "data": "synthetic (seeded generators; random-init weights of the layer shape)",
        "config": CONFIG, "e2e": res["e2e"], "gpu_launches": res["gpu_launches"],
        "roofline": res["roofline"], "clocks": res["clocks"],
    }
    if "cpu_baseline" in res:
        line["cpu_baseline"] = res["cpu_baseline"]
    if "decode_batch" in res:
        line["decode_batch"] = res["decode_batch"]
    if prefill:
        line["prefill"] = prefill
    if gdn:
        line["gdn_scan"] = gdn
    if attn:
        line["decode_attention"] = attn
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)
    return 0


if __name__ == "__main__":
    sys.exit(main())
