#!/usr/bin/env python
"""Benchmark of the routed MoE expert FFN layer on GB300.

One step = one pass of the whole hot path over one batch: routing + aligned
prefix-sum endpoints + token scatter with input quantisation
(moe_route_scatter), grouped GEMM1, live-row SiLU*mul + e4m3/UE8M0 quant,
grouped GEMM2, top-k weighted combine, on the DeepSeek-style W4A8 layer
(E=32 experts, top-6, T=4096 tokens, hidden 4096, intermediate 2048, MXFP4
weights, capacity 28,672 rows). Synthetic seeded inputs; weights resident.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica of the layer on its own
GPU (the path has no exchange step on one GPU); value = routed rows of all
ranks / max-over-ranks time. `--impl reference` times the CPU oracle (the
plain restatement of the method) on the host cores on bounded samples of the
same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE FFN μs/layer & routed rows/s; act-quant μs; % of TC/HBM roofline"
UNIT = "routed rows/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extras", action="store_true")
    p.add_argument("--profile-kernel", choices=["route_scatter", "gemm1_act", "gemm2", "combine", "act_quant",
                                                  "kimi_layer", "kimi_route_scatter", "decode_fp8",
                                                  "decode_mxfp4", "decode_fp8_tc5", "decode_mxfp4_tc5"],
                   help="set up the layer, run one full step, then launch only this step's kernel "
                        "warmup + steps times and exit (for ncu captures); prints no JSON line. "
                        "act_quant launches the standalone live-row act-quant kernel at the "
                        "microbench shape (3,072 live of 28,672 rows, I = 2,048); kimi_layer runs "
                        "the Kimi-shaped layer warmup + steps times and prints its timings; "
                        "kimi_route_scatter launches only its routing + scatter (no weights); "
                        "decode_fp8 / decode_mxfp4 run the sparse decode over 2 layers on the mma.sync "
                        "path, the _tc5 forms on the tcgen05 path (T from --decode-tokens)")
    p.add_argument("--decode-tokens", type=int, default=1)
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def max_over_ranks(ms, pg, device="cuda"):
    """Length of a timed region over all ranks: each rank runs its own replica
    (no data-path collective), so the job takes as long as its slowest rank."""
    if not pg:
        return ms
    import torch
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(tt, op=pg.ReduceOp.MAX)
    return float(tt.item())


def whole_job_rate(world, units_per_step, steps, ms):
    """Units processed by all ranks per second over a region of `ms`
    milliseconds (weak scaling: every rank processes units_per_step)."""
    return world * units_per_step * steps / (ms / 1e3)


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("grouped_gemm.cu", "tcgen05.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "moe_expert_ffn_scatter_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or
    None when the kernel source changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(name)
    if not d or d.get("source_sha256_16") != kernel_source_hash():
        return None
    return d["dram_bytes_per_launch"]


def workload_config(cfg):
    return {"workload": cfg.name, "T": cfg.T, "E": cfg.E, "k": cfg.k, "H": cfg.H, "I": cfg.I, "A": cfg.A,
            "cap": cfg.cap, "routing": "softmax top-k, renormalised", "weights": "MXFP4 e2m1 + UE8M0 group 32",
            "activations": "e4m3 + UE8M0 group 128",
            "l2": "inputs larger than L2: about 0.9 GB touched per step (weights 0.43 GB, capacity buffers)"}


# ----------------------------------------------------------------- clocks
class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (the driver's
    libnvidia-ml, read-only queries) on a background thread every ~2 ms, so
    that even a timed region of a few milliseconds holds several samples.
    start()/stop() bracket the timed region itself."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, device):
        import ctypes
        import threading
        self.ct, self.threading = ctypes, threading
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        # the CUDA device's PCI address: NVML numbers the GPUs on its own
        import torch
        props = torch.cuda.get_device_properties(device)
        if all(hasattr(props, f) for f in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
            bus = b"%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h))
        else:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(int(device), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for device %d" % device)
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.rows, self.run, self.thread = [], False, None

    def _sample(self):
        ct = self.ct
        clk, mx, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        ok = self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0  # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.reasons_fn(self.h, ct.byref(rs))
        if ok:
            self.rows.append((clk.value, mx.value, rs.value))

    def _loop(self):
        while self.run:
            self._sample()
            time.sleep(0.002)

    def start(self):
        self.rows, self.run = [], True
        self.thread = self.threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        self.run = False
        self.thread.join()
        self._sample()  # at least one reading taken as the region ends
        self.lib.nvmlShutdown()
        sm = [r[0] for r in self.rows]
        reasons = sorted({n for r in self.rows for bit, n in self.REASONS.items() if r[2] & bit})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in self.rows),
                "reasons": reasons, "samples": len(self.rows), "source": "NVML, every ~2 ms inside the timed region"}


def clock_sampler(device):
    try:
        return NvmlClockSampler(device)
    except (OSError, AttributeError):
        return ClockSampler(device)


class ClockSampler:
    """Fallback: nvidia-smi every 20 ms; only the samples stamped inside the
    timed region count."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)  # nvidia-smi start-up; its samples before the region are dropped below
        self.t0 = time.time()

    def stop(self):
        t1 = time.time()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        import datetime
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if self.t0 <= ts <= t1:
                rows.append(parts[1:])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no sample inside the timed region"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "source": "nvidia-smi, every 20 ms inside the timed region"}


# ------------------------------------------------------------ CPU baseline
def oracle_sample(cfg, inp, n_tokens, seed=0):
    """Time the oracle (routing + the layer for n_tokens sampled tokens)."""
    import numpy as np
    import oracle as orc

    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(cfg.T, n_tokens, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    ids, w = orc.route_softmax_topk(inp.logits[toks], cfg.k)
    full_ids = np.zeros((cfg.T, cfg.k), np.int32)
    full_w = np.zeros((cfg.T, cfg.k), np.float32)
    full_ids[toks], full_w[toks] = ids, w
    orc.ffn_tokens(inp.x, full_ids, full_w, inp.w13, inp.w13_sf, inp.w2, inp.w2_sf, toks)
    return time.perf_counter() - t0


def cpu_baseline(cfg, inp, budget_s=15.0):
    import oracle as orc

    # the oracle spreads tokens over the host threads: calibrate on one round
    # of tokens per thread, then size the sample to about budget_s seconds
    nt = max(1, orc.num_threads())
    t1 = oracle_sample(cfg, inp, nt, seed=1)
    rounds = int(max(1, budget_s / max(t1, 1e-6)))
    n = int(min(cfg.T, nt * rounds))
    t = oracle_sample(cfg, inp, n, seed=2)
    return {"value": n * cfg.k / t, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
            "sample": "%d of %d tokens (%d routed rows) of the same layer: oracle routing + per-token "
                      "FFN (fp64 GEMMs) in %.2f s" % (n, cfg.T, n * cfg.k, t)}


def time_oracle(fn, min_s=1.0, max_reps=50):
    """Median wall time of fn() (the oracle, as it stands) over repetitions
    that together take about min_s seconds; returns (seconds, reps)."""
    t0 = time.perf_counter()
    fn()
    ts = [time.perf_counter() - t0]
    while sum(ts) < min_s and len(ts) < max_reps:
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
    return statistics.median(ts), len(ts)


def oracle_baseline(seconds, reps, unit_us, sample):
    import oracle as orc
    return {"value": unit_us(seconds), "unit": "us", "cores": orc.num_threads(), "kind": "oracle",
            "sample": "%s; median of %d runs" % (sample, reps)}


# --------------------------------------------------------------- reference
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from moe_expert_ffn_scatter_gb300 import synth
    import oracle as orc

    cfg = synth.DEEPSEEK
    inp = synth.ffn_inputs(cfg)
    nt = max(1, orc.num_threads())
    t1 = oracle_sample(cfg, inp, nt, seed=1)
    n = int(nt * max(1, int(4.0 / max(t1, 1e-6))))  # about 4 s of CPU work per step
    for i in range(args.warmup):
        oracle_sample(cfg, inp, n, seed=100 + i)
    times = [oracle_sample(cfg, inp, n, seed=1000 + i) for i in range(args.steps)]
    total = sum(times)
    value = args.steps * n * cfg.k / total
    conf = workload_config(cfg)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": conf,
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                             "sample": "%d tokens (%d routed rows) of %d per step" % (n, n * cfg.k, cfg.T)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours
def layer_parts(B, ctx, L, cfg, stream, x, logits, bias=None):
    """The layer's four launch groups as closures, in step order: route +
    scatter (3 kernels), GEMM1 with the fused SiLU*mul/quant epilogue, GEMM2,
    combine."""
    ld = L.a_sf.shape[1]

    def route_scatter():
        L.route_scatter(x, logits, bias, stream=stream)

    g2_format = L.w_format | (B.MOE_GEMM_A_GROUP32 if L.group == 32 else 0)

    def gemm1_act():
        B.moe_grouped_gemm_act_quant(ctx, L.a_fp8, L.a_sf, ld, L.expert_ends, cfg.E, cfg.A, cfg.cap, L.w13,
                                     L.w13_sf, L.gemm1_format, cfg.I, cfg.H, L.act_fp8, L.act_sf,
                                     kind=L.act_kind, limit=L.limit, stream=stream, situ=L.situ, group=L.group)

    def gemm2():
        B.moe_grouped_gemm(ctx, L.act_fp8, L.act_sf, ld, L.expert_ends, cfg.E, cfg.A, cfg.cap, L.w2, L.w2_sf,
                           g2_format, cfg.H, cfg.I, L.down, stream=stream)

    def combine():
        B.moe_combine(ctx, L.down, cfg.H, L.topk_w, L.src2dst, cfg.T, cfg.k, cfg.rsf, L.out, stream=stream)

    return {"route_scatter": route_scatter, "gemm1_act": gemm1_act, "gemm2": gemm2, "combine": combine}


def run_ours(args):
    import numpy as np
    import torch

    from moe_expert_ffn_scatter_gb300 import binding as B
    from moe_expert_ffn_scatter_gb300 import synth
    from moe_expert_ffn_scatter_gb300.layer import MoEFFNLayer

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if args.profile_kernel == "act_quant":
        profile_act_quant(args, B, synth, torch, np, local)
        return
    if args.profile_kernel and args.profile_kernel.startswith("decode_"):
        ctx = B.Context(local)
        wfmt = B.MOE_WFMT_FP8_PER_EXPERT if "fp8" in args.profile_kernel else B.MOE_WFMT_MXFP4_G32
        tc5 = args.profile_kernel.endswith("_tc5")
        decode_microbench(ctx, B, synth, torch, np, peaks()[0]["hbm_gbs"], n_layers=2, with_oracle=False,
                          reps=args.warmup + args.steps, fmts=(wfmt,), tokens=() if tc5 else (args.decode_tokens,),
                          tc5_tokens=(args.decode_tokens,) if tc5 else (), use_graph=False)
        return
    if args.profile_kernel == "kimi_route_scatter":
        from moe_expert_ffn_scatter_gb300.layer import MoEFFNLayer
        cfg = synth.KIMI
        inp = synth.ffn_inputs(cfg)
        L = MoEFFNLayer(B.Context(local), T=cfg.T, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I, A=cfg.A, cap=cfg.cap,
                        routing=B.MOE_ROUTE_SIGMOID_BIAS_TOPK, act_kind=B.MOE_ACT_SILU_CLAMP, limit=cfg.limit)
        x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
        logits, bias = torch.from_numpy(inp.logits).cuda(), torch.from_numpy(inp.bias).cuda()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for i in range(args.warmup + args.steps):
            if i == args.warmup: ev[0].record()
            L.route_scatter(x, logits, bias)
        ev[1].record()
        torch.cuda.synchronize()
        if B.moe_get_device_error(L.ctx) != 0:
            raise RuntimeError("device error")
        print("route_scatter us %.2f" % (1e3 * ev[0].elapsed_time(ev[1]) / max(1, args.steps)))
        return
    if args.profile_kernel == "kimi_layer":
        pk, _ = peaks()
        fp8_peak = 2.0 * pk["bf16_tflops"]
        res = kimi_layer_bench(B.Context(local), B, synth, torch, np, pk["hbm_gbs"], fp8_peak,
                               steps=args.steps, warmup=args.warmup)
        print(json.dumps(res))
        return
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist

    cfg = synth.DEEPSEEK
    inp = synth.ffn_inputs(cfg)
    ctx = B.Context(local)
    layer = MoEFFNLayer(ctx, T=cfg.T, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I, A=cfg.A, cap=cfg.cap, fused=True)
    layer.load_weights(inp.w13, inp.w13_sf, inp.w2, inp.w2_sf)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
    logits = torch.from_numpy(inp.logits).cuda()
    stream = torch.cuda.current_stream()
    L = layer
    parts = layer_parts(B, ctx, L, cfg, stream, x, logits)

    def step(ev=None):
        # the same launches as MoEFFNLayer.forward (route_scatter + moe_ffn_forward
        # with the fused GEMM1), made through the component entry points so that
        # each kernel is timed inside the timed region
        for j, f in enumerate(parts.values()):
            if ev is not None: ev[j].record(stream)
            f()
        if ev is not None: ev[4].record(stream)

    kernels_per_step = 3 + 1 + 1 + 1
    if args.profile_kernel:
        step()
        only = parts[args.profile_kernel]
        for _ in range(args.warmup + args.steps):
            only()
        torch.cuda.synchronize()
        if B.moe_get_device_error(ctx) != 0:
            raise RuntimeError("device error")
        return

    # Routing changes every step: the expert columns of the logits are permuted
    # before each step (a new permutation per step, seeds 100 + i), which
    # permutes the per-expert counts. The permuted logits are staged on the
    # device beforehand; each step starts with a 512 KB device copy of its
    # logits into the fixed-address buffer the layer reads.
    n_all = args.warmup + args.steps
    staged = torch.from_numpy(np.stack([np.ascontiguousarray(inp.logits[:, np.random.default_rng(100 + i).permutation(cfg.E)])
                                        for i in range(n_all)])).cuda()

    # The whole layer (route + scatter + GEMM1 with the fused act-quant + GEMM2
    # + combine, the calls MoEFFNLayer.forward makes) captured once in a CUDA
    # graph and replayed: the configuration's own form of the step.
    gstream = torch.cuda.Stream()
    gstream.wait_stream(stream)
    with torch.cuda.stream(gstream):
        logits.copy_(staged[0])
        layer.forward(x, logits, stream=gstream)
    gstream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream):
        layer.forward(x, logits, stream=gstream)
    torch.cuda.synchronize()

    def replay_step(i):
        logits.copy_(staged[i], non_blocking=True)
        graph.replay()

    for i in range(args.warmup):
        replay_step(i)
    torch.cuda.synchronize()
    if B.moe_get_device_error(ctx) != 0:
        raise RuntimeError("device error during warm-up")

    clocks = clock_sampler(local)
    if pg: pg.barrier()
    torch.cuda.synchronize()
    clocks.start()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for i in range(args.warmup, n_all):
        replay_step(i)
    g1.record(stream)
    torch.cuda.synchronize()
    if pg: pg.barrier()
    total_ms = max_over_ranks(g0.elapsed_time(g1), pg)
    graph_out = L.out.view(torch.int16).cpu().numpy().copy()
    # the last replay's output equals an eager forward on the same routing
    layer.forward(x, logits, stream=stream)
    torch.cuda.synchronize()
    if not np.array_equal(graph_out, L.out.view(torch.int16).cpu().numpy()):
        raise RuntimeError("graph replay and eager forward differ")

    # The same steps launched eagerly through the component entry points, with
    # CUDA events between the kernels: each kernel's own time (the roofline
    # figures below come from this region).
    for i in range(args.warmup):
        logits.copy_(staged[i], non_blocking=True)
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        logits.copy_(staged[args.warmup + i], non_blocking=True)
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    eager_ms = max_over_ranks(t_start.elapsed_time(t_end), pg)
    if B.moe_get_device_error(ctx) != 0:
        raise RuntimeError("device error during the timed region")
    names = ["route_scatter", "gemm1_act", "gemm2", "combine"]
    per = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)) / args.steps
           for j, n in enumerate(names)}
    ms_step = total_ms / args.steps
    R = cfg.R
    value = whole_job_rate(world, R, args.steps, total_ms)

    pk, pk_kind = peaks()
    # The GEMMs run for a few hundred microseconds inside a region of a few
    # milliseconds at full clock: the burst peak applies (the sustained one was
    # measured under the power cap over seconds).
    fp8_peak = 2.0 * pk["bf16_tflops"]
    fp8_peak_sustained = 2.0 * pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    hbm = pk["hbm_gbs"]
    g1_flop = 2.0 * R * (2 * cfg.I) * cfg.H
    g2_flop = 2.0 * R * cfg.H * cfg.I
    g1_tf = g1_flop / (per["gemm1_act"] * 1e-3) / 1e12
    g2_tf = g2_flop / (per["gemm2"] * 1e-3) / 1e12
    # algorithmic bytes of the HBM-bound steps (live rows only)
    G_H = cfg.H // 128
    rs_bytes = cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4 + R * (cfg.H + 4 * ((G_H + 3) // 4)) + R * 8 + cfg.T * cfg.k * 8
    cb_bytes = R * cfg.H * 2 + cfg.T * cfg.H * 2 + cfg.T * cfg.k * 8
    kern = {
        "route_scatter": {"us": 1e3 * per["route_scatter"], "gbs": rs_bytes / (per["route_scatter"] * 1e-3) / 1e9,
                          "frac_of_hbm": rs_bytes / (per["route_scatter"] * 1e-3) / 1e9 / hbm},
        "gemm1_act": {"us": 1e3 * per["gemm1_act"], "tflops": g1_tf, "frac_of_fp8_peak": g1_tf / fp8_peak},
        "gemm2": {"us": 1e3 * per["gemm2"], "tflops": g2_tf, "frac_of_fp8_peak": g2_tf / fp8_peak},
        "combine": {"us": 1e3 * per["combine"], "gbs": cb_bytes / (per["combine"] * 1e-3) / 1e9,
                    "frac_of_hbm": cb_bytes / (per["combine"] * 1e-3) / 1e9 / hbm},
        "eager_us_per_layer": 1e3 * eager_ms / args.steps,
    }
    roofline = {"bound": "tensor",
                "kernel": "gemm1_act (grouped_gemm_pair_kernel on this layer: CTA-pair tcgen05 mxf8f6f4 "
                          "block-scaled GEMM1 with SiLU*mul + e4m3/UE8M0 quantisation in its epilogue)",
                "achieved": g1_tf, "peak": fp8_peak, "unit": "TFLOP/s", "frac": g1_tf / fp8_peak,
                "traffic": recorded_traffic("gemm1_act"),
                "peak_note": "%s burst bf16 x 2 (the dense FP8/FP6/FP4-in-mxf8f6f4 rate is twice bf16): %.1f TFLOP/s "
                             "of measured; against the measured sustained bf16 x 2 (%.1f, taken under the power cap "
                             "at a median %s MHz) the fraction is %.3f" % (
                                 pk_kind, fp8_peak, fp8_peak_sustained,
                                 pk.get("clocks_under_load", {}).get("sm_mhz_median", "?"), g1_tf / fp8_peak_sustained),
                "algorithmic": "2*R*2I*H = %.1f GFLOP per launch over live rows only" % (g1_flop / 1e9),
                "timed_in": "the eager region of this run (CUDA events between the kernels, on the launching stream)"}

    # ---------------------------------------------- end to end (host buffers)
    # Every step copies its inputs (x, logits) from pinned host memory and
    # reads its output back into pinned host memory, through the public API
    # (MoEFFNLayer.forward). Pipelined (the e2e value): the upload of step
    # i+1 and the read-back of step i run on their own streams while step i
    # computes, with double-buffered device inputs and outputs; events keep a
    # buffer from being overwritten before its step has used it. Sequential
    # (reported beside it): copy in, compute, copy out, one after the other.
    e2e = None
    if True:
        xh = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).pin_memory()
        lh = torch.from_numpy(inp.logits).pin_memory()
        ohs = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        xds = [torch.empty_like(x) for _ in range(2)]
        lgds = [torch.empty_like(logits) for _ in range(2)]
        outs = [torch.empty_like(layer.out) for _ in range(2)]
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

        def seq_step():
            xds[0].copy_(xh, non_blocking=True)
            lgds[0].copy_(lh, non_blocking=True)
            out = layer.forward(xds[0], lgds[0], stream=stream)
            ohs[0].copy_(out, non_blocking=True)

        state = {"in_free": [None, None], "out_free": [None, None]}

        def pipe_step(i):
            b = i & 1
            with torch.cuda.stream(h2d_s):
                if state["in_free"][b] is not None:
                    h2d_s.wait_event(state["in_free"][b])
                xds[b].copy_(xh, non_blocking=True)
                lgds[b].copy_(lh, non_blocking=True)
                up = torch.cuda.Event()
                up.record(h2d_s)
            stream.wait_event(up)
            if state["out_free"][b] is not None:
                stream.wait_event(state["out_free"][b])
            layer.forward(xds[b], lgds[b], stream=stream, out=outs[b])
            done = torch.cuda.Event()
            done.record(stream)
            state["in_free"][b] = done
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done)
                ohs[b].copy_(outs[b], non_blocking=True)
                rb = torch.cuda.Event()
                rb.record(d2h_s)
            state["out_free"][b] = rb

        def timed(run):
            torch.cuda.synchronize()
            if pg: pg.barrier()
            torch.cuda.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            h2d_s.wait_event(a0)
            d2h_s.wait_event(a0)
            run()
            for s_ in (h2d_s, d2h_s):
                ev = torch.cuda.Event()
                ev.record(s_)
                stream.wait_event(ev)
            a1.record(stream)
            torch.cuda.synchronize()
            return max_over_ranks(a0.elapsed_time(a1), pg)

        def run_seq(n):
            for _ in range(n):
                seq_step()

        def run_pipe(n):
            state["in_free"], state["out_free"] = [None, None], [None, None]
            for i in range(n):
                pipe_step(i)

        timed(lambda: run_seq(max(3, args.warmup)))
        s_ms = timed(lambda: run_seq(args.steps))
        ref_out = ohs[0].view(torch.int16).numpy().copy()
        timed(lambda: run_pipe(max(3, args.warmup)))
        e_ms = timed(lambda: run_pipe(args.steps))
        for oh in ohs[:min(2, args.steps)]:
            if not np.array_equal(oh.view(torch.int16).numpy(), ref_out):
                raise RuntimeError("pipelined and sequential end-to-end outputs differ")
        e2e = {"value": whole_job_rate(world, R, args.steps, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": xh.numel() * 2 + lh.numel() * 4, "d2h_bytes_per_step": ohs[0].numel() * 2,
               "ms_per_step": e_ms / args.steps,
               "pipelined": "upload of step i+1 and read-back of step i on their own streams, overlapping "
                            "step i's compute (double-buffered device inputs/outputs)",
               "sequential_value": whole_job_rate(world, R, args.steps, s_ms),
               "sequential_ms_per_step": s_ms / args.steps,
               "api": "MoEFFNLayer.forward: moe_route_scatter + moe_ffn_forward, pinned host x/logits in, out back"}

    extras = {}
    if not args.no_extras:
        extras["act_quant_microbench"] = actq_microbench(ctx, B, synth, torch, np, hbm)
        extras["decode_microbench"] = decode_microbench(ctx, B, synth, torch, np, hbm)
        extras["tiny_layer"] = tiny_layer_bench(ctx, B, synth, torch, np)
        extras["kimi_layer"] = kimi_layer_bench(ctx, B, synth, torch, np, hbm, fp8_peak)

    conf = workload_config(cfg)
    conf["step"] = ("the layer captured once in a CUDA graph and replayed; before each replay a 512 KB device "
                    "copy brings that step's logits, whose expert columns are permuted (a new permutation per "
                    "step), so the per-expert counts change between replays")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "us_per_layer": 1e3 * ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e2m1 (fp32 accumulate)", "data": "synthetic",
            "config": conf, "roofline": roofline, "kernels": kern, "clocks": clk, "e2e": e2e,
            "gpu_launches": kernels_per_step * args.steps}
    line.update(extras)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def profile_act_quant(args, B, synth, torch, np, device):
    rows, I, E = synth.ACTQ_ROWS, synth.ACTQ_I, synth.ACTQ_E
    ctx = B.Context(device)
    gu, counts = synth.actq_inputs(full=False)
    g = torch.from_numpy(gu.view(np.int16)).view(torch.bfloat16).cuda()
    out = torch.empty((rows, I), dtype=torch.uint8, device="cuda")
    sf = torch.empty((I // 512, rows), dtype=torch.int32, device="cuda")
    ends = torch.empty((E,), dtype=torch.int32, device="cuda")
    B.moe_expert_ends_from_counts(ctx, torch.from_numpy(counts).cuda(), 128, ends)
    for _ in range(args.warmup + args.steps):
        B.moe_act_quant(ctx, g, out, sf, ends, E, 128, rows, I)
    torch.cuda.synchronize()
    if B.moe_get_device_error(ctx) != 0:
        raise RuntimeError("device error")


def tiny_layer_bench(ctx, B, synth, torch, np, reps=200):
    """The tiny layer (E = 4, top-2, T = 64, H = 256, I = 128): a latency
    figure. The layer is captured in a CUDA graph and replayed reps times;
    the oracle computes the same whole layer (routing, scatter, both grouped
    GEMMs, act-quant, combine) on the host cores."""
    import oracle as orc
    from moe_expert_ffn_scatter_gb300.layer import MoEFFNLayer

    cfg = synth.TINY
    inp = synth.ffn_inputs(cfg)
    L = MoEFFNLayer(ctx, T=cfg.T, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I, A=cfg.A, cap=cfg.cap)
    L.load_weights(inp.w13, inp.w13_sf, inp.w2, inp.w2_sf)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
    logits = torch.from_numpy(inp.logits).cuda()
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        L.forward(x, logits, stream=gs)
    gs.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        L.forward(x, logits, stream=gs)
    for _ in range(10):
        graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    if B.moe_get_device_error(ctx) != 0:
        raise RuntimeError("device error in the tiny layer")
    us = 1e3 * e0.elapsed_time(e1) / reps

    def oracle_layer():
        ids, w = orc.route_softmax_topk(inp.logits, cfg.k)
        ends, s2d, a, a_sf = orc.scatter(ids, inp.x, cfg.E, cfg.A, cfg.cap)
        gu = orc.grouped_gemm(a, a_sf, ends, cfg.A, inp.w13, inp.w13_sf)
        act, act_sf = orc.act_quant(gu, ends, cfg.A)
        down = orc.grouped_gemm(act, act_sf, ends, cfg.A, inp.w2, inp.w2_sf)
        return orc.combine(down, w, s2d)

    sec, reps_o = time_oracle(oracle_layer)
    del graph, L
    return {"workload": cfg.name, "us_per_layer": us, "routed_rows_per_s": cfg.R / (us * 1e-6),
            "timing": "CUDA graph of the whole layer, %d replays back to back" % reps,
            "cpu_baseline": oracle_baseline(sec, reps_o, lambda t: 1e6 * t, "the whole tiny layer by the oracle")}


def kimi_layer_bench(ctx, B, synth, torch, np, hbm, fp8_peak, steps=5, warmup=3):
    """The Kimi-shaped layer (E = 896, top-16, T = 2,048, H = 3,584, I = 3,072,
    sigmoid + bias routing, clamp 25) at full size, timed kernel by kernel.
    About 37 routes per expert: each expert's weights are used by one 128-row
    tile, so the GEMMs stream 14.8 GB of MXFP4 weights per layer and are bound
    by HBM, not by the tensor cores; both fractions are reported."""
    from moe_expert_ffn_scatter_gb300.layer import MoEFFNLayer

    cfg = synth.KIMI
    inp = synth.ffn_inputs(cfg)
    L = MoEFFNLayer(ctx, T=cfg.T, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I, A=cfg.A, cap=cfg.cap,
                    routing=B.MOE_ROUTE_SIGMOID_BIAS_TOPK, act_kind=B.MOE_ACT_SILU_CLAMP, limit=cfg.limit,
                    rsf=cfg.rsf)
    L.load_expert_weights(lambda e: synth.expert_weights(cfg, e))
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
    logits = torch.from_numpy(inp.logits).cuda()
    bias = torch.from_numpy(inp.bias).cuda()
    stream = torch.cuda.current_stream()
    parts = list(layer_parts(B, ctx, L, cfg, stream, x, logits, bias).items())
    for _ in range(warmup):
        for _, f in parts:
            f()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(steps)]
    for i in range(steps):
        for j, (_, f) in enumerate(parts):
            evs[i][j].record(stream)
            f()
        evs[i][-1].record(stream)
    torch.cuda.synchronize()
    if B.moe_get_device_error(ctx) != 0:
        raise RuntimeError("device error in the Kimi-shaped layer")
    per = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)) / steps for j, (n, _) in
           enumerate(parts)}
    ends = L.expert_ends.cpu().numpy().astype(np.int64)
    start = np.concatenate([[0], (ends[:-1] + cfg.A - 1) // cfg.A * cfg.A])
    counts = ends - start
    live_e = int((counts > 0).sum())
    tiles = int(((counts + 127) // 128).sum())
    R, H, I = cfg.R, cfg.H, cfg.I
    w1_bytes = live_e * (2 * I * H // 2 + 2 * I * H // 32)
    w2_bytes = live_e * (H * I // 2 + H * I // 32)
    g1_bytes = w1_bytes + R * (H + H // 128) + R * (I + I // 128)
    g2_bytes = w2_bytes + R * (I + I // 128) + R * H * 2

    def gemm(name, flop, tile_flop, nbytes):
        us = 1e3 * per[name]
        return {"us": us, "tflops_live": flop / (us * 1e-6) / 1e12,
                "frac_of_fp8_peak_live": flop / (us * 1e-6) / 1e12 / fp8_peak,
                "frac_of_fp8_peak_issued": tile_flop / (us * 1e-6) / 1e12 / fp8_peak,
                "gbs": nbytes / (us * 1e-6) / 1e9, "frac_of_hbm": nbytes / (us * 1e-6) / 1e9 / hbm,
                "bytes": nbytes}

    us_layer = 1e3 * sum(per.values())
    res = {"workload": cfg.name, "us_per_layer": us_layer, "routed_rows_per_s": R / (us_layer * 1e-6),
           "live_experts": live_e, "live_tiles": tiles,
           "route_scatter_us": 1e3 * per["route_scatter"], "combine_us": 1e3 * per["combine"],
           "gemm1_act": gemm("gemm1_act", 2.0 * R * 2 * I * H, 2.0 * tiles * 128 * 2 * I * H, g1_bytes),
           "gemm2": gemm("gemm2", 2.0 * R * H * I, 2.0 * tiles * 128 * H * I, g2_bytes)}
    del L, parts
    torch.cuda.empty_cache()
    return res


def actq_microbench(ctx, B, synth, torch, np, hbm, reps=50, with_oracle=True):
    """Live-row act-quant at 3,072 live / 28,672 allocated rows (I = 2,048),
    the all-live full buffer through the endpoint path, and the dense launch."""
    rows, I, E = synth.ACTQ_ROWS, synth.ACTQ_I, synth.ACTQ_E
    res = {}
    for name, full in (("live", False), ("full", True)):
        gu, counts = synth.actq_inputs(full=full)
        g = torch.from_numpy(gu.view(np.int16)).view(torch.bfloat16).cuda()
        out = torch.empty((rows, I), dtype=torch.uint8, device="cuda")
        sf = torch.empty((I // 512, rows), dtype=torch.int32, device="cuda")
        ends = torch.empty((E,), dtype=torch.int32, device="cuda")
        B.moe_expert_ends_from_counts(ctx, torch.from_numpy(counts).cuda(), 128, ends)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        variants = [(name, ends)] + ([("dense", None)] if full else [])
        for vname, e in variants:
            ts = []
            for i in range(reps + 3):
                flush.fill_(i & 0xFF)  # evict the inputs from L2 between launches
                s0 = torch.cuda.Event(enable_timing=True)
                s1 = torch.cuda.Event(enable_timing=True)
                s0.record()
                B.moe_act_quant(ctx, g, out, sf, e, E, 128, rows, I)
                s1.record()
                torch.cuda.synchronize()
                if i >= 3:
                    ts.append(s0.elapsed_time(s1))
            live_rows = int(counts.sum()) if e is not None else rows
            nbytes = live_rows * (2 * I * 2 + I + 4 * (I // 512))
            us = 1e3 * statistics.median(ts)
            res[vname] = {"us": us, "gbs": nbytes / (us * 1e-6) / 1e9, "frac_of_hbm": nbytes / (us * 1e-6) / 1e9 / hbm,
                          "live_rows": live_rows}
            if with_oracle:
                import oracle as orc
                ends_np = None if e is None else orc.endpoints(counts, 128)[1]
                sec, reps_o = time_oracle(lambda: orc.act_quant(gu, ends_np, 128))
                res[vname]["cpu_baseline"] = oracle_baseline(
                    sec, reps_o, lambda t: 1e6 * t,
                    "the whole launch (%d rows, SiLU*mul + e4m3/UE8M0 group 128) by the oracle" % live_rows)
    if "full" in res and "dense" in res:
        res["full_over_dense"] = res["full"]["us"] / res["dense"]["us"]
    # Back to back: 20 launches in a row over 20 device copies of the live-row
    # input (0.5 GB of live rows in all, so every launch reads HBM), timed
    # together: the kernel's own time per launch without the per-launch event
    # and launch overhead of the figures above.
    gu, counts = synth.actq_inputs(full=False)
    g0 = torch.from_numpy(gu.view(np.int16)).view(torch.bfloat16).cuda()
    copies = [g0.clone() for _ in range(20)]
    del g0
    out = torch.empty((rows, I), dtype=torch.uint8, device="cuda")
    sf = torch.empty((I // 512, rows), dtype=torch.int32, device="cuda")
    ends = torch.empty((E,), dtype=torch.int32, device="cuda")
    B.moe_expert_ends_from_counts(ctx, torch.from_numpy(counts).cuda(), 128, ends)
    ts = []
    for rep in range(6):
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        for gc in copies:
            B.moe_act_quant(ctx, gc, out, sf, ends, E, 128, rows, I)
        s1.record()
        torch.cuda.synchronize()
        if rep >= 1:
            ts.append(s0.elapsed_time(s1) / len(copies))
    live_rows = int(counts.sum())
    nbytes = live_rows * (2 * I * 2 + I + 4 * (I // 512))
    us = 1e3 * statistics.median(ts)
    res["live_back_to_back"] = {"us": us, "gbs": nbytes / (us * 1e-6) / 1e9,
                                "frac_of_hbm": nbytes / (us * 1e-6) / 1e9 / hbm, "live_rows": live_rows,
                                "launches": len(copies)}
    del copies
    torch.cuda.empty_cache()
    return res


def decode_microbench(ctx, B, synth, torch, np, hbm, n_layers=24, reps=5, fmts=None, tokens=(1, 2, 4, 8),
                      tc5_tokens=(1, 2, 4, 8, 32, 128), use_graph=True, with_oracle=True):
    """gpt-oss-shaped sparse decode (E=32, top-4, H=I=2,880), FP8-per-expert and
    MXFP4 weights: the mma.sync path (no workspace) at `tokens`, the tcgen05
    path (workspace) at `tc5_tokens` (keys *_tc5). 24 layers with their own
    weight copies run in sequence, so L2 (126 MB) cannot serve the 0.4-0.8 GB
    of weights per layer. Bytes counted: weights (+ scales, bias) of the
    distinct experts selected."""
    d = synth.decode_inputs(8)
    x_all = synth.decode_inputs(128, fp8=False, mxfp4=False)  # token rows and logits for T > 8
    E, k, H, I = synth.DECODE_E, synth.DECODE_K, synth.DECODE_H, synth.DECODE_I
    res = {}
    oracle_done = {}
    for fmt_name, wfmt, W in (("fp8", B.MOE_WFMT_FP8_PER_EXPERT, d.fp8), ("mxfp4", B.MOE_WFMT_MXFP4_G32, d.mxfp4)):
        if fmts is not None and wfmt not in fmts:
            continue
        layers = []
        base = {kk: torch.from_numpy(np.ascontiguousarray(v)).cuda() for kk, v in W.items()}
        for _ in range(n_layers):
            layers.append({kk: v.clone() for kk, v in base.items()})
        del base
        per_expert = sum(v[0].numel() * v.element_size() for kk, v in layers[0].items() if kk not in ("gu_scale", "d_scale"))
        for T, tc5 in [(t, False) for t in tokens] + [(t, True) for t in tc5_tokens]:
            src = d if T <= 8 else x_all
            x = torch.from_numpy(src.x[:T].view(np.int16)).view(torch.bfloat16).cuda()
            ws = B.decode_workspace(T, k, H, I, E) if tc5 else None
            # routing is an input of this call: the 4 largest generator logits per token,
            # slot weights 1/4 each (the decode GEMVs' cost does not depend on them)
            ids_np = np.argsort(-src.logits[:T], axis=1, kind="stable")[:, :k].astype(np.int32)
            ids = torch.from_numpy(ids_np).cuda()
            w = torch.full((T, k), 0.25, dtype=torch.float32, device="cuda")
            uniq = len(set(ids_np.ravel().tolist()))
            bf = lambda *shape: torch.empty(shape, dtype=torch.bfloat16, device="cuda")
            y1, act, y2, out = bf(T, k, 2 * I), bf(T * k, I), bf(T, k, H), bf(T, H)

            def run_layers():
                for L in layers:
                    kw = (dict(w_gu_scale=L["gu_scale"], w_d_scale=L["d_scale"]) if wfmt == 0 else
                          dict(w_gu_sf=L["gu_sf"], w_d_sf=L["d_sf"]))
                    B.moe_sparse_gemv_decode(ctx, x=x, topk_ids=ids, topk_w=w, expert_start=0, num_local_experts=E,
                                             wfmt=wfmt, w_gu=L["w_gu"], b_gu=L["b_gu"], w_d=L["w_d"], b_d=L["b_d"],
                                             y1=y1, act=act, y2=y2, out=out, T=T, H=H, I=I, k=k, workspace=ws,
                                             path=B.MOE_DECODE_TCGEN05 if tc5 else B.MOE_DECODE_AUTO, **kw)
            # decode steps are launch-bound on the host: capture the 24 layers once
            # in a CUDA graph (the layer calls only enqueue fixed grids) and replay
            run_layers()
            torch.cuda.synchronize()
            if not use_graph:  # plain launches, for profilers
                for _ in range(reps):
                    run_layers()
                torch.cuda.synchronize()
                continue
            gs = torch.cuda.Stream()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                run_layers()
            graph.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                graph.replay()
            e1.record()
            torch.cuda.synchronize()
            del graph
            us_layer = 1e3 * e0.elapsed_time(e1) / (reps * n_layers)
            nbytes = uniq * per_expert
            key = "%s_T%d%s" % (fmt_name, T, "_tc5" if tc5 else "")
            res[key] = {"us_per_layer": us_layer, "us_per_24_layers": us_layer * n_layers,
                        "unique_experts": uniq, "bytes_per_layer": nbytes,
                        "gbs": nbytes / (us_layer * 1e-6) / 1e9,
                        "frac_of_hbm": nbytes / (us_layer * 1e-6) / 1e9 / hbm}
            if with_oracle and (T, fmt_name) not in oracle_done:
                import oracle as orc
                xs = src.x[:T]
                wnp = np.full((T, k), 0.25, np.float32)
                sec, reps_o = time_oracle(lambda: orc.decode(xs, ids_np, wnp, W, wfmt, I), min_s=0.5, max_reps=5)
                oracle_done[(T, fmt_name)] = oracle_baseline(
                    sec, reps_o, lambda t: 1e6 * t,
                    "one whole layer (T = %d, %d slots: GEMV, GLU, GEMV, weighted sum) by the oracle" % (T, T * k))
            if with_oracle:
                res[key]["cpu_baseline"] = oracle_done[(T, fmt_name)]
        del layers
        torch.cuda.empty_cache()
    if B.moe_get_device_error(ctx) != 0:
        raise RuntimeError("device error in the decode microbench")
    return res


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
