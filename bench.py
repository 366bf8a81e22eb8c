"""Benchmark of the top-k routed MoE layer on GB300 (one JSON line on rank 0).

One step = one pass of the whole layer path over one batch: the prefill workload (T = 8192
tokens, H = 2048, 256 experts top-8 + shared expert, I = 512, bf16; 4 distinct layers, layer
l+1 reading bf16(x_0 + out_l)) through moe_forward.  `value` is MoE-layer tokens/s: tokens x
layers / seconds.  The decode workload (T = 1, 40 distinct layers, ~64.7 GB of weights,
captured as one CUDA graph) is timed in the same run and reported under "decode" as
us/layer.  Inputs are resident in HBM when the timed region starts; the per-layer weights
(1.6 GB) are larger than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, fp64, OpenMP over tokens) on the host cores,
on a bounded sample of the same workload per step.  Under torchrun each rank runs an
independent replica (the layer has no exchange step at this scale: replicas only).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s (prefill T=8192) & decode µs/layer; % of BF16 TC / HBM peak"
UNIT = "tokens/s"


def _dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if _cuda_ok() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def _cuda_ok():
    import torch
    return torch.cuda.is_available()


def _barrier(pg):
    if pg is not None:
        pg.barrier()


def _max_over_ranks(pg, v, device):
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None
        self.window = None  # (t0, t1) wall-clock seconds of the timed region

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if self.window and rows:
            # keep the samples taken inside the timed region (timestamps are local wall time)
            inside = []
            for r in rows:
                try:
                    ts = time.mktime(time.strptime(r[9].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + r[9].split(".")[1]) if "." in r[9] else 0.0
                except (IndexError, ValueError):
                    continue
                if self.window[0] - 0.05 <= ts <= self.window[1] + 0.05:
                    inside.append(r)
            if inside:
                rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------------ ours --

# dram__bytes_read.sum + dram__bytes_write.sum of one gate/up launch (routed experts + the shared
# expert, T=8192, H=2048, E=256, k=8, I=I_s=512) from an ncu capture of the current kernel, or None
# while the kernel has changed since the last capture: 1.42330 GB read + 72.50 MB written.
GATEUP_DRAM_BYTES = 1_495_805_952
# the same per layer for the one-token decode chain on bf16 weights (decode_chain_kernel<0>,
# H=2048, E=256, k=8, I=I_s=512; a 2-layer capture halved), or None until captured for the current
# kernel: 115.68 MB read + 3.40 MB written for 2 layers.
DECODE_CHAIN_DRAM_BYTES_PER_LAYER = 59_542_144
# the same for the chain on E4M3 expert weights (decode_chain_kernel<1>): 59.02 MB + 0.55 MB.
DECODE_CHAIN_Q8_DRAM_BYTES_PER_LAYER = 29_783_296
# the same for the chain on 4-bit expert weights (decode_chain_kernel<2>): 37.70 MB + 0.03 MB.
DECODE_CHAIN_Q4_DRAM_BYTES_PER_LAYER = 18_863_104


def _algorithmic(shape, T, experts_touched=None):
    """Flops of the layer's matrix products and bytes of the minimum weight+activation
    traffic, per layer, for T tokens."""
    H, E, k, I, Is = shape.hidden, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter
    gateup = 2.0 * T * k * H * 2 * I
    down = 2.0 * T * k * I * H
    shared_gu = 2.0 * T * H * 2 * Is
    shared = shared_gu + 2.0 * T * Is * H
    router = 2.0 * T * H * E
    # a shared expert as wide as the routed ones runs inside the routed gate/up launch
    gateup_launch = gateup + (shared_gu if Is == I else 0.0)
    # the gate/up launch's own minimum traffic: every routed expert's gate and up rows (all are
    # touched at this size), the shared expert's, each token row once, and h written (k + 1 rows a
    # token)
    touched = E if experts_touched is None else experts_touched
    gateup_bytes = 2 * (touched * 2 * I * H + 2 * Is * H + T * H + T * (k + 1) * I)
    return {"gateup_flops": gateup, "gateup_launch_flops": gateup_launch, "down_flops": down,
            "shared_flops": shared, "router_flops": router, "total_flops": gateup + down + shared + router,
            "gateup_launch_bytes": gateup_bytes}


def _decode_layer_bytes(shape):
    """All of one layer's weights (what the decode chain keeps resident)."""
    H, E, I, Is = shape.hidden, shape.n_experts, shape.inter, shape.shared_inter
    return 2 * (E * H + 3 * E * H * I + 3 * H * Is)


def _decode_bytes(shape):
    H, E, k, I, Is = shape.hidden, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter
    return E * H * 2 + k * 3 * H * I * 2 + 3 * H * Is * 2


def _decode_bytes_q8(shape):
    """The bytes one token reads with E4M3 expert weights: the bf16 router, one byte per expert
    weight of the k routed and the shared expert, and their fp32 row scales."""
    H, E, k, I, Is = shape.hidden, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter
    return E * H * 2 + k * 3 * H * I + 3 * H * Is + 4 * (k * (2 * I + H) + (2 * Is + H if Is else 0))


def _decode_bytes_q4(shape):
    """The bytes one token reads with 4-bit expert weights: the bf16 router, half a byte per
    expert weight of the k routed and the shared expert, and their fp32 block scales (one per 32)."""
    H, E, k, I, Is = shape.hidden, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter
    n = k * 3 * H * I + 3 * H * Is
    return E * H * 2 + n // 2 + 4 * (n // 32)


def run_ours(args, world, rank, local, pg):
    import torch
    from sparse_moe_router_gb300 import abi, inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    abi.load()
    peaks = _peaks()

    # ------------------------------------------------------------- prefill (value) --
    wl = inputs.WORKLOADS["prefill8k"]
    shape, T, L = wl.shape, wl.T, (args.layers or wl.n_layers)
    layers, x0 = inputs.make(wl, device=dev, n_layers=L)
    cfg = abi.config_of(shape)
    ws = abi.alloc_workspace(cfg, min(T, 8192))
    wts = [abi.weights(l) for l in layers]
    xa = x0.clone()
    xb = torch.empty_like(x0)
    xc = torch.empty_like(x0)
    out = torch.empty_like(x0)
    stream = torch.cuda.current_stream()

    def step(x_in):
        # layer l+1 reads bf16(x_0 + out_l): the residual add is fused into moe_forward
        x = x_in
        for l in range(L):
            nxt = xb if (x is not xb) else xc
            abi.moe_forward(cfg, wts[l], x, T, out, nxt, ws, stream, resid=x_in)
            x = nxt
        return x

    # The step as the library's resident graph (moe_graph_create): the L moe_forward calls captured
    # once, replayed by one moe_graph_launch per step.  Creating it runs the step once eagerly.
    graph = abi.Graph(cfg, wts, T, xa, out, xb, xc, ws, stream, resid=xa, keep=layers)
    for _ in range(args.warmup):
        graph.launch(stream)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0

    # The timed region: K steps, nothing but the layer's own launches on the stream.
    clocks = ClockSampler(local)
    clocks.start()
    _barrier(pg)
    torch.cuda.synchronize()
    n_launch0 = abi.moe_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_w0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        graph.launch(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(t_w0, time.time())
    launches = abi.moe_launch_count() - n_launch0
    _barrier(pg)
    clk = clocks.stop()
    t_ms = ev0.elapsed_time(ev1)
    t_ms = _max_over_ranks(pg, t_ms, dev)
    # The per-kernel split (and the roofline's kernel time): the same K steps again, launched
    # eagerly (moe_forward per layer) with a CUDA-event pair around every launch, on its stream.  The events time each kernel; they also put
    # a few microseconds between kernels, which is why they stay out of the region timed above.
    _barrier(pg)
    torch.cuda.synchronize()
    abi.timing_enable(True)
    for _ in range(args.steps):
        step(xa)
    torch.cuda.synchronize()
    abi.timing_enable(False)
    per_kernel = {}
    for name in abi.timing_classes():
        n, ms = abi.timing_read(name)
        if n:
            per_kernel[name] = {"launches": n, "total_ms": round(ms, 4), "avg_us": round(1e3 * ms / n, 2)}
    assert abi.moe_check_status(ws) == 0
    ms_per_step = t_ms / args.steps
    layer_tokens = T * L
    value = world * layer_tokens * args.steps / (t_ms * 1e-3)
    alg = _algorithmic(shape, T)
    gu = per_kernel.get("gateup_gemm")
    roofline = None
    if gu:
        # The kernel is timed per launch (CUDA-event pairs, a fraction of a second of work at the
        # box's full SM clock): the burst peak is its denominator.  At this shape it sits at the
        # ridge, so the fraction of the HBM bound on its own algorithmic bytes is reported beside.
        t_gu = gu["avg_us"] * 1e-6
        achieved = alg["gateup_launch_flops"] / t_gu / 1e12
        pk = peaks["bf16_tflops"]
        gbs = alg["gateup_launch_bytes"] / t_gu / 1e9
        roofline = {"bound": "tensor", "kernel": "gateup_gemm", "achieved": round(achieved, 1),
                    "peak": pk, "unit": "TFLOP/s", "frac": round(achieved / pk, 4),
                    "frac_of_sustained_peak": round(achieved / peaks["bf16_tflops_sustained"], 4),
                    "traffic": GATEUP_DRAM_BYTES, "peak_source": peaks["source"] + " bf16 burst",
                    "flops_per_launch": alg["gateup_launch_flops"],
                    "hbm_side": {"algorithmic_bytes": alg["gateup_launch_bytes"], "achieved_gbs": round(gbs, 1),
                                 "peak_gbs": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4)},
                    "kernel_us": gu["avg_us"],
                    "kernel_time": "CUDA-event pairs around every launch, in a second pass of the K timed steps"}
    layer_tflops = alg["total_flops"] * L * args.steps / (t_ms * 1e-3) / 1e12

    # ------------------------------------------------------------------------ e2e --
    # Every step copies its input from pinned host memory and its result back.  The copies run on
    # their own streams (one per direction, so an input copy never queues behind a result copy
    # that waits for its step), with double-buffered device input and result: step i's copies
    # overlap the layers of steps i-1 and i+1.  The timed region ends after the last copy back.
    e2e = None
    if not args.skip_e2e:
        x_host = x0.cpu().pin_memory()
        out_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
        xin = [torch.empty_like(x0) for _ in range(2)]
        res = [torch.empty_like(x0) for _ in range(2)]
        h2d_s = torch.cuda.Stream(device=dev)
        d2h_s = torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        in_ready, step_done, res_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        for b in range(2):  # nothing to wait for before the first uses
            step_done[b].record(stream)
            res_free[b].record(d2h_s)
        # one resident graph per buffer pair: layer 0 reads xin[b], the last layer writes res[b]
        graphs = [abi.Graph(cfg, wts, T, xin[b], out, res[b], xc, ws, stream, resid=xin[b], keep=layers)
                  for b in range(2)]

        def e2e_steps(n):
            for i in range(n):
                b = i & 1
                with torch.cuda.stream(h2d_s):
                    h2d_s.wait_event(step_done[b])  # step i-2 no longer reads xin[b]
                    xin[b].copy_(x_host, non_blocking=True)
                    in_ready[b].record(h2d_s)
                stream.wait_event(in_ready[b])
                stream.wait_event(res_free[b])  # step i-2's result has left res[b]
                graphs[b].launch(stream)
                step_done[b].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(step_done[b])
                    out_host[b].copy_(res[b], non_blocking=True)
                    res_free[b].record(d2h_s)
            for b in range(2):
                stream.wait_event(res_free[b])

        e2e_steps(2)
        torch.cuda.synchronize()
        # three timed windows of K steps each: the host-memory side of the copies is shared with
        # the rest of the machine, so the median window is reported (all three beside it)
        windows = []
        for _ in range(3):
            _barrier(pg)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_steps(args.steps)
            e1.record(stream)
            torch.cuda.synchronize()
            windows.append(_max_over_ranks(pg, e0.elapsed_time(e1), dev))
        te = statistics.median(windows)
        nbytes = x0.numel() * 2
        e2e = {"value": round(world * layer_tokens * args.steps / (te * 1e-3), 1), "unit": UNIT,
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
               "ms_per_step": round(te / args.steps, 4),
               "windows_ms_per_step": [round(w / args.steps, 4) for w in windows], "statistic": "median of 3 windows",
               "host_pinned": bool(x_host.is_pinned() and all(o.is_pinned() for o in out_host)),
               "path": "pinned host x -> moe_graph_launch (the 4 moe_forward layers, captured once by "
                       "moe_graph_create; C-ABI) -> pinned host out; the copies on "
                       "their own streams (one per direction), double-buffered, overlapping the neighbouring steps' layers"}

    del layers, wts
    torch.cuda.empty_cache()

    # -------------------------------------------------- the other prefill workloads --
    workloads = None
    if not args.skip_workloads:
        workloads = run_workloads(args, dev, pg, peaks)

    prefill_q8 = None
    if not args.skip_q8:
        prefill_q8 = run_prefill_q8(args, dev, pg, peaks)

    # --------------------------------------------------------------------- decode --
    decode = None
    if not args.skip_decode:
        decode = run_decode(args, dev, pg, peaks)

    # --------------------------------------------------------------- cpu baseline --
    cpu = None
    if rank == 0 and not args.skip_cpu:
        cpu = cpu_baseline(wl, seconds=args.cpu_seconds)

    res = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded normal weights/activations, random-init layer shape)",
           "config": {"workload": "prefill T=8192, H=2048, E=256 top-8 + shared (I=Is=512), 4 distinct "
                                  "layers, layer l+1 reads bf16(x_0 + out_l)",
                      "tokens": T, "layers": L, "parallelism": "replicas" if world > 1 else "single GPU",
                      "l2": "no flush: each layer's weights (1.6 GB) exceed the 129 MB L2",
                      "value_definition": "tokens x layers / s (one token through one MoE layer)",
                      "launch": "one moe_graph_launch per step: the layers' moe_forward calls captured once by "
                                "moe_graph_create"},
           "layer_tflops": round(layer_tflops, 1),
           "roofline": roofline, "per_kernel": per_kernel, "gpu_launches": int(launches),
           "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "decode": decode, "workloads": workloads,
           "prefill_e4m3_weights": prefill_q8,
           "peaks": peaks}
    return res


def _graph_ms(abi, cfg, wts, T, x, ws, stream, steps, warmup, keep):
    """Median-free mean time of one replay of the layer stack `wts` on x's T tokens, captured by
    moe_graph_create (each layer l+1 reads bf16(x + out_l)); CUDA events on the launching stream."""
    import torch
    out, xb, xc = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
    g = abi.Graph(cfg, wts, T, x, out, xb, xc, ws, stream, resid=x, keep=keep)
    for _ in range(warmup):
        g.launch(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.launch(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    g.destroy()
    return e0.elapsed_time(e1) / steps


def _eager_split(abi, cfg, wts, T, x, ws, stream):
    """Per-kernel CUDA-event averages of one eager pass of the layers (moe_forward per layer)."""
    import torch
    out, nxt = torch.empty_like(x), torch.empty_like(x)
    abi.timing_enable(True)
    for w in wts:
        abi.moe_forward(cfg, w, x, T, out, nxt, ws, stream, resid=x)
    torch.cuda.synchronize()
    abi.timing_enable(False)
    res = {}
    for name in abi.timing_classes():
        n, ms = abi.timing_read(name)
        if n:
            res[name] = {"launches": n, "avg_us": round(1e3 * ms / n, 2)}
    return res


def run_workloads(args, dev, pg, peaks):
    """The other two prefill workloads, each under its own key: T=1024 with Zipf(1.0) router
    bias (one layer, HBM-bound by the roofline) and T=13,337 composed as 8192+4096+1024+25 with
    Zipf(1.5) and four dead experts (four layers), with a per-piece split."""
    import numpy as np
    import torch
    from sparse_moe_router_gb300 import abi, inputs

    stream = torch.cuda.current_stream()
    res = {}
    for name in ("prefill1k", "prompt13337"):
        wl = inputs.WORKLOADS[name]
        shape, T, L = wl.shape, wl.T, wl.n_layers
        layers, x = inputs.make(wl, device=dev)
        cfg = abi.config_of(shape)
        ws = abi.alloc_workspace(cfg, min(T, 8192))
        wts = [abi.weights(l) for l in layers]
        # realised routing of the first layer (touched experts, skew)
        ids = torch.empty(T, shape.top_k, dtype=torch.int32, device=dev)
        tw = torch.empty(T, shape.top_k, dtype=torch.float32, device=dev)
        wsr = abi.alloc_workspace(cfg, T)
        abi.moe_route(cfg, wts[0], x, T, None, ids, tw, wsr)
        torch.cuda.synchronize()
        del wsr
        counts = np.bincount(ids.cpu().numpy().ravel(), minlength=shape.n_experts)
        touched = int((counts > 0).sum())
        ms = _max_over_ranks(pg, _graph_ms(abi, cfg, wts, T, x, ws, stream, max(20, args.steps // 4), args.warmup,
                                           layers), dev)
        us_layer = 1e3 * ms / L
        alg = _algorithmic(shape, T, experts_touched=touched)
        H, E, I, Is = shape.hidden, shape.n_experts, shape.inter, shape.shared_inter
        layer_bytes = 2 * (touched * 3 * I * H + 3 * Is * H + E * H + 2 * T * H)
        tflops = alg["total_flops"] / (us_layer * 1e-6) / 1e12
        gbs = layer_bytes / (us_layer * 1e-6) / 1e9
        r = {"workload": wl.note, "tokens": T, "layers": L, "us_per_layer": round(us_layer, 2),
             "tokens_per_s": round(T / (us_layer * 1e-6), 1),
             "layer_tokens_per_s": round(T * L / (ms * 1e-3), 1),
             "tflops": round(tflops, 1), "tc_frac_of_burst": round(tflops / peaks["bf16_tflops"], 4),
             "algorithmic_bytes_per_layer": layer_bytes, "gbs": round(gbs, 1),
             "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
             "experts_touched": touched, "rows_per_expert_max": int(counts.max()),
             "rows_per_expert_mean": round(float(counts.mean()), 1), "empty_experts": int((counts == 0).sum()),
             "per_kernel_eager": _eager_split(abi, cfg, wts[:1], T, x, ws, stream),
             "launch": "moe_graph_create of the %d moe_forward layers, one moe_graph_launch per step" % L}
        if name == "prompt13337":
            pieces, t0 = [], 0
            for pc in abi.moe_plan_pieces(T):
                xs = x[t0:t0 + pc]
                pms = _max_over_ranks(pg, _graph_ms(abi, cfg, wts[:1], pc, xs, ws, stream, 20, args.warmup, layers),
                                      dev)
                pieces.append({"tokens": pc, "us": round(1e3 * pms, 2),
                               "tokens_per_s": round(pc / (pms * 1e-3), 1)})
                t0 += pc
            r["pieces_one_layer"] = pieces
            r["pieces_sum_us"] = round(sum(p["us"] for p in pieces), 2)
        res[name] = r
        del layers, wts, x, ws
        torch.cuda.empty_cache()
    return res


def run_prefill_q8(args, dev, pg, peaks):
    """The prefill workloads with E4M3 expert weights (moe_forward_q8): the bf16 layers quantised on
    the device (moe_quantize_e4m3), the layer stack captured as one CUDA graph."""
    import torch
    from sparse_moe_router_gb300 import abi, inputs

    s = torch.cuda.Stream(device=dev)
    res = {}
    for name in args.q8_workloads.split(","):
        wl = inputs.WORKLOADS[name]
        shape, T, L = wl.shape, wl.T, wl.n_layers
        layers_bf, x0 = inputs.make(wl, device=dev)
        with torch.cuda.stream(s):
            layers = [abi.quantize_layer(l, s) for l in layers_bf]
        torch.cuda.synchronize()
        del layers_bf
        cfg = abi.config_of(shape)
        ws = abi.alloc_workspace(cfg, min(T, 8192))
        wts = [abi.weights_q8(l) for l in layers]
        bufs = [torch.empty_like(x0), torch.empty_like(x0)]
        out = torch.empty_like(x0)

        def chain():
            x = x0
            for l in range(L):
                nxt = bufs[l % 2]
                abi.moe_forward_q8(cfg, wts[l], x, T, out, nxt, ws, s, resid=x0)
                x = nxt

        with torch.cuda.stream(s):
            chain()
        torch.cuda.synchronize()
        assert abi.moe_check_status(ws) == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                chain()
        torch.cuda.synchronize()
        steps = max(20, args.steps // 4)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            for _ in range(args.warmup):
                g.replay()
            torch.cuda.synchronize()
            e0.record(s)
            for _ in range(steps):
                g.replay()
            e1.record(s)
        torch.cuda.synchronize()
        ms = _max_over_ranks(pg, e0.elapsed_time(e1) / steps, dev)
        del g
        abi.timing_enable(True)
        with torch.cuda.stream(s):
            abi.moe_forward_q8(cfg, wts[0], x0, T, out, bufs[0], ws, s, resid=x0)
        torch.cuda.synchronize()
        abi.timing_enable(False)
        split = {}
        for kn in abi.timing_classes():
            n, t = abi.timing_read(kn)
            if n:
                split[kn] = {"launches": n, "avg_us": round(1e3 * t / n, 2)}
        us_layer = 1e3 * ms / L
        alg = _algorithmic(shape, T)
        res[name] = {"tokens": T, "layers": L, "us_per_layer": round(us_layer, 2),
                     "layer_tokens_per_s": round(T * L / (ms * 1e-3), 1),
                     "tflops": round(alg["total_flops"] / (us_layer * 1e-6) / 1e12, 1),
                     "per_kernel_eager": split,
                     "weights": "E4M3 codes + fp32 row scales for every expert matrix (router bf16), quantised "
                                "on the device from the bf16 workload"}
        del layers, wts, ws
        torch.cuda.empty_cache()
    return res


def run_decode_only(args, world, rank, local, pg):
    """--decode-only: the decode measurement alone, as its own JSON line."""
    import torch
    from sparse_moe_router_gb300 import abi

    torch.cuda.set_device(local)
    abi.load()
    d = run_decode(args, torch.device("cuda", local), pg, _peaks())
    return {"metric": "MoE layer decode us/layer (T=1)", "value": d["us_per_layer"], "unit": "us/layer",
            "n_gpus": world, "higher_is_better": False, "decode": d}


def run_decode(args, dev, pg, peaks):
    import torch
    from sparse_moe_router_gb300 import abi, inputs

    wl = inputs.WORKLOADS["decode"]
    shape, L = wl.shape, (args.decode_layers or wl.n_layers)
    layers, x0 = inputs.make(wl, device=dev, n_layers=L)
    cfg = abi.config_of(shape)
    wts = [abi.weights(l) for l in layers]
    s = torch.cuda.Stream(device=dev)

    def graph_time(x_start, one_launch=False, wts_q8=None, wts_q4=None):
        """Median time of the 40-layer chain for x_start's tokens, captured as one CUDA graph:
        one moe_forward call per layer, or (one_launch) one moe_decode_chain call for all, or
        (wts_q8 / wts_q4) one moe_decode_chain_q8 / _q4 call on the quantised copies of the layers."""
        T = x_start.shape[0]
        ws = abi.alloc_workspace(cfg, T)
        bufs = [x_start.clone(), torch.empty_like(x_start), torch.empty_like(x_start)]
        out = torch.empty_like(x_start)

        def chain():
            # layer l+1 reads bf16(x_0 + out_l), fused into the layer's last kernel
            if wts_q8 is not None:
                abi.moe_decode_chain_q8(cfg, wts_q8, bufs[0], out, bufs[1], ws, s, resid=bufs[0])
                return
            if wts_q4 is not None:
                abi.moe_decode_chain_q4(cfg, wts_q4, bufs[0], out, bufs[1], ws, s, resid=bufs[0])
                return
            if one_launch:
                abi.moe_decode_chain(cfg, wts, bufs[0], out, bufs[1], ws, s, resid=bufs[0])
                return
            x = bufs[0]
            for l in range(L):
                nxt = bufs[1 + (l % 2)]
                abi.moe_forward(cfg, wts[l], x, T, out, nxt, ws, s, resid=bufs[0])
                x = nxt

        with torch.cuda.stream(s):
            for _ in range(3):
                chain()
        torch.cuda.synchronize()
        assert abi.moe_check_status(ws) == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                chain()
        torch.cuda.synchronize()
        reps = max(5, args.steps)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        times = []
        n_launch0 = abi.moe_launch_count()
        with torch.cuda.stream(s):   # replay() launches on the current stream: time on that stream
            for _ in range(max(3, args.warmup)):
                g.replay()
            torch.cuda.synchronize()
            for _ in range(reps):
                e0.record(s)
                g.replay()
                e1.record(s)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
        assert abi.moe_launch_count() == n_launch0  # replays launch from the graph, not the library
        assert abi.moe_check_status(ws) == 0
        del g
        return times, chain

    # the decode step: all layers in one cooperative launch (moe_decode_chain); the same stack as
    # one moe_forward call per layer is reported beside it
    times_calls, _ = graph_time(x0)
    times, chain = graph_time(x0, one_launch=True)
    us_calls = 1e3 * _max_over_ranks(pg, statistics.median(times_calls), dev) / L
    reps = len(times)
    t_med = statistics.median(times)
    t_med = _max_over_ranks(pg, t_med, dev)
    us_layer = 1e3 * t_med / L
    nbytes = _decode_bytes(shape)
    gbs = nbytes / (us_layer * 1e-6) / 1e9
    # per-kernel split of one eager chain (outside the graph)
    abi.timing_enable(True)
    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    abi.timing_enable(False)
    split = {}
    for name in ("decode_chain", "decode_router", "decode_experts"):
        n, ms = abi.timing_read(name)
        if n:
            split[name] = {"launches": n, "avg_us": round(1e3 * ms / n, 2)}
    # a few tokens at once (multi-token prediction, speculative verification): 2..4 tokens take
    # the decode path, each selected expert streamed once for all tokens that chose it
    small = []
    for T in (2, 3, 4):
        _, xT = inputs.make(inputs.custom(shape, T=T, seed=100 + T), device=dev, n_layers=0)
        tT = _max_over_ranks(pg, statistics.median(graph_time(xT)[0]), dev)
        small.append({"T": T, "us_per_layer": round(1e3 * tT / L, 3),
                      "tokens_per_s": round(T * L / (tT * 1e-3), 1)})
    # the same stack with E4M3 expert weights (row scales; the router stays bf16), quantised on the
    # device from the bf16 layers, through moe_decode_chain_q8
    q8 = None
    if not args.skip_q8:
        with torch.cuda.stream(s):
            layers_q8 = [abi.quantize_layer(l, s) for l in layers]
        torch.cuda.synchronize()
        tq = _max_over_ranks(pg, statistics.median(graph_time(x0, wts_q8=[abi.weights_q8(l) for l in layers_q8])[0]),
                             dev)
        del layers_q8
        us_q8 = 1e3 * tq / L
        nq = _decode_bytes_q8(shape)
        gq = nq / (us_q8 * 1e-6) / 1e9
        q8 = {"us_per_layer": round(us_q8, 3), "bytes_per_layer": nq,
              "roofline": {"bound": "hbm", "achieved": round(gq, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(gq / peaks["hbm_gbs"], 4), "traffic": DECODE_CHAIN_Q8_DRAM_BYTES_PER_LAYER,
                           "traffic_kernel": "decode_chain_kernel<1>"}}
    # and with 4-bit expert weights (scale per block of 32; the router stays bf16), quantised on the
    # device from the bf16 layers, through moe_decode_chain_q4
    q4 = None
    if not args.skip_q8:
        with torch.cuda.stream(s):
            layers_q4 = [abi.quantize_layer_q4(l, s) for l in layers]
        torch.cuda.synchronize()
        tq = _max_over_ranks(pg, statistics.median(graph_time(x0, wts_q4=[abi.weights_q4(l) for l in layers_q4])[0]),
                             dev)
        del layers_q4
        us_q4 = 1e3 * tq / L
        nq = _decode_bytes_q4(shape)
        gq = nq / (us_q4 * 1e-6) / 1e9
        q4 = {"us_per_layer": round(us_q4, 3), "bytes_per_layer": nq,
              "roofline": {"bound": "hbm", "achieved": round(gq, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(gq / peaks["hbm_gbs"], 4), "traffic": DECODE_CHAIN_Q4_DRAM_BYTES_PER_LAYER,
                           "traffic_kernel": "decode_chain_kernel<2>"}}
    return {"workload": "decode T=1, %d distinct layers (%.1f GB of weights), one moe_decode_chain launch "
                        "in a CUDA graph" % (L, L * _decode_layer_bytes(shape) / 1e9),
            "us_per_layer": round(us_layer, 3), "graph_ms": round(t_med, 4), "reps": reps,
            "us_per_layer_one_call_per_layer": round(us_calls, 3),
            "p10_p90_ms": [round(sorted(times)[len(times) // 10], 4),
                           round(sorted(times)[(9 * len(times)) // 10], 4)],
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "frac_of_8000": round(gbs / 8000.0, 4), "bytes_per_layer": nbytes,
                         "traffic": DECODE_CHAIN_DRAM_BYTES_PER_LAYER, "traffic_kernel": "decode_chain_kernel<0>",
                         "peak_source": peaks["source"] + " hbm copy"},
            "eager_kernel_avg_us": split, "small_batch": small, "e4m3_weights": q8, "int4_weights": q4}


def cpu_baseline(wl, seconds=12.0):
    """The CPU oracle, as it stands, on a bounded sample of the prefill workload's tokens."""
    import numpy as np
    import torch

    from oracle import moe_oracle as orc
    from sparse_moe_router_gb300 import inputs

    layers, x = inputs.make(wl, device="cuda" if torch.cuda.is_available() else "cpu", n_layers=1)
    hl = inputs.layer_to_host(layers[0])
    xs = inputs.to_u16(x)
    layers0 = layers[0]
    del layers
    threads = orc.threads(0)
    k = wl.shape.top_k
    # calibrate on a few tokens, then size the sample to about `seconds`
    n0 = max(threads, 8)
    t0 = time.perf_counter()
    orc.forward(np.ascontiguousarray(xs[:n0]), hl, k)
    dt = time.perf_counter() - t0
    n = int(min(wl.T, max(n0, seconds / max(dt / n0, 1e-9))))
    n = max(threads, (n // threads) * threads)
    t0 = time.perf_counter()
    orc.forward(np.ascontiguousarray(xs[:n]), hl, k)
    dt = time.perf_counter() - t0
    res = {"value": round(n / dt, 2), "unit": UNIT, "cores": threads, "kind": "oracle",
           "sample": "%d of the %d tokens of one layer of the prefill workload (fp64 C oracle, "
                     "OpenMP over tokens), %.1f s" % (n, wl.T, dt)}
    if torch.cuda.is_available():
        res["parity"] = _parity_sample(wl, layers0, x, hl, xs, orc)
    return res


def _parity_sample(wl, layer, x, hl, xs, orc, rows=512):
    """The GPU layer (moe_forward on the workload's first layer) against the oracle on a row
    sample, with the oracle taking the GPU's routing (as the parity tests do): max |diff|, rel L2
    and the rows whose ids differ from the oracle's own selection on the GPU's logits."""
    import numpy as np
    import torch

    from sparse_moe_router_gb300 import abi, inputs

    T, k = wl.T, wl.shape.top_k
    cfg = abi.config_of(wl.shape)
    ws = abi.alloc_workspace(cfg, min(T, 8192))
    wts = abi.weights(layer)
    out = torch.empty_like(x)
    abi.moe_forward(cfg, wts, x, T, out, None, ws)
    logits = torch.empty(T, wl.shape.n_experts, dtype=torch.float32, device=x.device)
    ids = torch.empty(T, k, dtype=torch.int32, device=x.device)
    w = torch.empty(T, k, dtype=torch.float32, device=x.device)
    abi.moe_route(cfg, wts, x, T, logits, ids, w, ws)
    torch.cuda.synchronize()
    assert abi.moe_check_status(ws) == 0
    sel = np.linspace(0, T - 1, rows).astype(np.int64)
    ids_h, w_h, lg = ids.cpu().numpy()[sel], w.cpu().numpy()[sel], logits.cpu().numpy()[sel]
    ref = orc.forward(np.ascontiguousarray(xs[sel]), hl, k, ids=ids_h, topk_w=w_h)["out"]
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g, r = f(inputs.to_u16(out)[sel]), f(ref)
    ids_o, _ = orc.route_from_logits(lg, k)
    return {"rows": rows, "max_abs": float(np.abs(g - r).max()),
            "rel_l2": float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)),
            "ids_mismatch_rows": int(np.sum(np.any(ids_o != ids_h, axis=1))),
            "bound": {"max_abs": 2e-2, "rel_l2": 5e-3}}


def run_oracle_table(args):
    """--oracle-table: the CPU oracle timed on the host cores for every workload, single-thread and
    on all allowed cores (T=8192 and T=13,337: all cores only), each interleaved with the GPU layer
    in A/B/B/A order (oracle, GPU, GPU, oracle) as the paired-order method of "AIMA Intel PTL
    Qwen3.6 35B U4 Engine" ("ABBA" blocks); the ratio is the median oracle time over the median
    GPU time of the same layer.  One layer each; the oracle runs its own routing on all tokens."""
    import numpy as np
    import torch
    from oracle import moe_oracle as orc
    from sparse_moe_router_gb300 import abi, inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    abi.load()
    stream = torch.cuda.current_stream()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    all_threads = orc.threads(0)
    plan = [("tiny", ("single-thread", "all-core")), ("decode", ("single-thread", "all-core")),
            ("prefill1k", ("single-thread", "all-core")), ("prefill8k", ("single-thread", "all-core")),
            ("prompt13337", ("single-thread", "all-core"))]
    # single-thread on the two large workloads: the first 512 tokens (tokens are independent, so
    # the per-token cost holds for the whole layer); about 15 s per oracle run
    sample_single = {"prefill8k": 512, "prompt13337": 512}
    rows = []
    for name, modes in plan:
        wl = inputs.WORKLOADS[name]
        layers, x = inputs.make(wl, device=dev, n_layers=1)
        cfg = abi.config_of(wl.shape)
        T = wl.T
        ws = abi.alloc_workspace(cfg, min(T, 8192))
        wts = [abi.weights(layers[0])]
        hl = inputs.layer_to_host(layers[0])
        xs = np.ascontiguousarray(inputs.to_u16(x))
        k = wl.shape.top_k

        def gpu_us():
            return 1e3 * _graph_ms(abi, cfg, wts, T, x, ws, stream, 20, 3, layers)

        ref = {}

        def oracle_s(nt, n_tok):
            t0 = time.perf_counter()
            r = orc.forward(np.ascontiguousarray(xs[:n_tok]), hl, k, n_threads=nt)
            dt = time.perf_counter() - t0
            if n_tok == T:
                ref.setdefault("r", r)
            return dt

        def parity():
            """The GPU layer (moe_forward) against the oracle's own run, over the rows whose expert
            set the two select alike (a near-tie may flip a selection; those rows are counted)."""
            out = torch.empty_like(x)
            ids = torch.empty(T, k, dtype=torch.int32, device=dev)
            tw = torch.empty(T, k, dtype=torch.float32, device=dev)
            wsr = abi.alloc_workspace(cfg, T)
            abi.moe_forward(cfg, wts[0], x, T, out, None, ws)
            abi.moe_route(cfg, wts[0], x, T, None, ids, tw, wsr)
            torch.cuda.synchronize()
            r = ref["r"]
            same = np.all(np.sort(ids.cpu().numpy(), 1) == np.sort(r["ids"], 1), axis=1)
            f = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            g, o = f(inputs.to_u16(out))[same], f(r["out"])[same]
            return {"rows": int(same.sum()), "rows_other_selection": int((~same).sum()),
                    "max_abs": float(np.abs(g - o).max()) if g.size else 0.0,
                    "rel_l2": float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-30)) if g.size else 0.0}

        for mode in reversed(modes):  # all-core first: its full run is the parity reference
            nt = 1 if mode == "single-thread" else all_threads
            n_tok = sample_single.get(name, T) if mode == "single-thread" else T
            a1 = oracle_s(nt, n_tok)
            b1, b2 = gpu_us(), gpu_us()
            a2 = oracle_s(nt, n_tok)
            a, b = statistics.median([a1, a2]), statistics.median([b1, b2])
            o_tps, g_tps = n_tok / a, T / (b * 1e-6)
            rows.append({"workload": name, "tokens": T, "oracle_tokens": n_tok, "mode": mode, "threads": nt,
                         "parity": parity() if "r" in ref else None,
                         "order": "oracle, GPU, GPU, oracle",
                         "oracle_s": [round(a1, 4), round(a2, 4)], "gpu_us": [round(b1, 2), round(b2, 2)],
                         "oracle_tokens_per_s": round(o_tps, 2), "gpu_tokens_per_s": round(g_tps, 1),
                         "ratio_gpu_over_oracle": round(g_tps / o_tps, 1)})
            print(json.dumps(rows[-1]), file=sys.stderr, flush=True)
        del layers, wts, x, ws, hl
        torch.cuda.empty_cache()
    return {"oracle_table": rows, "host_cores_allowed": cores, "oracle_threads_all_core": all_threads,
            "oracle": "plain C, fp64 accumulation, OpenMP over tokens; one layer, the oracle's own routing",
            "gpu": "one moe_forward layer captured by moe_graph_create, mean of 20 replays"}


def run_reference(args, world, rank):
    """--impl reference: the CPU oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return None
    import numpy as np
    import torch

    from oracle import moe_oracle as orc
    from sparse_moe_router_gb300 import inputs

    wl = inputs.WORKLOADS["prefill8k"]
    layers, x = inputs.make(wl, device="cuda" if torch.cuda.is_available() else "cpu", n_layers=1)
    hl = inputs.layer_to_host(layers[0])
    xs = inputs.to_u16(x)
    del layers
    threads = orc.threads(0)
    k = wl.shape.top_k
    n0 = max(threads, 8)
    t0 = time.perf_counter()
    orc.forward(np.ascontiguousarray(xs[:n0]), hl, k)
    per_tok = (time.perf_counter() - t0) / n0
    # each step: about args.ref_step_seconds of oracle work, less when the whole run (warm-up and
    # timed steps) would otherwise exceed args.ref_total_seconds
    step_s = min(args.ref_step_seconds, args.ref_total_seconds / max(1, args.steps + args.warmup))
    n = int(max(1, min(wl.T, step_s / max(per_tok, 1e-9))))
    if n >= threads:
        n = (n // threads) * threads
    threads = min(threads, n)
    sample = np.ascontiguousarray(xs[:n])
    for _ in range(args.warmup):
        orc.forward(sample, hl, k)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.forward(sample, hl, k)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    desc = "%d of the %d tokens of one prefill layer per step (fp64 C oracle, OpenMP over tokens)" % (n, wl.T)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * dt / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "prefill T=8192, H=2048, E=256 top-8 + shared (I=Is=512); "
                                   "bounded token sample per step", "tokens_per_step": n},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "kind": "oracle", "cores": threads,
                             "sample": desc},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)  # ~1 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-q8", action="store_true", help="skip the quantised-weight (E4M3, 4-bit) measurements")
    ap.add_argument("--q8-workloads", default="prefill8k,prefill1k",
                    help="prefill workloads timed with E4M3 expert weights (comma list)")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-workloads", action="store_true",
                    help="skip the T=1024 and T=13,337 prefill workloads")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="prefill layers per step (default: the workload's 4); fewer only for profiler captures")
    ap.add_argument("--decode-only", action="store_true",
                    help="run the decode measurement alone (for profiler captures)")
    ap.add_argument("--decode-layers", type=int, default=0,
                    help="decode layers (default: the workload's 40); fewer only for profiler captures")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the CPU oracle on every workload (single-thread and all cores, A/B/B/A with the GPU)")
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--ref-total-seconds", type=float, default=120.0,
                    help="bound on the reference arm's oracle work over all its warm-up and timed steps")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local, pg = _dist_init()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    elif args.oracle_table:
        res = run_oracle_table(args) if rank == 0 else None
    elif args.decode_only:
        res = run_decode_only(args, world, rank, local, pg)
    else:
        res = run_ours(args, world, rank, local, pg)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
