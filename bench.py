#!/usr/bin/env python
"""Benchmark of the GB300 ternary linear layer (one JSON line on stdout).

Metric: "ternary linear int8 TOPS @M=512; decode GEMV weight-stream GB/s @M=1".

  prefill  (headline `value`): the fused gate+up projection of the 27B model,
           M=512 tokens, K=5120, N=34816. One step = the 512-token batch through
           64 layer buffers (64 distinct weight sets, 2.95 GB, so no step finds
           its weights in the 129 MB L2): per layer rotate+quantise (K1) then the
           tensor-core GEMM with fused rescale (K3). TOPS = 64 * 2 M N K / step.
  decode   (`decode` object): M=1, K=5120, N=17408 over 64 layer buffers (1.47 GB);
           per layer rotate+quantise (K1) then the dp4a GEMV (K2), captured in one
           CUDA graph per step. GB/s = 64 * (packed + qT + sw bytes) / step. The
           GEMV kernel alone (64 back-to-back launches) gives the roofline figure;
           the single-launch fused variant (tl_linear_decode_fused) is timed beside it.

Inputs are seeded synthetic draws with the workloads' shapes and distributions,
generated on the device; they are resident in HBM before timing starts.
`e2e` repeats both through the public API with pinned host buffers: each step
copies every layer's x in and its y back inside the timed region (prefill:
TernaryLinear layers driven by tl.HostPipeline, copies overlapping the kernels;
decode: the whole step as one tl.GraphStep CUDA graph).
`--impl reference` times the CPU oracle instead (see oracle/).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS = 64
PREFILL = dict(name="gate_up", M=512, K=5120, N=34816)
DECODE = dict(name="decode", M=1, K=5120, N=17408)
METRIC = "ternary linear int8 TOPS @M=512; decode GEMV weight-stream GB/s @M=1"
CONFIG_SWEEP_M = (1, 4, 16, 64, 256, 1024, 4096)   # the M-sweep points reported in `configs`
EVENT_EVERY = 16   # prefill layers between two event-timed prefill launches (4 of 64 per step)
CONFIG = {
    "workload": "prefill fused gate+up M=512 K=5120 N=34816, one step = 64 layer buffers; "
                "decode M=1 K=5120 N=17408, one step = 64 layer buffers",
    "layers_per_step": LAYERS,
    "l2": "inputs larger than L2: 64 distinct layer buffers (2.95 GB prefill, 1.47 GB decode weights)",
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def weight_bytes(N: int, K: int) -> int:
    return N * K // 4 + (K // 128) * N + 4 * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        power = [v for v in (num(r[3]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ CPU oracle timing

def oracle_rate(kind: str, budget_s: float, min_reps: int = 1, M_s=None, N_s=None):
    """Time the CPU oracle, as it stands, on a bounded sample of a workload.

    Returns (rate, unit, sample description, reps, seconds, threads).
    """
    from oracle import ternary_linear as O
    from quantized_linear_layers_block_gb300 import synth

    cfg = PREFILL if kind == "prefill" else DECODE
    M = M_s or cfg["M"]
    N = N_s or (1024 if kind == "prefill" else cfg["N"])
    L = synth.config_inputs(cfg["name"], M=M, N=N)
    reps, t0 = 0, time.perf_counter()
    while True:
        O.layer(L.x_bits, L.codes, L.s)
        reps += 1
        el = time.perf_counter() - t0
        if reps >= min_reps and el >= budget_s:
            break
    threads = os.cpu_count()
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        if info:
            threads = max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    if kind == "prefill":
        rate = 2.0 * M * N * cfg["K"] * reps / el / 1e12
        unit = "TOPS"
    else:
        rate = weight_bytes(N, cfg["K"]) * reps / el / 1e9
        unit = "GB/s"
    sample = (f"oracle.layer (numpy; fp64 BLAS matmul on {threads} threads, the rest one thread) "
              f"on M={M}, N={N} of {cfg['N']} rows, K={cfg['K']}: {reps} rep(s) in {el:.2f} s")
    return rate, unit, sample, reps, el, threads


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def oracle_rate_1core(kind: str, budget_s: float):
    """oracle_rate on the same sample in a fresh interpreter whose BLAS and OpenMP pools have one
    thread (the pools are sized when numpy loads, so this needs its own process). Returns the
    rate, or None if the child failed."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    code = ("import json, bench; r = bench.oracle_rate(%r, %r); print(json.dumps(r[0]))"
            % (kind, budget_s))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True,
                             text=True, timeout=600)
        return float(json.loads(out.stdout.strip().splitlines()[-1]))
    except Exception:
        return None


def reference_main(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    steps = args.steps + args.warmup
    per_step = max(0.02, min(1.0, 90.0 / max(steps, 1)))
    # shrink the sample until one oracle step fits the per-step budget
    M_s, N_s = PREFILL["M"], 1024
    while True:
        el = oracle_rate("prefill", 0.0, 1, M_s, N_s)[4]
        if el <= per_step or (M_s <= 16 and N_s <= 128):
            break
        if N_s > 128:
            N_s //= 2
        else:
            M_s //= 2
    for _ in range(args.warmup):
        oracle_rate("prefill", 0.0, 1, M_s, N_s)
    rate, unit, sample, reps, el, threads = oracle_rate("prefill", 0.0, args.steps, M_s, N_s)
    drate, dunit, dsample, _, _, _ = oracle_rate("decode", 0.0, 1, 1, 2048)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": unit, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / reps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic", "config": dict(CONFIG, parallelism="cpu oracle"),
        "cpu_baseline": {"value": rate, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "decode": {"metric": "decode GEMV weight-stream GB/s @M=1", "value": drate, "unit": dunit,
                   "sample": dsample},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def main(argv=None):
    global LAYERS
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-steps-per-step", type=int, default=32)
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="layer buffers per step (64 = the model's depth; fewer only for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--one", default=None, metavar="KERNEL:WORKLOAD:M",
                    help="instead of the benchmark line: run one kernel (prefill, decode, decode_tc "
                         "or picked) on one layer of a workload five times (for a profiler capture)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload kernel times (down_proj M=256, the M-sweep subset)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the benchmark line: the M sweep 1..4096 over both MLP shapes, "
                         "one JSON line per point (prefill kernel, and decode kernel for M <= 32)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return reference_main(args)
    if args.sweep:
        return sweep_main(args)
    if args.one:
        return one_main(args)

    import torch

    LAYERS = args.layers
    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from quantized_linear_layers_block_gb300 import synth, tl
    from quantized_linear_layers_block_gb300.replicas import Replicas

    reps_ = Replicas(device=dev)      # replicas: no exchange on the data path
    barrier = reps_.barrier
    max_over_ranks = reps_.max

    # ---------------- inputs: 64 layer buffers per workload, resident in HBM
    P, D = PREFILL, DECODE
    pre_layers, dec_layers = [], []
    dec_scales = []
    for li in range(LAYERS):
        codes, s, x = synth.torch_config_layer(P["name"], li, device=str(dev))
        lay = tl.TernaryLinear(codes, s, device=dev)
        del codes, s
        pre_layers.append((lay, x, torch.empty((P["M"], P["N"]), dtype=torch.bfloat16, device=dev)))
        codes, s, x = synth.torch_config_layer(D["name"], li, device=str(dev))
        lay = tl.TernaryLinear(codes, s, device=dev)
        del codes
        dec_layers.append((lay, x, torch.empty((D["M"], D["N"]), dtype=torch.bfloat16, device=dev)))
        dec_scales.append(s.contiguous())
    torch.cuda.synchronize()
    if tl.tl_get_status() != tl.TL_OK:
        raise RuntimeError("device status after packing")

    xq_p = torch.empty((P["M"], P["K"]), dtype=torch.float16, device=dev)
    sx_p = torch.empty((P["M"],), dtype=torch.float32, device=dev)
    xq_d = torch.empty((D["M"], D["K"]), dtype=torch.int8, device=dev)
    xr_d = torch.empty((D["M"], D["K"]), dtype=torch.float32, device=dev)
    sx_d = torch.empty((D["M"],), dtype=torch.float32, device=dev)
    ws_p = pre_layers[0][0]._workspace(P["M"])
    stream = torch.cuda.current_stream(dev)

    def prefill_layer(li, ev=None):
        lay, x, y = pre_layers[li]
        tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_F16, xq=xq_p, sx=sx_p)
        if ev is not None:
            ev[0].record(stream)
        tl.tl_linear_prefill(lay.packed, lay.qT, lay.sw, xq_p, sx_p, P["N"], P["K"], tl.TL_BF16,
                             y=y, workspace=ws_p)
        if ev is not None:
            ev[1].record(stream)

    def decode_layer(li):
        # the decode step: rotate+quantise (K1), then the GEMV (K2)
        lay, x, y = dec_layers[li]
        tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_I8, xq=xq_d, sx=sx_d)
        tl.tl_linear_decode(lay.packed, lay.qT, lay.sw, xq_d, sx_d, D["N"], D["K"], tl.TL_BF16, y=y)

    def decode_kernel_only(li):
        lay, _, y = dec_layers[li]
        tl.tl_linear_decode(lay.packed, lay.qT, lay.sw, xq_d, sx_d, D["N"], D["K"], tl.TL_BF16, y=y)

    def decode_f32act(li):
        lay, x, y = dec_layers[li]
        tl.tl_rotate_act(x, xr=xr_d)
        tl.tl_linear_decode_f32act(lay.packed, dec_scales[li], xr_d, D["N"], D["K"], tl.TL_BF16, y=y)

    def decode_f32act_kernel(li):
        lay, _, y = dec_layers[li]
        tl.tl_linear_decode_f32act(lay.packed, dec_scales[li], xr_d, D["N"], D["K"], tl.TL_BF16, y=y)

    def decode_fused(li):
        lay, x, y = dec_layers[li]
        tl.tl_linear_decode_fused(lay.packed, lay.qT, lay.sw, x, D["N"], D["K"], tl.TL_BF16, y=y)

    # M = 16 at the decode shape: the whole layer as TernaryLinear runs it (K1 with the fp16
    # image, then the mma.sync tensor-core decode), and that kernel alone
    M16 = 16
    _, _, x16 = synth.torch_config_layer(D["name"], 0, M=M16, device=str(dev))
    y16 = torch.empty((M16, D["N"]), dtype=torch.bfloat16, device=dev)
    xq16 = torch.empty((M16, D["K"]), dtype=torch.float16, device=dev)
    sx16 = torch.empty((M16,), dtype=torch.float32, device=dev)
    ws16 = dec_layers[0][0]._workspace(M16)
    tl.tl_rotate_quant_act(x16, xq_dtype=tl.TL_F16, xq=xq16, sx=sx16)

    def layer16(li):
        dec_layers[li][0].forward(x16, out=y16)

    kind16 = dec_layers[0][0].kernel_for(M16)

    def kernel16(li):
        lay = dec_layers[li][0]
        if kind16 == "decode_tc":
            tl.tl_linear_decode_tc(lay.packed, lay.qT, lay.sw, xq16, sx16, D["N"], D["K"],
                                   tl.TL_BF16, y=y16)
        else:
            tl.tl_linear_prefill(lay.packed, lay.qT, lay.sw, xq16, sx16, D["N"], D["K"], tl.TL_BF16,
                                 y=y16, workspace=ws16)

    # warm-up (also resolves driver entry points and kernel attributes before capture)
    for _ in range(args.warmup):
        for li in range(LAYERS):
            prefill_layer(li)
            decode_layer(li)
    torch.cuda.synchronize()

    g_dec = torch.cuda.CUDAGraph()
    g_dk = torch.cuda.CUDAGraph()
    g_df = torch.cuda.CUDAGraph()
    g_ff = torch.cuda.CUDAGraph()
    g_fk = torch.cuda.CUDAGraph()
    for li in range(LAYERS):          # resolve the float decode's kernel attributes before capture
        decode_f32act(li)
    torch.cuda.synchronize()
    with torch.cuda.graph(g_ff, capture_error_mode="relaxed"):
        for li in range(LAYERS):
            decode_f32act(li)
    with torch.cuda.graph(g_fk, capture_error_mode="relaxed"):
        for li in range(LAYERS):
            decode_f32act_kernel(li)
    with torch.cuda.graph(g_dec, capture_error_mode="relaxed"):
        for li in range(LAYERS):
            decode_layer(li)
    with torch.cuda.graph(g_dk, capture_error_mode="relaxed"):
        for li in range(LAYERS):
            decode_kernel_only(li)
    with torch.cuda.graph(g_df, capture_error_mode="relaxed"):
        for li in range(LAYERS):
            decode_fused(li)
    g_16 = torch.cuda.CUDAGraph()
    g_16k = torch.cuda.CUDAGraph()
    for li in range(LAYERS):
        layer16(li)
    torch.cuda.synchronize()
    with torch.cuda.graph(g_16, capture_error_mode="relaxed"):
        for li in range(LAYERS):
            layer16(li)
    with torch.cuda.graph(g_16k, capture_error_mode="relaxed"):
        for li in range(LAYERS):
            kernel16(li)
    for _ in range(args.warmup):
        g_dec.replay()
        g_dk.replay()
        g_df.replay()
        g_ff.replay()
        g_fk.replay()
        g_16.replay()
        g_16k.replay()
    torch.cuda.synchronize()
    if tl.tl_get_status() != tl.TL_OK:
        raise RuntimeError("device status after warm-up")

    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else f"GPU-{uuid}")
    clocks.start()

    # ---------------- timed prefill: K steps, each the batch through the layers.
    # The prefill kernel's own duration is taken with CUDA events around the
    # launches of every EVENT_EVERY-th layer: an event recorded between two
    # launches ends the programmatic-launch overlap of the next kernel's
    # prologue with the previous one (about 10 us per layer when every layer
    # carries events), so the sampled layers pay it and the rest run as a
    # plain model step does.
    K = args.steps
    sampled = [li for li in range(LAYERS) if li % EVENT_EVERY == 0]
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K * len(sampled))]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    i = 0
    for _ in range(K):
        for li in range(LAYERS):
            if li % EVENT_EVERY == 0:
                prefill_layer(li, evs[i])
                i += 1
            else:
                prefill_layer(li)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    pre_ms = max_over_ranks(t_start.elapsed_time(t_end))
    k3_ms = statistics.fmean(a.elapsed_time(b) for a, b in evs)

    # ---------------- timed decode: Kd steps (graph replays), each 1 token through the layers
    Kd = K * args.decode_steps_per_step
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for _ in range(Kd):
        g_dec.replay()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    dec_ms = max_over_ranks(t_start.elapsed_time(t_end))
    clk = clocks.stop()

    # the GEMV kernel alone, 64 back-to-back launches on the layer buffers: its
    # average duration is the roofline figure; then the fused single-launch layer
    def graph_us(g, reps):
        t_start.record(stream)
        for _ in range(reps):
            g.replay()
        t_end.record(stream)
        torch.cuda.synchronize()
        return 1e3 * t_start.elapsed_time(t_end) / (reps * LAYERS)

    reps = max(8, Kd // 4)
    k2_ms = graph_us(g_dk, reps) * 1e-3
    fused_us = graph_us(g_df, reps)
    f32_layer_us = graph_us(g_ff, reps)
    f32_kernel_us = graph_us(g_fk, reps)
    m16_layer_us = graph_us(g_16, reps)
    m16_kernel_us = graph_us(g_16k, reps)
    status = tl.tl_get_status()
    if status != tl.TL_OK:
        raise RuntimeError(f"device status after timing: {tl.tl_strerror(status)}")

    # ---------------- int8 128-group codec (compress, decompress-and-add), 1584 x 5120
    codec = codec_bench(dev, stream, max(4, args.warmup), max(8, K))

    # ---------------- end to end through the public API with pinned host buffers: every
    # step copies each layer's input in and its output back, synchronised at the end of
    # the step (prefill: tl.HostPipeline overlaps the copies with the neighbouring layers'
    # kernels)
    e2e_steps = 0 if args.no_e2e else max(1, min(K, 8))
    e2e_dsteps = 0 if args.no_e2e else max(1, min(Kd, 64))
    xh_p = [x.cpu().pin_memory() for _, x, _ in pre_layers]
    xh_d = [x.cpu().pin_memory() for _, x, _ in dec_layers]
    yh_p = [torch.empty((P["M"], P["N"]), dtype=torch.bfloat16).pin_memory() for _ in range(LAYERS)]
    yh_d = [torch.empty((D["M"], D["N"]), dtype=torch.bfloat16).pin_memory() for _ in range(LAYERS)]
    pipe = tl.HostPipeline(dev)
    for li in range(LAYERS):                       # warm the pipeline's buffers
        pipe.submit(pre_layers[li][0], xh_p[li], yh_p[li])
        pipe.submit(dec_layers[li][0], xh_d[li], yh_d[li])
    pipe.synchronize()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for li in range(LAYERS):
            pipe.submit(pre_layers[li][0], xh_p[li], yh_p[li])
        pipe.synchronize()
    e2e_pre_s = max(max_over_ranks(time.perf_counter() - t0), 1e-9)
    # decode: the whole step (64 x: copy in, rotate+quantise, decode, copy out) is one
    # CUDA graph (tl.GraphStep), one host launch per step
    dstep = tl.GraphStep([dec_layers[li][0] for li in range(LAYERS)], [D["M"]] * LAYERS, dev)
    for li in range(LAYERS):
        dstep.inputs[li].copy_(xh_d[li])
    for _ in range(3):
        dstep.run()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_dsteps):
        dstep.run()
    e2e_dec_s = max(max_over_ranks(time.perf_counter() - t0), 1e-9)

    # ---------------- the other workloads: down_proj at 256 tokens and a subset of the M sweep
    # over both MLP shapes (kernel time per layer, 8 layer buffers each, outside the timed steps)
    peaks0, _ = load_peaks()
    configs = None
    if not args.no_configs:
        configs = time_points(tl, synth, dev, stream,
                              [("down_proj", 256)] + [(nm, m) for nm in ("sweep_up", "sweep_down")
                                                      for m in CONFIG_SWEEP_M],
                              hbm_peak=float(peaks0.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                              tc_peak=float(peaks0.get("bf16_tflops_sustained",
                                                       FALLBACK_PEAKS["bf16_tflops_sustained"])))

    # ---------------- figures
    flop_layer = 2.0 * P["M"] * P["N"] * P["K"]
    tops = ws * K * LAYERS * flop_layer / (pre_ms * 1e-3) / 1e12
    wb = weight_bytes(D["N"], D["K"])
    gbs = ws * Kd * LAYERS * wb / (dec_ms * 1e-3) / 1e9
    peaks, peak_src = load_peaks()
    tc_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    k3_tops = flop_layer / (k3_ms * 1e-3) / 1e12
    dec_alg_bytes = wb + D["M"] * D["K"] + 4 * D["M"] + 2 * D["M"] * D["N"]
    k2_gbs = dec_alg_bytes / (k2_ms * 1e-3) / 1e9
    traffic = _profiled_traffic()
    flop16 = 2.0 * 16 * D["N"] * D["K"]

    line = {
        "metric": METRIC, "value": tops, "unit": "TOPS", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": pre_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": dict(CONFIG, layers_per_step=LAYERS, parallelism=f"replicas x{ws}"),
        "roofline": {"bound": "tensor", "achieved": k3_tops, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": k3_tops / tc_peak, "traffic": traffic.get("prefill_kernel"),
                     "kernel": "prefill_kernel (K3)",
                     "timing": f"CUDA events around the prefill launch of every {EVENT_EVERY}th "
                               f"layer of the timed steps ({K * len(sampled)} launches)",
                     # the kernel runs inside a long dense step (the power cap applies), hence
                     # the sustained peak; the fraction of the burst peak beside it
                     "timed_region_s": pre_ms * 1e-3,
                     "frac_burst": k3_tops / float(peaks.get("bf16_tflops",
                                                             FALLBACK_PEAKS["bf16_tflops"])),
                     "peak_source": f"{peak_src} bf16_tflops_sustained (the int8 GEMM runs on "
                                    "kind::f16 tensor cores; fp16 and bf16 share the rate)"},
        "decode": {
            "metric": "decode GEMV weight-stream GB/s @M=1", "value": gbs, "unit": "GB/s",
            "steps": Kd, "ms_per_step": dec_ms / Kd, "layer_us": dec_ms * 1e3 / (Kd * LAYERS),
            "kernel_us": k2_ms * 1e3, "fused_layer_us": fused_us,
            "roofline": {"bound": "hbm", "achieved": k2_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": k2_gbs / hbm_peak, "traffic": traffic.get("decode_kernel"),
                         "kernel": "decode1_kernel (K2) M=1, graph of 64 back-to-back launches",
                         "peak_source": f"{peak_src} hbm_gbs"},
            "e2e": {"value": ws * e2e_dsteps * LAYERS * wb / e2e_dec_s / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": LAYERS * D["M"] * D["K"] * 2,
                    "d2h_bytes_per_step": LAYERS * D["M"] * D["N"] * 2},
        },
        "kernels_us": {"prefill_kernel": k3_ms * 1e3, "decode_kernel": k2_ms * 1e3,
                       "prefill_step_rest": (pre_ms / (K * LAYERS) - k3_ms) * 1e3},
        "e2e": {"value": ws * e2e_steps * LAYERS * flop_layer / e2e_pre_s / 1e12, "unit": "TOPS",
                "h2d_bytes_per_step": LAYERS * P["M"] * P["K"] * 2,
                "d2h_bytes_per_step": LAYERS * P["M"] * P["N"] * 2},
        "decode16": {
            "metric": "ternary linear int8 TOPS @M=16, decode shape (K=5120, N=17408)",
            "value": flop16 / (m16_layer_us * 1e-6) / 1e12, "unit": "TOPS",
            "layer_us": m16_layer_us, "kernel_us": m16_kernel_us,
            "kernel": f"{kind16} (TernaryLinear's choice for M = 16 at K = 5120); 64 layer "
                      "buffers in a CUDA graph",
            # the operation at M = 16 moves 23 MB of weights for 2.85 GOP: HBM-bound against
            # the measured peaks (the weight stream takes longer than the tensor work)
            "roofline": {"bound": "hbm", "achieved": wb / (m16_kernel_us * 1e-6) / 1e9,
                         "peak": hbm_peak, "unit": "GB/s",
                         "frac": wb / (m16_kernel_us * 1e-6) / 1e9 / hbm_peak,
                         "peak_source": f"{peak_src} hbm_gbs",
                         "floor_us": wb / hbm_peak / 1e3,
                         "traffic": traffic.get("prefill_kernel_narrow_M16" if kind16 == "prefill"
                                                else "decode_tc_kernel")},
        },
        "decode_f32act": {
            "metric": "float-activation decode GEMV weight-stream GB/s @M=1",
            "layer_us": f32_layer_us, "kernel_us": f32_kernel_us,
            "value": wb / (f32_layer_us * 1e-6) / 1e9, "unit": "GB/s",
            "kernel_GB/s": (wb + 2 * D["N"] * (D["K"] // 128) + 4 * D["K"]) / (f32_kernel_us * 1e-6) / 1e9,
            "bound": "alu",
            "note": "rotation (fp32) then the fp32 GEMV from packed codes and fp16 scales; "
                    "64 layer buffers in a CUDA graph",
        },
        "codec": codec,
        "configs": configs,
        "gpu_launches": K * LAYERS * 2 + Kd * LAYERS * 2,
        "clocks": clk,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, unit, sample, _, _, threads = oracle_rate("prefill", 10.0)
        line["cpu_baseline"] = {"value": rate, "unit": unit, "cores": threads, "kind": "oracle",
                                "sample": sample, "cpu": cpu_model(),
                                "value_1core": oracle_rate_1core("prefill", 10.0)}
        drate, dunit, dsample, _, _, _ = oracle_rate("decode", 5.0)
        line["decode"]["cpu_baseline"] = {"value": drate, "unit": dunit, "cores": threads,
                                          "kind": "oracle", "sample": dsample,
                                          "value_1core": oracle_rate_1core("decode", 5.0)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    reps_.close()
    return 0


def time_points(tl, synth, dev, stream, points, nl: int = 8, hbm_peak=None, tc_peak=None) -> list:
    """Kernel time per layer of named workloads at given token counts.

    points: (workload name, M) pairs. For each workload `nl` layer buffers
    (larger than L2 together) are drawn with its recipe; for each M the kernel
    TernaryLinear picks runs over the buffers in a CUDA graph (rotate+quantise
    outside the timed launches), and the prefill kernel beside it when that is
    not the one picked. Returns one dict per point with the times, TOPS,
    weight GB/s and the roofline of the picked kernel: HBM-bound below the
    M where the weight stream and the tensor work take equally long at the
    measured peaks, tensor-bound above."""
    import torch
    out = []
    cache = {}
    for name, M in points:
        if name not in cache:
            cache.clear()
            layers = []
            for li in range(nl):
                codes, s_, _ = synth.torch_config_layer(name, li, M=1, device=str(dev))
                layers.append(tl.TernaryLinear(codes, s_, device=dev))
                del codes, s_
            cache[name] = layers
        layers = cache[name]
        N, K = layers[0].N, layers[0].K
        _, _, x = synth.torch_config_layer(name, 1000, M=M, device=str(dev))
        xq16, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_F16)
        xq8, _ = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_I8)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = layers[0]._workspace(M)
        fns = {
            "prefill": lambda l: tl.tl_linear_prefill(l.packed, l.qT, l.sw, xq16, sx, N, K, tl.TL_BF16,
                                                      y=y, workspace=ws),
            "decode": lambda l: tl.tl_linear_decode(l.packed, l.qT, l.sw, xq8, sx, N, K, tl.TL_BF16, y=y),
            "decode_tc": lambda l: tl.tl_linear_decode_tc(l.packed, l.qT, l.sw, xq16, sx, N, K,
                                                          tl.TL_BF16, y=y),
        }
        picked = layers[0].kernel_for(M)
        kinds = [picked] + (["prefill"] if picked != "prefill" else [])
        wb = weight_bytes(N, K)
        line = {"workload": name, "M": M, "K": K, "N": N, "kernel": picked}
        for kind in kinds:
            fn = fns[kind]
            for l in layers:
                fn(l)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()          # no host launch cost between the kernels
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                for l in layers:
                    fn(l)
            g.replay()
            torch.cuda.synchronize()
            reps = max(3, min(40, int(4e5 // max(M, 64))))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            us = 1e3 * e0.elapsed_time(e1) / (reps * nl)
            key = "us" if kind == picked else f"{kind}_us"
            line[key] = round(us, 2)
            if kind == picked:
                line["tops"] = round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1)
                line["weight_GB/s"] = round(wb / (us * 1e-6) / 1e9, 1)
                if hbm_peak and tc_peak:
                    flops = 2.0 * M * N * K
                    if wb / (hbm_peak * 1e9) >= flops / (tc_peak * 1e12):
                        line["roofline"] = {"bound": "hbm", "frac": round(wb / (us * 1e-6) / 1e9 / hbm_peak, 3)}
                    else:
                        line["roofline"] = {"bound": "tensor",
                                            "frac": round(flops / (us * 1e-6) / 1e12 / tc_peak, 3)}
        if tl.tl_get_status() != tl.TL_OK:
            raise RuntimeError(f"device status during {name} M={M}")
        out.append(line)
    return out


def one_main(args) -> int:
    """One kernel on one layer of a workload, five launches (for ncu captures)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_linear_layers_block_gb300 import synth, tl
    kind, name, m = args.one.split(":")
    M = int(m)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    codes, s_, x = synth.torch_config_layer(name, 0, M=M, device=str(dev))
    lay = tl.TernaryLinear(codes, s_, device=dev)
    N, K = lay.N, lay.K
    if kind == "picked":
        kind = lay.kernel_for(M)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_I8 if kind == "decode" else tl.TL_F16)
    for _ in range(5):
        if kind == "decode":
            tl.tl_linear_decode(lay.packed, lay.qT, lay.sw, xq, sx, N, K, tl.TL_BF16, y=y)
        elif kind == "decode_tc":
            tl.tl_linear_decode_tc(lay.packed, lay.qT, lay.sw, xq, sx, N, K, tl.TL_BF16, y=y)
        else:
            tl.tl_linear_prefill(lay.packed, lay.qT, lay.sw, xq, sx, N, K, tl.TL_BF16, y=y,
                                 workspace=lay._workspace(M))
    torch.cuda.synchronize()
    st = tl.tl_get_status()
    print(json.dumps({"one": args.one, "kernel": kind, "M": M, "N": N, "K": K, "status": st}))
    return 0 if st == tl.TL_OK else 1


def sweep_main(args) -> int:
    """The M sweep of the workloads (one JSON line per point; see time_points)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from quantized_linear_layers_block_gb300 import synth, tl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, _ = load_peaks()
    points = [(name, M) for name in ("sweep_up", "sweep_down") for M in synth.SWEEP_M]
    for line in time_points(tl, synth, dev, stream, points,
                            hbm_peak=float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                            tc_peak=float(peaks.get("bf16_tflops_sustained",
                                                    FALLBACK_PEAKS["bf16_tflops_sustained"]))):
        print(json.dumps(line), flush=True)
    return 0


def codec_bench(dev, stream, warmup: int, reps: int) -> dict:
    """Times tl_codec_quant and tl_codec_dequant_add (one peer) on the 1584 x 5120
    payload, rotating over 16 payload buffers (260 MB of bf16, larger than L2)."""
    import torch
    from quantized_linear_layers_block_gb300 import synth, tl
    c = synth.CODEC
    R, H, nb = c["R"], c["H"], 16
    own = synth.torch_codec_parts(c["seed"], R, H, nb, c["outlier_frac"], c["outlier_factor"], device=str(dev))
    q = [torch.empty((1, R, H), dtype=torch.int8, device=dev) for _ in range(nb)]
    sc = [torch.empty((1, R, H // 128), dtype=torch.float32, device=dev) for _ in range(nb)]
    out = [torch.empty((R, H), dtype=torch.bfloat16, device=dev) for _ in range(nb)]

    def run_quant(i):
        tl.tl_codec_quant(own[i], q=q[i][0], scale=sc[i][0])

    def run_dq(i):
        tl.tl_codec_dequant_add(own[i], q[(i + 1) % nb], sc[(i + 1) % nb], out=out[i])

    res = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    bytes_q = 2 * R * H + R * H + 4 * R * (H // 128)
    bytes_dq = 2 * R * H + R * H + 4 * R * (H // 128) + 2 * R * H
    peaks, _ = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    for name, fn, nbytes in (("quant", run_quant, bytes_q), ("dequant_add", run_dq, bytes_dq)):
        for i in range(nb):          # resolve attributes before capture
            fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()   # one graph of nb launches: no host launch cost inside
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for i in range(nb):
                fn(i)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / (reps * nb)
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us": us, "GB/s": gbs, "bytes": nbytes, "frac_hbm": gbs / hbm}
    if tl.tl_get_status() != tl.TL_OK:
        raise RuntimeError("device status after the codec timing")
    res["workload"] = f"R={R} H={H} bf16, one peer; 16 payload buffers (larger than L2)"
    res["launches"] = 2 * nb * (reps + warmup + 2)
    return res


def _profiled_traffic() -> dict:
    """DRAM bytes per launch of the current kernels from the committed ncu summary, if any."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


if __name__ == "__main__":
    sys.exit(main())
