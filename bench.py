"""Benchmark of the fused Conv1d + normalization operator on GB300.

Default workload: Conv1d(128 -> 256, k=3, pad 1/1) + GroupNorm(32) on x[16, 128, 1024] fp32 (TF32
tensor cores), the configuration the headline metric is quoted on. One step = the whole hot path:
weight packing + the fused conv/statistics/normalize kernel, through the C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Under torchrun every rank runs the same per-GPU workload on its own GPU and its own seeded batch
(weak scaling, no collective on the data path); the timed region is bracketed by a barrier and a
device synchronize, and the slowest rank's time is reported. `--impl reference` times the CPU
oracle on the host cores instead (rank 0 only).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense TF32 / BF16 tensor rate


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.device_index = device_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def workload_by_name(name):
    if name in synth.BY_NAME:
        return synth.BY_NAME[name]
    if name in ("ln_avgpool3d_gelu", synth.LN_AVGPOOL3D_GELU.name):
        return synth.LN_AVGPOOL3D_GELU
    if name in ("p4", "conv_transpose3d", synth.CONV_TRANSPOSE3D.name):
        return synth.CONV_TRANSPOSE3D
    short = {"conv_gn": synth.CONV_GN, "conv_gn_tiny": synth.CONV_GN_TINY, "causal_conv": synth.CAUSAL_CONV,
             "linear_gn_rowmin": synth.LINEAR_GN_ROWMIN, "conv_ln_gelu_bf16": synth.CONV_LN_GELU_BF16,
             "causal_conv_gn32": synth.CAUSAL_CONV_GN32}
    return short[name]


def config_of(wl, extra):
    cfg = {"workload": wl.name, "N": wl.N, "C_in": wl.C_in, "C_out": wl.C_out, "T": wl.T, "k": wl.k,
           "stride": wl.stride, "pad": [wl.pad_left, wl.pad_right], "dilation": wl.dilation,
           "norm": ["none", "group", "channel_layer"][wl.norm], "groups": wl.groups,
           "post": ["none", "gelu_erf", "rowmin_bias"][wl.post], "T_out": wl.T_out,
           "gemm_mnk": list(wl.gemm_mnk)}
    cfg.update(extra)
    return cfg


def dtype_name(wl, path, math=0):
    if wl.dtype == synth.DTYPE_BF16:
        return "bf16"
    if path == "simt":
        return "f32"
    return "tf32x3" if math == 3 else "tf32"


# ------------------------------------------------------------------------------------------ oracle arm

def time_oracle(wl, seconds=10.0, max_runs=50, n_rows=None, single_seconds=0.0):
    """Time the CPU oracle on `n_rows` batch entries of the workload (whole workload by default), on
    all host cores; with single_seconds > 0 also on one thread (one batch entry per run)."""
    import oracle
    rows = wl.N if n_rows is None else n_rows
    sub = wl.replace(N=rows)
    inp = synth.make_inputs(wl, seed=0, n_rows=rows)
    p = oracle.params_of(sub)
    threads = oracle.default_threads()
    oracle.conv1d_norm(p, inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"], inp["bias2"], nthreads=threads)
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.conv1d_norm(p, inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"], inp["bias2"],
                           nthreads=threads)
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds or runs >= max_runs:
            break
    flops = sub.flops * runs
    out = {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{runs} run(s) of the full operator on {rows} of {wl.N} batch entries "
                     f"({sub.flops / 1e9:.3f} GFLOP each), {el:.1f} s wall"}
    if single_seconds > 0:
        one = wl.replace(N=1)
        inp1 = synth.make_inputs(wl, seed=0, n_rows=1)
        p1 = oracle.params_of(one)
        runs1, t1 = 0, time.perf_counter()
        while True:
            oracle.conv1d_norm(p1, inp1["x"], inp1["w"], inp1["b"], inp1["gamma"], inp1["beta"], inp1["bias2"],
                               nthreads=1)
            runs1 += 1
            el1 = time.perf_counter() - t1
            if el1 >= single_seconds or runs1 >= max_runs:
                break
        out["single_thread"] = {"value": one.flops * runs1 / el1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                                "sample": f"{runs1} run(s) on 1 batch entry ({one.flops / 1e9:.3f} GFLOP "
                                          f"each), {el1:.1f} s wall"}
    return out


def reference_arm(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    rows = max(1, min(wl.N, args.oracle_rows))
    sub = wl.replace(N=rows)
    inp = synth.make_inputs(wl, seed=0, n_rows=rows)
    p = oracle.params_of(sub)
    threads = oracle.default_threads()
    run = lambda: oracle.conv1d_norm(p, inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"], inp["bias2"],
                                     nthreads=threads)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    value = sub.flops / (ms / 1e3) / 1e12
    line = {"impl": "reference", "metric": args.metric, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, {"oracle_rows_per_step": rows}),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: the full operator on {rows} of {wl.N} batch entries"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------ our arm

EXTRA_WORKLOADS = ("conv_gn_tiny", "causal_conv", "linear_gn_rowmin", "conv_ln_gelu_bf16")
# forced two-pass plans on the largest outputs: where the memory-bound normalize pass is measured
NORMALIZE_PASS_WORKLOADS = ("causal_conv_gn32", "conv_ln_gelu_bf16")


class ConvRun:
    """One operator configuration through the C ABI on device-resident inputs: the descriptor, its
    rank's inputs, rotating x / y buffer sets (more than 2x L2 of them unless one set already
    exceeds L2) and CUDA graphs of whole steps (every kernel of the operator, as the library
    enqueues them): one per set, and for the timed blocks one graph of a block's K steps."""

    def __init__(self, c1n, wl, args, dev, rank, math_mode=None, path=None, mainloop=None):
        import torch
        self.torch, self.wl, self.dev = torch, wl, dev
        math_mode = args.math if math_mode is None else math_mode
        path = args.path if path is None else path
        mainloop = args.mainloop if mainloop is None else mainloop
        params = c1n.make_params(wl.N, wl.C_in, wl.C_out, wl.T, wl.k, wl.stride, wl.pad_left, wl.pad_right,
                                 wl.dilation, wl.norm, wl.groups, wl.eps, wl.post, wl.dtype, math_mode, path, mainloop)
        self.op = op = c1n.Conv1dNorm(params, device=dev)
        self.path, self.math = op.path, math_mode
        # Weak scaling: rank r runs the per-GPU workload on batch rows [r*N, (r+1)*N) of one global
        # batch of world*N entries (GroupNorm / LayerNorm / row-min statistics are per sample or per
        # row, so no data crosses ranks).
        self.inp = inp = shard_inputs(wl, rank)
        self.bf = bf = wl.dtype == synth.DTYPE_BF16
        self.tdt = tdt = torch.bfloat16 if bf else torch.float32

        def dev_t(a, cast=True):
            if a is None:
                return None
            t = torch.from_numpy(a).to(dev)
            return t.to(tdt) if (cast and bf) else t

        self.w = dev_t(inp["w"])
        self.b, self.ga, self.be, self.b2 = (dev_t(inp[k], cast=False) for k in ("b", "gamma", "beta", "bias2"))
        x0 = dev_t(inp["x"])
        self.y_shape = (wl.N, wl.C_out, op.T_out)
        self.per_set = x0.numel() * x0.element_size() + int(np.prod(self.y_shape)) * (2 if bf else 4)
        self.n_sets = 1 if self.per_set >= L2_BYTES else min(16, math.ceil(2 * L2_BYTES / self.per_set))
        self.xs = [x0] + [x0.clone() for _ in range(self.n_sets - 1)]
        self.ys = [torch.empty(self.y_shape, dtype=op.out_dtype(), device=dev) for _ in range(self.n_sets)]
        self.am = (torch.empty((wl.N, op.T_out), dtype=torch.int32, device=dev)
                   if wl.post == synth.POST_ROWMIN_BIAS else None)
        self.stream = torch.cuda.current_stream(dev)
        self.graphs = None
        self.block_graphs = {}
        # kernels of one step, and of one call with the weights already packed
        self.kernels = op.info.kernels
        self.kernels_packed = self.kernels - (1 if self.path not in ("simt", "tc_linear") else 0)

    def step(self, i):
        j = i % self.n_sets
        self.op(self.xs[j], self.w, self.b, self.ga, self.be, bias2=self.b2, out=self.ys[j], argmin=self.am)

    def packed_call(self, i):
        j = i % self.n_sets
        self.op(self.xs[j], self.w, self.b, self.ga, self.be, bias2=self.b2, out=self.ys[j], argmin=self.am,
                weights_packed=True)

    def prepare(self, warmup, eager=False):
        for i in range(warmup):
            self.step(i)
        self.torch.cuda.synchronize()
        self.op.check()
        self.graphs = None if eager else capture_graphs(self.step, self.n_sets, self.dev)
        for i in range(max(3, warmup)):
            self.run_step(i)
        self.torch.cuda.synchronize()

    def run_step(self, i):
        if self.graphs:
            self.graphs[i % self.n_sets].replay()
        else:
            self.step(i)

    @property
    def launch_mode(self):
        return ("one CUDA graph per timed block, holding its K steps (each step one operator call, x / y "
                "rotating over the buffer sets)" if self.graphs else "eager")

    def run_block(self, steps, i0):
        """Steps i0 .. i0 + steps - 1: one replay of a graph of those K steps (captured once per K
        and starting buffer set), or the eager loop."""
        if not self.graphs:
            for k in range(steps):
                self.step(i0 + k)
            return
        key = (steps, i0 % self.n_sets)
        if key not in self.block_graphs:
            g = capture_graphs(lambda j: [self.step(i0 + k) for k in range(steps)], 1, self.dev)
            self.block_graphs[key] = g[0] if g else None
        g = self.block_graphs[key]
        if g is None:
            for k in range(steps):
                self.run_step(i0 + k)
        else:
            g.replay()

    def timed_blocks(self, steps, min_seconds, barrier, pg=None, i0=0):
        """Time back-to-back blocks of exactly `steps` steps, each bracketed by a barrier and a device
        synchronize on both sides and timed with CUDA events on the launching stream, until the blocks
        cover at least `min_seconds` (3 blocks at least). Every block runs steps i0 .. i0 + K - 1 (one
        replay of the same block graph; consecutive steps use different buffer sets, and so do the
        last step of a block and the first of the next when there are several sets). Returns (ms
        per step of each block, max over ranks)."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if self.n_sets > 1 and (steps - 1) % self.n_sets == 0:
            i0_next = 1  # (K - 1) a multiple of the set count: shift alternate blocks by one set
        else:
            i0_next = 0
        starts = [i0, i0 + i0_next]
        for i in starts:  # capture and warm the block graphs before timing
            self.run_block(steps, i)
        torch.cuda.synchronize()

        def block(i):
            barrier()
            torch.cuda.synchronize()
            e0.record(self.stream)
            self.run_block(steps, i)
            e1.record(self.stream)
            torch.cuda.synchronize()
            barrier()
            return e0.elapsed_time(e1) / steps

        first = block(starts[0])
        n_blocks = max(3, math.ceil(min_seconds * 1e3 / max(first * steps, 1e-3)))
        if pg is not None:  # every rank runs the same number of blocks
            t = torch.tensor([n_blocks], device=self.dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            n_blocks = int(t[0])
        ms = [block(starts[(r + 1) % 2]) for r in range(n_blocks)]
        if pg is not None:
            t = torch.tensor(ms, device=self.dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            ms = [float(v) for v in t]
        self.op.check()
        return ms

    def back_to_back_ms(self, launches=20, reps=10):
        """Mean device time of one operator call with the weights already packed, from one CUDA
        graph of `launches` calls back to back (inputs rotating over the buffer sets), timed with
        CUDA events around `reps` replays. With one kernel per call this is that kernel's average
        launch duration. None when the graph cannot be captured. (A plan without a separate weight
        pack is timed as it runs in a step.)"""
        torch = self.torch
        call = self.step if self.kernels_packed == self.kernels else self.packed_call
        if call is self.packed_call:
            self.op.pack_weights(self.w)
        g = capture_graphs(lambda j: [call(i) for i in range(launches)], 1, self.dev)
        if not g:
            return None
        for _ in range(2):
            g[0].replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for _ in range(reps):
            g[0].replay()
        e1.record(self.stream)
        torch.cuda.synchronize()
        self.op.check()
        return e0.elapsed_time(e1) / (reps * launches)

    def kernel_marks(self, i0):
        """Per-kernel device times of one step from the library's event marks (an event pair around
        each kernel inside a replayed graph: each time includes the pair's own overhead)."""
        return kernel_times(self.op, self.step, i0, self.dev, n=5, graphs=bool(self.graphs))

    def close(self):
        self.op.close()
        self.graphs = None
        self.xs = self.ys = None
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def conv_roofline(wl, run, peaks, kern, b2b_ms):
    """Roofline entry of the dominant kernel (the conv kernel with its fused epilogue). Algorithmic
    bytes: x and w read once, the per-channel parameters, and the conv kernel's output written once
    (y, or the fp32 raw tile on the two-pass plans); FLOPs = 2 M N K."""
    path = run.path
    flops = wl.flops
    nbytes = wl.algorithmic_bytes
    y_elems = wl.N * wl.C_out * wl.T_out
    if kern.get("normalize") is not None or kern.get("rowmin") is not None:
        nbytes += y_elems * (4 - wl.elem_bytes)  # raw fp32 tile instead of y
    conv_name = "simt_conv" if path == "simt" else "tc_conv"
    if b2b_ms is not None and run.kernels_packed == 1:
        conv_ms = b2b_ms
        timing = ("back to back: one CUDA graph of 20 launches of the kernel"
                  + ("" if run.kernels_packed == run.kernels else " (weights packed once)")
                  + ", events around the replays")
    elif b2b_ms is not None and conv_name == "tc_conv" and path == "tc_linear":
        conv_ms = b2b_ms  # conservative: includes the small finisher kernel that follows it
        timing = ("back to back: graph of 20 operator calls (this kernel + the row-min finisher), events around the "
                  "replays; the finisher's time is counted against this kernel")
    else:
        conv_ms = kern.get(conv_name, b2b_ms)
        timing = "event pair around the kernel inside a replayed graph (includes the pair's own overhead: an upper bound)"
    # The kernel is timed after seconds of back-to-back calls (the timed blocks come first), where
    # the power cap sets the clock: the tensor peak is the sustained cuBLAS figure, the burst one
    # is reported beside it.
    ratio = 1.0 if run.bf else TF32_PER_BF16
    tc_peak = peaks["bf16_tflops_sustained"] * ratio
    tc_burst = peaks["bf16_tflops"] * ratio
    t_flop = flops / (tc_peak * 1e12)
    t_byte = nbytes / (peaks["hbm_gbs"] * 1e9)
    if path == "simt":
        ach = flops / (conv_ms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": ach, "peak": FP32_FMA_PEAK_TFLOPS, "unit": "TFLOP/s",
                "frac": ach / FP32_FMA_PEAK_TFLOPS}
    elif t_byte >= t_flop:
        ach = nbytes / (conv_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
    else:
        ach = flops / (conv_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s", "frac": ach / tc_peak,
                "frac_of_burst_peak": ach / tc_burst}
    roof.update({"traffic": read_traffic(wl.name, path),
                 "peak_source": peaks["source"] + ("" if run.bf else " (bf16 x 1.1/2.25 for tf32)"),
                 "peak_kind": ("copy bandwidth" if roof["bound"] == "hbm" else
                               "sustained (the kernel is timed after seconds of back-to-back calls)"
                               if roof["bound"] == "tensor" else "derived"),
                 "kernel": f"tc_conv_kernel ({path})" if path != "simt" else "simt_conv_kernel",
                 "kernel_ms": conv_ms, "kernel_timing": timing, "kernels_ms_event_pairs": kern,
                 "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                 "tensor_frac": (flops / (conv_ms / 1e3) / 1e12) / tc_peak,
                 "hbm_frac": (nbytes / (conv_ms / 1e3) / 1e9) / peaks["hbm_gbs"]})
    return roof


def rowmin_finisher(wl, kern, peaks):
    """GB/s of the row-min finisher (per-(row, channel block) partials read, y and argmin written)
    from its event-pair time (an upper bound on the kernel time, so a lower bound on GB/s)."""
    ms = kern.get("rowmin_finish")
    if not ms:
        return None
    n_cb = -(-wl.C_out // 256)
    nbytes = wl.N * wl.T_out * (n_cb * 8 + 4) + wl.N * wl.C_out * wl.T_out * wl.elem_bytes + 4 * wl.C_out
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"kernel": "rowmin_finish_kernel", "ms_event_pair": ms, "bytes": nbytes, "GB/s": gbs,
            "frac": gbs / peaks["hbm_gbs"]}


def measure_workload(c1n, wl, args, dev, rank, peaks, steps, min_seconds, barrier, pg=None, path=None):
    """One workload measured the way the headline is (without e2e and oracle legs): returns a dict
    for the line's `workloads` object."""
    run = ConvRun(c1n, wl, args, dev, rank, path=path)
    sampler = None
    try:
        run.prepare(args.warmup, eager=args.eager)
        sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
        if sampler:
            sampler.start()
        ms_blocks = run.timed_blocks(steps, min_seconds, barrier, pg)
        ms = statistics.median(ms_blocks)
        kern = run.kernel_marks(args.warmup + steps)
        b2b = run.back_to_back_ms()
        clocks = sampler.stop() if sampler else None
        sampler = None
        roof = conv_roofline(wl, run, peaks, kern, b2b)
        out = {"workload": wl.name, "gemm_mnk": list(wl.gemm_mnk), "plan": run.path,
               "cta_pair": int(run.op.info.cta_pair), "dtype": dtype_name(wl, run.path, run.math),
               "ms_per_step": ms, "tflops": wl.flops / (ms / 1e3) / 1e12, "blocks": len(ms_blocks),
               "steps_per_block": steps, "kernels_per_step": run.kernels, "roofline": roof,
               "normalize_pass": normalize_pass_roofline(wl, kern, peaks), "clocks": clocks}
        fin = rowmin_finisher(wl, kern, peaks) if wl.post == synth.POST_ROWMIN_BIAS else None
        if fin:
            out["finisher"] = fin
        return out
    finally:
        if sampler:
            sampler.stop()
        run.close()


def our_arm(args, wl):
    import torch
    import gemm_groupnorm_accelerator_gb300 as c1n

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    c1n.load()
    peaks = load_peaks()

    def barrier():
        if pg is not None:
            pg.barrier()

    run = ConvRun(c1n, wl, args, dev, rank)
    run.prepare(args.warmup, eager=args.eager)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    # Timed region: R back-to-back blocks of exactly --steps steps inside a window of at least
    # --min-seconds, so the clock sampler sees the GPU under load; the median block is reported.
    ms_blocks = run.timed_blocks(args.steps, args.min_seconds, barrier, pg)
    ms = statistics.median(ms_blocks)
    value, ms = aggregate([ms], wl.flops, world)
    kern = run.kernel_marks(args.warmup + args.steps)
    b2b = run.back_to_back_ms()
    roof = conv_roofline(wl, run, peaks, kern, b2b)
    if run.kernels_packed < run.kernels:  # the weight pack is a kernel of its own
        roof["pack_ms_graph_per_call"] = time_replays(lambda i: run.op.pack_weights(run.w), run.n_sets, dev,
                                                      args.steps, eager=not run.graphs)
    norm_pass = normalize_pass_roofline(wl, kern, peaks)

    e2e = measure_e2e(args, wl, run.op, run.inp, dev, run.tdt, run.bf, run.w, run.b, run.ga, run.be, run.b2, run.am)
    if pg is not None:
        t = torch.tensor([e2e["ms_per_step"]], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        e2e["ms_per_step"] = float(t[0])
        e2e["value"] = wl.flops * world / (e2e["ms_per_step"] / 1e3) / 1e12
    config = config_of(wl, {"path": run.path, "cta_pair": int(run.op.info.cta_pair),
                            "parallelism": f"dp{world}" if world > 1 else "single",
                            "l2": f"inputs rotate over {run.n_sets} x/y buffer sets "
                                  f"({run.n_sets * run.per_set / 2**20:.0f} MiB > 129 MiB L2)"
                            if run.n_sets > 1 else "working set larger than L2",
                            "step": "one operator call through the C ABI: weight pack + fused kernel",
                            "launch": run.launch_mode,
                            "timed_region": f"{len(ms_blocks)} blocks of {args.steps} steps (median block reported; "
                                            f"every block bracketed by barrier + synchronize)"})
    launches = args.steps * run.kernels
    run.close()

    # The other workloads and the normalize-pass measurements, in the same process and under the
    # same clock record (one GPU per process: rank 0 of a single-GPU run only).
    workloads, norm_runs = {}, {}
    default_run = args.workload == synth.CONV_GN.name and world == 1 and not args.no_extra
    if default_run:
        for name in EXTRA_WORKLOADS:
            w2 = workload_by_name(name)
            workloads[name] = measure_workload(c1n, w2, args, dev, rank, peaks, args.steps, args.extra_seconds,
                                               barrier)
        for name in NORMALIZE_PASS_WORKLOADS:
            w2 = workload_by_name(name)
            r = measure_workload(c1n, w2, args, dev, rank, peaks, args.steps, args.extra_seconds, barrier,
                                 path=c1n.PATH_TC_TWO_PASS)
            norm_runs[name] = {"workload": w2.name, "plan": r["plan"], "ms_per_step": r["ms_per_step"],
                               "passes": r["normalize_pass"], "conv_roofline": r["roofline"]}
    clocks = sampler.stop() if sampler else None
    if norm_pass is None and norm_runs:
        norm_pass = {"forced two-pass plans (the normalize pass on the largest outputs)": norm_runs}

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = time_oracle(wl, seconds=args.cpu_seconds, single_seconds=2.0)
        line = {"metric": args.metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": dtype_name(wl, run.path, args.math), "data": "synthetic",
                "config": config, "roofline": roof, "normalize_pass": norm_pass, "workloads": workloads or None,
                "cpu_baseline": cpu,
                "e2e": {k: e2e[k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "pipeline")},
                "gpu_launches": launches, "clocks": clocks}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def capture_graphs(fn, n, dev):
    """One CUDA graph per call fn(j), j < n, captured on a side stream; None if capture fails (the
    bench then times the eager loop and says so)."""
    import torch
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for j in range(n):
                fn(j)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        graphs = []
        for j in range(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(j)
            graphs.append(g)
        torch.cuda.synchronize()
        return graphs
    except Exception as e:  # pragma: no cover - depends on the driver
        print(f"bench: CUDA graph capture failed ({e}); timing the eager loop", file=sys.stderr)
        torch.cuda.synchronize()
        return None


def time_replays(fn, n_sets, dev, steps, eager=False):
    """Mean device ms of fn(i) over `steps` calls, replayed from per-set graphs unless eager."""
    import torch
    graphs = None if eager else capture_graphs(fn, n_sets, dev)
    run = (lambda i: graphs[i % n_sets].replay()) if graphs else fn
    for i in range(3):
        run(i)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for i in range(steps):
        run(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def kernel_times(op, step, i0, dev, n=5, graphs=True):
    """Mean device time per kernel name over n profiled steps (the library's event marks, recorded
    inside a replayed graph when graphs=True, so host launch gaps do not count)."""
    import torch
    acc = {}
    op.set_profiling(True)
    try:
        step(i0)  # an eager profiled run creates the library's events before any capture
        torch.cuda.synchronize()
        g = capture_graphs(lambda j: step(i0), 1, dev) if graphs else None
        for i in range(n):
            if g:
                g[0].replay()
            else:
                step(i0 + i)
            try:
                times = op.kernel_times()
            except Exception as e:  # pragma: no cover - event timing inside graphs unsupported
                print(f"bench: kernel times from the graph failed ({e}); using eager steps", file=sys.stderr)
                g = None
                step(i0 + i)
                times = op.kernel_times()
            for name, ms in times:
                acc.setdefault(name, []).append(ms)
    finally:
        op.set_profiling(False)
    torch.cuda.synchronize()
    return {k: statistics.mean(v) for k, v in acc.items()}


def normalize_pass_roofline(wl, kern, peaks):
    """GB/s of the memory-bound passes of a two-pass plan: statistics (read the fp32 raw tile) and
    normalize (read raw + write y), against the measured HBM copy bandwidth; None when the plan
    fuses normalization into the conv kernel. When the conv epilogue writes partial statistics, the
    statistics pass is a small merge of those partials (its time only)."""
    y_elems = wl.N * wl.C_out * wl.T_out
    out = {}
    for name, nbytes in (("gn_stats", 4 * y_elems), ("ln_stats", 4 * y_elems),
                         ("normalize", (4 + wl.elem_bytes) * y_elems)):
        if name in kern and kern[name] > 0:
            gbs = nbytes / (kern[name] / 1e3) / 1e9
            out[name] = {"ms": kern[name], "bytes": nbytes, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"],
                         "timing": "event pair around the kernel in a replayed graph (an upper bound on its time)"}
    for name in ("gn_merge", "ln_merge"):
        if name in kern and kern[name] > 0:
            out[name] = {"ms": kern[name]}
    return out or None


def measure_e2e(args, wl, op, inp, dev, tdt, bf, w_dev, b_dev, ga_dev, be_dev, b2_dev, am):
    """The operator end to end through the C ABI, fed from and read back to pinned host memory: every
    step copies its inputs (x and the parameters) host -> device, runs the operator (weight pack
    included) and copies y device -> host, all inside the timed region. Steps are pipelined over
    three streams and two buffer sets, as a serving loop would run them: while step i computes,
    step i+1's inputs upload and step i-1's output downloads. The K steps of a block are captured
    once as one CUDA graph (the copies, the operator's kernels and the cross-stream dependencies),
    so the host does not pace the loop; eager launches when capture is refused."""
    import torch
    host = {}
    for k in ("x", "w"):
        t = torch.from_numpy(inp[k])
        host[k] = (t.to(tdt) if bf else t).pin_memory()
    for k in ("b", "gamma", "beta", "bias2"):
        host[k] = None if inp[k] is None else torch.from_numpy(inp[k]).pin_memory()
    nbuf = 2
    dsets = [{k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in host.items()}
             for _ in range(nbuf)]
    ys = [torch.empty((wl.N, wl.C_out, op.T_out), dtype=op.out_dtype(), device=dev) for _ in range(nbuf)]
    y_hosts = [torch.empty(ys[0].shape, dtype=ys[0].dtype).pin_memory() for _ in range(nbuf)]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = y_hosts[0].numel() * y_hosts[0].element_size()
    s_in, s_op, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_op = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf

    def step(i):
        j = i % nbuf
        d = dsets[j]
        if used[j]:
            s_in.wait_event(ev_op[j])    # the operator of step i - nbuf has read set j
            s_op.wait_event(ev_out[j])   # ... and step i - nbuf's y has been read back
        with torch.cuda.stream(s_in):
            for k, v in host.items():
                if v is not None:
                    d[k].copy_(v, non_blocking=True)
            ev_in[j].record(s_in)
        s_op.wait_event(ev_in[j])
        with torch.cuda.stream(s_op):
            op(d["x"], d["w"], d["b"], d["gamma"], d["beta"], bias2=d["bias2"], out=ys[j], argmin=am)
            ev_op[j].record(s_op)
        s_out.wait_event(ev_op[j])
        with torch.cuda.stream(s_out):
            y_hosts[j].copy_(ys[j], non_blocking=True)
            ev_out[j].record(s_out)
        used[j] = True

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    graph = None
    if not args.eager:
        try:
            cap = torch.cuda.Stream(dev)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                fork = torch.cuda.Event()
                fork.record(cap)
                for s_ in (s_in, s_op, s_out):
                    s_.wait_event(fork)
                used[:] = [False] * nbuf  # no step of the block waits on work outside it
                for i in range(args.steps):
                    step(i)
                for s_ in (s_in, s_op, s_out):
                    join = torch.cuda.Event()
                    join.record(s_)
                    cap.wait_event(join)
            torch.cuda.synchronize()
            for _ in range(2):
                graph.replay()
            torch.cuda.synchronize()
        except Exception as e:  # pragma: no cover - depends on the driver
            print(f"bench: e2e graph capture failed ({e}); timing the eager loop", file=sys.stderr)
            torch.cuda.synchronize()
            graph = None
            used[:] = [False] * nbuf
    main = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph is not None:
        reps = 5
        e0.record(main)
        for _ in range(reps):
            graph.replay()
        e1.record(main)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * args.steps)
        pipe = (f"one CUDA graph per block of {args.steps} steps (H2D of the step's inputs from pinned memory, "
                f"the operator through the C ABI, D2H of y), 3 streams (H2D / operator / D2H), 2 buffer sets, "
                f"{reps} blocks")
    else:
        e0.record(s_in)
        for i in range(args.steps):
            step(i)
        s_out.wait_event(ev_out[(args.steps - 1) % nbuf])
        e1.record(s_out)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        pipe = "eager launches, 3 streams (H2D / operator / D2H), 2 buffer sets"
    return {"value": wl.flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "pipeline": pipe}


def shard_inputs(wl, rank, seed=0):
    """Inputs of rank `rank`: batch rows [rank*N, (rank+1)*N) of the global batch."""
    return synth.make_inputs(wl, seed=seed, n_rows=wl.N, row_offset=rank * wl.N)


def aggregate(ms_per_rank, flops_per_rank, world):
    """Whole-job throughput: all ranks' work divided by the slowest rank's time (TFLOP/s)."""
    slowest = max(ms_per_rank)
    return flops_per_rank * world / (slowest / 1e3) / 1e12, slowest


def read_traffic(workload, path):
    """DRAM bytes per launch of the main kernel from a committed ncu summary, if it was taken on the
    current sources of that kernel (its .cu file and the shared headers); None otherwise."""
    try:
        from gemm_groupnorm_accelerator_gb300 import _build_lib
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        rec = d.get(f"{workload}:{path}", d.get(workload))  # a workload with several plans: one key each
        if rec and rec.get("path") == path and \
                rec.get("source_fingerprint") == _build_lib.kernel_fingerprint(rec.get("source_file", "")):
            return rec["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# ----------------------------------------------------------------- [p4]'s LayerNorm(W) + AvgPool3d + GELU

def lnpool_config(wl, extra):
    cfg = {"workload": wl.name, "z": [wl.N, wl.C, wl.D, wl.H, wl.W], "out": list(wl.out_shape), "eps": wl.eps,
           "sum_weight": wl.sum_weight, "affine": wl.has_affine}
    cfg.update(extra)
    return cfg


def lnpool_oracle_sample(wl, seconds):
    """Time the oracle on a bounded number of (n, c) slices; GB/s of the operator's bytes."""
    import oracle
    per_slice = wl.algorithmic_bytes / (wl.N * wl.C)
    n = 8
    inp = synth.make_lnpool_inputs(wl, n_slices=n)
    threads = oracle.default_threads()
    run = lambda: oracle.ln_avgpool3d_gelu(inp["z"], wl.eps, wl.sum_weight, inp["gamma"], inp["beta"],
                                           nthreads=threads)
    run()
    runs, t0 = 0, time.perf_counter()
    while True:
        run()
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds or runs >= 200:
            break
    return {"value": per_slice * n * runs / el / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{runs} run(s) on {n} of {wl.N * wl.C} (n, c) slices, {el:.1f} s wall"}


def lnpool_arm(args, wl):
    """The memory-bound pass on its own: GB/s of z read + output written (+ gamma / beta)."""
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            cpu = lnpool_oracle_sample(wl, seconds=max(1.0, args.cpu_seconds))
            line = {"impl": "reference", "metric": "LayerNorm(W)+AvgPool3d+GELU GB/s", "value": cpu["value"],
                    "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "f64", "data": "synthetic", "config": lnpool_config(wl, {}), "cpu_baseline": cpu,
                    "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        return
    import torch
    import gemm_groupnorm_accelerator_gb300 as c1n
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    c1n.load()
    peaks = load_peaks()
    inp = synth.make_lnpool_inputs(wl, n_slices=wl.N * wl.C, slice_offset=rank * wl.N * wl.C)
    z = torch.from_numpy(inp["z"]).to(dev).view(wl.N, wl.C, wl.D, wl.H, wl.W)
    ga = torch.from_numpy(inp["gamma"]).to(dev) if inp["gamma"] is not None else None
    be = torch.from_numpy(inp["beta"]).to(dev) if inp["beta"] is not None else None
    out = torch.empty(wl.out_shape, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda i: c1n.ln_avgpool3d_gelu(z, wl.sum_weight, ga, be, eps=wl.eps, out=out)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    graphs = capture_graphs(step, 1, dev) if not args.eager else None
    run_step = (lambda i: graphs[0].replay()) if graphs else step
    for i in range(3):
        run_step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        run_step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    clocks = sampler.stop() if sampler else None
    ms = t0.elapsed_time(t1) / args.steps
    if pg is not None:
        t = torch.tensor([ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t[0])
    nbytes = wl.algorithmic_bytes
    value = nbytes * world / (ms / 1e3) / 1e9
    ach = nbytes / (ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
            "traffic": None, "peak_source": peaks["source"], "kernel": "ln_avgpool3d_gelu_kernel",
            "kernel_ms": ms, "algorithmic_bytes": nbytes}
    # end to end: z from pinned host memory in and the pooled output back, every step
    zh = torch.from_numpy(inp["z"]).pin_memory()
    oh = torch.empty(wl.out_shape, dtype=torch.float32).pin_memory()
    e_steps = max(1, min(args.steps, 5))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e_steps):
        z.view(-1).copy_(zh.view(-1), non_blocking=True)
        step(i)
        oh.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1) / e_steps
    e2e = {"value": nbytes * world / (e_ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": zh.numel() * 4,
           "d2h_bytes_per_step": oh.numel() * 4}
    if rank == 0:
        cpu = None if (world > 1 or args.no_cpu_baseline) else lnpool_oracle_sample(wl, seconds=args.cpu_seconds)
        line = {"metric": "LayerNorm(W)+AvgPool3d+GELU GB/s", "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": lnpool_config(wl, {"parallelism": f"dp{world}" if world > 1 else "single",
                                             "l2": "working set larger than L2",
                                             "launch": "cuda graph replay" if graphs else "eager"}),
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps, "clocks": clocks}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


FP32_FMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # 152 SMs x 128 fp32 lanes x FMA at 2.07 GHz


def p4_oracle_sample(wl, lp, seconds):
    """The oracle's model (ConvTranspose3d, then + scalar, LayerNorm, AvgPool3d, GELU) on one batch
    entry at a time for about `seconds` of wall time, on the host's cores; TFLOP/s of the transposed
    convolution's useful multiply-adds."""
    import oracle
    inp = synth.make_convt3d_inputs(wl, n_rows=1)
    gb = synth.make_lnpool_inputs(lp.replace(N=1, C=1, D=2, H=2))
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    runs = 0
    while True:
        y = oracle.conv_transpose3d(inp["x"], inp["w"], inp["b"], stride=wl.stride, pad=wl.pad, out_pad=wl.out_pad,
                                    nthreads=threads)
        oracle.ln_avgpool3d_gelu(y[0].astype(np.float32), lp.eps, lp.sum_weight, gb["gamma"], gb["beta"],
                                 nthreads=threads)
        runs += 1
        el = time.perf_counter() - t0
        if el >= max(1.0, seconds) or runs >= 20:
            break
    return {"value": wl.flops / wl.N * runs / el / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{runs} run(s) of the model on 1 of {wl.N} batch entries, {el:.1f} s wall",
            "ms_per_sample": el / runs * 1e3}


def p4_arm(args, wl):
    """[p4]'s model after its weights on one GPU: ConvTranspose3d, + scalar, LayerNorm(W), AvgPool3d,
    GELU -- by default in one tensor-core kernel; --p4-two-kernel runs the ConvTranspose3d operator
    (tensor cores unless --math 1 asks for the CUDA cores) and then the pass. TFLOP/s of the
    transposed convolution's useful multiply-adds."""
    world, rank, local = dist_env()
    lp = synth.LN_AVGPOOL3D_GELU
    if args.impl == "reference":
        if rank == 0:
            cpu = p4_oracle_sample(wl, lp, args.cpu_seconds)
            value = cpu["value"]
            print(json.dumps({"impl": "reference", "metric": "p4 ConvTranspose3d+LayerNorm+AvgPool3d+GELU TFLOP/s",
                              "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                              "warmup": args.warmup, "ms_per_step": cpu["ms_per_sample"], "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                              "config": {"workload": wl.name}, "cpu_baseline": cpu,
                              "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
        return
    import torch
    import gemm_groupnorm_accelerator_gb300 as c1n
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    c1n.load()
    peaks = load_peaks()
    inp = synth.make_convt3d_inputs(wl, n_rows=wl.N, row_offset=rank * wl.N)
    gb = synth.make_lnpool_inputs(lp.replace(N=1, C=1, D=2, H=2))
    x, w, b = (torch.from_numpy(inp[k]).to(dev) for k in ("x", "w", "b"))
    ga, be = torch.from_numpy(gb["gamma"]).to(dev), torch.from_numpy(gb["beta"]).to(dev)
    Do, Ho, Wo = wl.out_dhw
    out = torch.empty((wl.N, wl.C_out, Do // 2, Ho // 2, Wo // 2), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    math = args.math if args.math in (1, 2) else 0
    cp = c1n.ConvT3dParams(wl.N, wl.C_in, wl.C_out, wl.D, wl.H, wl.W, wl.k, wl.stride, wl.pad, wl.out_pad, math)
    # Default: the whole model in one tensor-core kernel (the convolution's output stays on chip);
    # --p4-two-kernel or --math 1: the ConvTranspose3d operator, then the LayerNorm/pool/GELU pass.
    fused = not args.p4_two_kernel and math != 1
    if fused:
        fws = torch.empty(c1n.conv_transpose3d_ln_avgpool3d_gelu_workspace_size(cp), dtype=torch.uint8, device=dev)
        model = lambda i: c1n.conv_transpose3d_ln_avgpool3d_gelu(x, w, b, lp.sum_weight, ga, be, eps=lp.eps, out=out,
                                                                 workspace=fws)
        step = model
        tensor_plan = True
        n_kernels = 3
    else:
        y = torch.empty((wl.N, wl.C_out, Do, Ho, Wo), dtype=torch.float32, device=dev)
        ws_bytes = c1n.conv_transpose3d_workspace_size(cp)
        tensor_plan = ws_bytes > 0  # only the tensor-core plan takes a workspace
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        convt = lambda i: c1n.conv_transpose3d(x, w, b, stride=wl.stride, pad=wl.pad, out_pad=wl.out_pad, out=y,
                                               math=math, workspace=ws)
        lnp = lambda i: c1n.ln_avgpool3d_gelu(y, lp.sum_weight, ga, be, eps=lp.eps, out=out)
        n_kernels = 4 if tensor_plan else 2

        def step(i):
            convt(i)
            lnp(i)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    clocks = sampler.stop() if sampler else None
    ms = t0.elapsed_time(t1) / args.steps
    if pg is not None:
        t = torch.tensor([ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t[0])
    value = wl.flops * world / (ms / 1e3) / 1e12
    # timed after the seconds-long timed region: the sustained tensor peak (burst beside it)
    tf32_peak = peaks["bf16_tflops_sustained"] * TF32_PER_BF16
    tf32_burst = peaks["bf16_tflops"] * TF32_PER_BF16
    if fused:
        # The contraction bounds the one-pass model: x (67 MB) in and the pooled output (134 MB) out
        # take ~30 us of HBM, the multiply-adds ~60 us of TF32 tensor time. The time is the whole
        # operator (channels-last copy of x, weight pack, convt3d_lnpool_fused_kernel).
        model_ms = time_replays(model, 1, dev, args.steps, eager=True)
        ach = wl.flops / (model_ms / 1e3) / 1e12
        fbytes = 4 * (inp["x"].size + inp["w"].size + inp["b"].size + 2 * wl.W * 2 + out.numel())
        # Issued MMA work of the one-pass kernel: a tile is 4 x 32 input voxels (MMA M = 128) of one
        # (n, d) plane; per tile and channel half the MMAs have N = the 864 resident weight rows (the
        # taps that meet an input, 27 per output parity class x C_out/2 = 32 channels of the half)
        # and K = C_in = 32; two channel halves per tile.
        assert (wl.C_in, wl.C_out, wl.k, wl.W) == (32, 64, 3, 32), "tile constants below assume the page's shape"
        tile_m, rows_per_half, halves = 4 * wl.W, 27 * (wl.C_out // 2), 2
        tiles = wl.N * wl.D * ((wl.H + 3) // 4)
        issued = 2.0 * tile_m * rows_per_half * wl.C_in * halves * tiles
        roof = {"bound": "tensor", "achieved": ach, "peak": tf32_peak, "unit": "TFLOP/s", "frac": ach / tf32_peak,
                "frac_of_burst_peak": ach / tf32_burst, "traffic": read_traffic(wl.name, "convt3d_lnpool_fused"),
                "peak_source": peaks.get("source", "MEASURED_PEAKS.json") + " (bf16 x 1.1/2.25 for tf32)",
                "peak_kind": "sustained (timed after the seconds-long timed region)",
                "kernel": "convt3d_lnpool_fused_kernel (timed with its channels-last copy and weight pack)",
                "kernel_ms": model_ms, "algorithmic_flops": wl.flops, "issued_mma_flops": issued,
                "algorithmic_bytes": fbytes, "hbm_frac": fbytes / (model_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                "kernels_ms": {"conv_transpose3d_ln_avgpool3d_gelu": model_ms}}
    else:
        convt_ms = time_replays(convt, 1, dev, args.steps, eager=True)
        lnp_ms = time_replays(lnp, 1, dev, args.steps, eager=True)
        ach = wl.flops / (convt_ms / 1e3) / 1e12
        common = {"kernels_ms": {"conv_transpose3d": convt_ms, "ln_avgpool3d_gelu": lnp_ms},
                  "ln_avgpool3d_gelu_hbm_frac": lp.algorithmic_bytes / (lnp_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
        if tensor_plan:
            # Writing y (8x the input voxels, 64 channels) outweighs the contraction on this shape:
            # the operator is bound by HBM. Bytes = x + w + b read once, y written once; the time is
            # the whole operator (channels-last copy of x, weight pack, convt3d_tc_kernel).
            gbs = wl.algorithmic_bytes / (convt_ms / 1e3) / 1e9
            roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"], "traffic": read_traffic(wl.name, "convt3d_tc"),
                    "peak_source": peaks.get("source", "MEASURED_PEAKS.json"),
                    "kernel": "convt3d_tc_kernel (timed with its channels-last copy and weight pack)",
                    "kernel_ms": convt_ms, "algorithmic_bytes": wl.algorithmic_bytes, "useful_tflops": ach,
                    "useful_tflops_frac_of_tf32": ach / tf32_peak, **common}
        else:
            roof = {"bound": "alu", "achieved": ach, "peak": FP32_FMA_PEAK_TFLOPS, "unit": "TFLOP/s",
                    "frac": ach / FP32_FMA_PEAK_TFLOPS, "traffic": None,
                    "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz",
                    "kernel": "conv_transpose3d_k3s2_kernel", "kernel_ms": convt_ms, "algorithmic_flops": wl.flops,
                    **common}
    xh = torch.from_numpy(inp["x"]).pin_memory()
    oh = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    e_steps = max(1, min(args.steps, 5))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e_steps):
        x.copy_(xh, non_blocking=True)
        step(i)
        oh.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1) / e_steps
    e2e = {"value": wl.flops * world / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": xh.numel() * 4,
           "d2h_bytes_per_step": oh.numel() * 4}
    if rank == 0:
        # the oracle on the host cores, after the GPU work (its threads would compete with the launches)
        cpu = None if (world > 1 or args.no_cpu_baseline) else p4_oracle_sample(wl, lp, args.cpu_seconds)
        line = {"metric": "p4 ConvTranspose3d+LayerNorm+AvgPool3d+GELU TFLOP/s", "value": value, "unit": "TFLOP/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "tf32" if tensor_plan else "f32", "data": "synthetic",
                "config": {"workload": wl.name, "x": [wl.N, wl.C_in, wl.D, wl.H, wl.W], "C_out": wl.C_out,
                           "k": wl.k, "stride": wl.stride, "pad": wl.pad, "out_pad": wl.out_pad,
                           "then": lp.name, "parallelism": f"dp{world}" if world > 1 else "single",
                           "math": "tensor (tf32)" if tensor_plan else "cuda cores (fp32 fma)",
                           "plan": "one-pass model kernel" if fused else "ConvTranspose3d, then the pass",
                           "l2": "working set larger than L2",
                           "launch": f"eager, {n_kernels} kernels per step"},
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": n_kernels * args.steps, "clocks": clocks}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synth.CONV_GN.name)
    ap.add_argument("--math", type=int, default=0, help="0 auto, 1 SIMT, 2 tensor, 3 tensor 3xTF32 (fp32-accurate)")
    ap.add_argument("--path", type=int, default=-1, help="force an execution path (c1n_path)")
    ap.add_argument("--mainloop", type=int, default=0, help="0 auto, 1 one CTA per tile, 2 CTA pairs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--p4-two-kernel", action="store_true",
                    help="p4 workload: ConvTranspose3d then the LayerNorm/pool/GELU pass instead of the one-pass kernel")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--oracle-rows", type=int, default=2, help="batch entries per reference-arm step")
    ap.add_argument("--metric", default="fused conv1d+GroupNorm TFLOP/s")
    ap.add_argument("--eager", action="store_true", help="time the eager launch loop instead of CUDA graph replays")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="the timed blocks of --steps steps repeat until they cover this long (clock sampling window)")
    ap.add_argument("--extra-seconds", type=float, default=0.3,
                    help="the same for each of the other workloads of the default run")
    ap.add_argument("--no-extra", action="store_true",
                    help="default run: skip the other workloads and the forced two-pass normalize measurements")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    wl = workload_by_name(args.workload)
    if isinstance(wl, synth.LnPoolWorkload):
        lnpool_arm(args, wl)
    elif isinstance(wl, synth.ConvT3dWorkload):
        p4_arm(args, wl)
    elif args.impl == "reference":
        reference_arm(args, wl)
    else:
        our_arm(args, wl)


if __name__ == "__main__":
    main()
