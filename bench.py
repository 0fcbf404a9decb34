"""Benchmark of the single-GPU MoE layer forward (one JSON line on rank 0).

A step is one whole forward -- routing, 1x128 FP8 quantisation + dispatch,
FC1 with the fused SwiGLU/re-quantisation epilogue, FC2, combine -- over one
batch of the workload, replayed from a CUDA graph.  L2 is flushed (a 256 MiB
write, outside the timed span) before every timed step; each step is timed
with CUDA events on the launching stream and the K step times are summed.
The timed capture has no events between its kernels; per-kernel times come
from a second capture with an event before every kernel, replayed for the
same number of steps right after.

The main line is the DeepSeek-V3-shaped prefill layer (T=8192, H=7168,
I=2048, E=256, top-8) unless --config says otherwise.  Beside it, under
"per_workload", the same run times the decode sweep (T = 8, 64, 256, 1024 on
the same weights), the skewed layer and the DeepSeek-V2-Lite-shaped layer the
same way (--no-records skips them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, float64) as it stands on the
host cores, each step a bounded sample of the same workload (every routed row
of a few random experts).
Under torchrun (N > 1) every rank runs its own replica of the workload (no
data-path collective: the layer does not shard on one-GPU machines); the time is
the max over ranks and the value counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer routed TFLOPS & tokens/s on 1 GB300; % of FP8-peak/HBM roofline"
L2_WARM_STEPS = 200  # back-to-back steps of the L2-warm figure
L2_BYTES = 129 << 20  # GB300 L2
REF_STEP_S = 4.0      # oracle seconds per reference-arm step
CPU_BASELINE_S = 15.0  # oracle seconds of the cpu_baseline leg
# Idle seconds between a workload's set-up (weight generation, binding) and its
# warm-up: the timed steps then start from the same power state whatever the
# set-up drew (within ~0.3 s of full load the part reaches its power limit and
# lowers the SM clock; the timed region is compared with the burst peak).
SETTLE_S = 1.5
# the per-workload record printed beside the main line (same run, same method)
RECORD_CONFIGS = ("v3prefill", "v3decode8", "v3decode64", "v3decode256", "v3decode1024", "skew",
                  "v2lite")

KERNELS = ["status_reset", "route_count", "route_scan", "route_scatter", "quant_dispatch", "fc1",
           "swiglu_quant", "fc2", "combine"]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=0,
                   help="timed steps (0: as many as fill about a second, at least 20, so the "
                        "clock samples fall inside the timed region)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--config", default="v3prefill")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--unfused", action="store_true", help="time the unfused reference path")
    p.add_argument("--gemm", default="auto", choices=["auto", "single", "pair"])
    p.add_argument("--format", default="deepseek", choices=["deepseek", "mxfp8", "per_tensor"],
                   help="scales: DeepSeek 1x128 / 128x128 blocks, MXFP8 1x32 along K, or per "
                        "tensor (one per expert weight matrix, static activation scales)")
    p.add_argument("--experts", type=int, default=0,
                   help="profiling only: the workload with this many experts (smaller weights)")
    p.add_argument("--tokens", type=int, default=0,
                   help="profiling only: the workload with this many tokens")
    p.add_argument("--gemms", default="auto", choices=["auto", "one_launch", "split"],
                   help="FC1 -> FC2 as one persistent launch, two launches, or chosen per forward")
    p.add_argument("--side-mlp", type=int, default=0,
                   help="measure the layer beside a shared-expert MLP of this intermediate size on "
                        "another stream, per SM budget (prints that sweep instead of the bench line)")
    p.add_argument("--sm-budget", type=int, default=0,
                   help="cap the SMs the layer occupies (moe_set_sm_budget; 0: every SM)")
    p.add_argument("--combine-in-fc2", action="store_true",
                   help="fold the combine into FC2 (single-CTA forwards; no combine kernel)")
    p.add_argument("--no-swap", action="store_true",
                   help="keep the M128 x N256 GEMMs for small forwards (no token-as-N kernels)")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-records", action="store_true",
                   help="skip the per-workload record beside the main line")
    p.add_argument("--records", default=",".join(RECORD_CONFIGS),
                   help="comma-separated workloads of the per-workload record (the main one is "
                        "skipped there)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def reduce_max(value: float, device) -> float:
    """max over the ranks of the initialised process group (value unchanged
    without one).  Replicas only: this is timing, not a data-path collective."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, units_per_step: float, steps: int, max_total_ms: float) -> float:
    """whole-job throughput: the units all ranks processed over the slowest rank's time"""
    return world * units_per_step * steps / (max_total_ms * 1e-3)


def strip_c_comments(src: str) -> str:
    """C/C++ source without comments and with whitespace collapsed, so that
    editing a comment does not count as changing the code."""
    import re
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":                       # string / char literal, kept whole
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def gemm_source_hash() -> str:
    """sha256 over the code (comments stripped) the grouped-GEMM kernel is
    compiled from."""
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh", "internal.h"):
        with open(os.path.join(ROOT, "serving_route_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_c_comments(fh.read()).encode())
    return h.hexdigest()


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch from the committed ncu record, or
    None when there is none for this workload or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    if rec.get("source_sha256") != gemm_source_hash():
        return None
    for e in rec.get("entries", []):
        if e["workload"] == workload and e["kernel"] == kernel:
            return e["dram_bytes_per_launch"]
    return None


def algorithmic_bytes(wl, counts):
    """compulsory HBM bytes of the layer: FP8 weights + scales of every expert
    with at least one route, x read (bf16), out write (bf16), routes."""
    touched = int((counts > 0).sum())
    w = touched * (2 * wl.I * wl.H + wl.H * wl.I + (2 * wl.I // 128) * (wl.H // 128) * 4
                   + (wl.H // 128) * (wl.I // 128) * 4)
    io = wl.T * wl.H * 2 * 2 + wl.T * wl.K * 8
    return w + io, touched


class ClockSampler:
    """nvidia-smi SM and memory clocks, power and throttle reasons, sampled
    every 100 ms."""

    def __init__(self, index: int):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, smax, mem, power, reasons = [], [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
            for dst, v in ((power, f[3]), (mem, f[9] if len(f) > 9 else "")):
                try:
                    dst.append(float(v))
                except ValueError:
                    pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "mem_mhz": statistics.median(mem) if mem else None,
                "power_w": statistics.median(power) if power else None,
                "reasons": sorted(reasons)}


def cpu_threads() -> int:
    """host threads the oracle uses: the cores this process may run on, or
    OMP_NUM_THREADS when that is set lower (the oracle's parallel loops are
    OpenMP)"""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    omp = os.environ.get("OMP_NUM_THREADS", "")
    return min(n, int(omp)) if omp.isdigit() and int(omp) > 0 else n


class OracleSampler:
    """Times the oracle on bounded samples of a workload, drawn by expert: a
    sample is every routed row of a few random non-empty experts (their expert
    FFN), with the tokens that route there (their quantisation and the combine
    of those routes).  This keeps the rows per expert of the real workload,
    which is what the oracle's cost and parallelism depend on (it decodes each
    expert's weights once per call and runs that expert's rows in parallel),
    while bounding a sample's work.  Weights are generated and quantised by the
    oracle's own quantiser for the sampled experts only, outside the timed
    span, and kept for later samples."""

    def __init__(self, wl, x_bits, idx, w, keep_experts: int = 64):
        self.wl, self.x, self.idx, self.w = wl, x_bits, idx, w
        flat = idx.ravel()
        self.counts = np.bincount(flat[flat >= 0], minlength=wl.E)
        self.nonempty = np.nonzero(self.counts)[0]
        self.cache = {}
        self.keep = keep_experts

    def weights(self, experts):
        import oracle
        from gen import problem
        missing = [e for e in experts if e not in self.cache]
        for c in range(0, len(missing), 8):
            part = missing[c:c + 8]
            w1q, w1s = oracle.quant_weights(problem.w1_f32(self.wl, part))
            w2q, w2s = oracle.quant_weights(problem.w2_f32(self.wl, part))
            for i, e in enumerate(part):
                self.cache[e] = (w1q[i], w1s[i], w2q[i], w2s[i])
        out = tuple(np.stack([self.cache[e][j] for e in experts]) for j in range(4))
        while len(self.cache) > self.keep:        # bounded host memory
            self.cache.pop(next(iter(self.cache)))
        return out

    def sample(self, n_experts: int, rng):
        """-> (seconds, routed FLOPs, routed rows, experts) of one timed oracle call."""
        import oracle
        n = int(max(1, min(n_experts, len(self.nonempty))))
        S = np.sort(rng.choice(self.nonempty, size=n, replace=False))
        inS = np.isin(self.idx, S)
        tokens = np.nonzero(inS.any(axis=1))[0]
        remap = np.full(self.wl.E, -1, np.int32)
        remap[S] = np.arange(n, dtype=np.int32)
        sub = self.idx[tokens]
        mini = np.where(inS[tokens], remap[np.clip(sub, 0, self.wl.E - 1)], -1).astype(np.int32)
        W = self.weights([int(e) for e in S])
        x = np.ascontiguousarray(self.x[tokens])
        w = np.ascontiguousarray(self.w[tokens])
        t0 = time.perf_counter()
        r = oracle.forward(x, mini, w, *W)
        dt = time.perf_counter() - t0
        assert r["err"] == 0
        rows = int(self.counts[S].sum())
        return dt, 6 * rows * self.wl.H * self.wl.I, rows, n

    def per_expert_seconds(self, rng) -> float:
        """calibration: one untimed call on one expert"""
        dt, _, _, _ = self.sample(1, rng)
        return max(dt, 1e-3)


def oracle_bounded_run(wl, x_bits, idx, w, target_s: float, rng):
    """One bounded sample of about target_s seconds of oracle work: experts are
    added in doubling batches until the timed calls reach target_s or every
    non-empty expert has been sampled.  Returns the cpu_baseline fields."""
    smp = OracleSampler(wl, x_bits, idx, w)
    total_t = total_f = total_r = total_e = 0
    n = 1
    while total_t < target_s and total_e < len(smp.nonempty):
        n = min(n, len(smp.nonempty) - total_e)
        dt, fl, rows, ne = smp.sample(n, rng)
        total_t += dt
        total_f += fl
        total_r += rows
        total_e += ne
        n *= 2
    return {"value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(),
            "kind": "oracle", "seconds": total_t,
            "sample": f"every routed row of {total_e} random experts of {wl.name} ({total_r} rows; "
                      "their expert FFN, the quantisation of the tokens routed there and the "
                      "combine of those routes), in doubling batches up to about "
                      f"{target_s:.0f} s of oracle time; weights quantised untimed"}


def run_reference(args):
    """The reference arm: the oracle as it stands on the host cores, each step a
    bounded sample of the workload (every routed row of a few random experts,
    sized from an untimed one-expert calibration to about REF_STEP_S seconds)."""
    from gen import configs, problem
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if args.steps <= 0:
        args.steps = 3
    wl = configs.WORKLOADS[args.config]
    x = problem.x_bits(wl)
    idx, w = wl.make_routes()
    smp = OracleSampler(wl, x, idx, w)
    rng = np.random.default_rng(0)
    per_expert = smp.per_expert_seconds(rng)
    n_exp = int(max(1, min(len(smp.nonempty), round(REF_STEP_S / per_expert))))
    times, flops, rows = [], [], []
    for s in range(args.warmup + args.steps):
        dt, fl, r, _ = smp.sample(n_exp, rng)
        if s >= args.warmup:
            times.append(dt)
            flops.append(fl)
            rows.append(r)
    total = sum(times)
    value = sum(flops) / total / 1e12
    sample = (f"every routed row of {n_exp} random experts of {wl.name} per step (mean "
              f"{statistics.mean(rows):.0f} rows: their expert FFN, the quantisation of the tokens "
              "routed there and the combine of those routes); weights quantised untimed")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "experts_per_step": n_exp},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def side_stream_sweep(args, torch, layer, x, idx, wts, wl, dev, flush):
    """The layer on one stream and a shared-expert MLP on another, per SM budget
    of the layer (moe_set_sm_budget), against the two run one after the other.
    The MLP is the caller's other work, not part of the library: a dense BF16
    SwiGLU FFN of intermediate size args.side_mlp over the same tokens, as
    torch matmuls.  Direct launches, L2 flushed before every repetition,
    median of the repetitions."""
    n = args.side_mlp
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    wgu = (torch.randn(wl.H, 2 * n, device=dev, generator=gen) * wl.H ** -0.5).to(torch.bfloat16)
    wd = (torch.randn(n, wl.H, device=dev, generator=gen) * n ** -0.5).to(torch.bfloat16)
    main_s, side_s = torch.cuda.Stream(), torch.cuda.Stream()

    def mlp():
        gu = x @ wgu
        return (torch.nn.functional.silu(gu[:, :n]) * gu[:, n:]) @ wd

    def layer_fwd():
        layer.forward(x, idx, wts, stream=main_s)

    def serial():
        layer_fwd()
        with torch.cuda.stream(main_s):
            mlp()

    def concurrent():
        fork = torch.cuda.Event()
        fork.record(main_s)
        side_s.wait_event(fork)
        with torch.cuda.stream(side_s):
            mlp()
        join = torch.cuda.Event()
        join.record(side_s)
        layer_fwd()
        main_s.wait_event(join)

    def timed(fn, reps=max(args.steps, 20), warm=max(args.warmup, 3)):
        ts = []
        for i in range(warm + reps):
            flush.zero_()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(main_s)
            fn()
            b.record(main_s)
            torch.cuda.synchronize()
            if i >= warm:
                ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def mlp_alone():
        with torch.cuda.stream(main_s):
            mlp()

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    layer_ms, mlp_ms, serial_ms = timed(layer_fwd), timed(mlp_alone), timed(serial)
    points = []
    for budget in [0] + [sms - d for d in (4, 8, 16, 24, 32, 48)]:
        layer.set_sm_budget(budget)
        points.append({"sm_budget": budget or sms, "ms": timed(concurrent),
                       "layer_alone_ms": timed(layer_fwd)})
    layer.set_sm_budget(0)
    st, bits = layer.read_status(main_s)
    if st != 0:
        raise RuntimeError(f"forward reported device status {bits:#x}")
    best = min(points, key=lambda p: p["ms"])
    print(json.dumps({
        "metric": "layer + side-stream shared-expert MLP, ms per step (lower is better)",
        "unit": "ms", "higher_is_better": False, "n_gpus": 1, "data": "synthetic",
        "config": {"workload": wl.name, "side_mlp_inter": n, "side_mlp": "BF16 SwiGLU FFN, torch matmuls",
                   "launch": "direct launches", "l2": "flushed before every repetition",
                   "gemm": ("cta pairs" if layer.tactic()["gemm_pair"] else "single cta")},
        "layer_ms": layer_ms, "mlp_ms": mlp_ms, "serial_ms": serial_ms,
        "concurrent": points, "best": best,
        "best_vs_serial": best["ms"] / serial_ms,
        "all_sms_vs_serial": points[0]["ms"] / serial_ms}))


def gpu_weights(torch, g, layer_cls, wl, fmt, dev, stream):
    """Weights of a workload generated on the GPU by the shared seeded
    generator and quantised there (moe_quantize_weights), in expert chunks."""
    mx, pt = fmt == "mxfp8", fmt == "per_tensor"
    sp = stream.cuda_stream
    w1q = torch.empty((wl.E, 2 * wl.I, wl.H), dtype=torch.uint8, device=dev)
    w1s = torch.empty((wl.E,) if pt else ((wl.E, 2 * wl.I, wl.H // 32) if mx
                                          else (wl.E, 2 * wl.I // 128, wl.H // 128)),
                      dtype=torch.float32, device=dev)
    w2q = torch.empty((wl.E, wl.H, wl.I), dtype=torch.uint8, device=dev)
    w2s = torch.empty((wl.E,) if pt else ((wl.E, wl.H, wl.I // 32) if mx
                                          else (wl.E, wl.H // 128, wl.I // 128)),
                      dtype=torch.float32, device=dev)
    chunk = 16
    with torch.cuda.stream(stream):
        for e0 in range(0, wl.E, chunk):
            ne = min(chunk, wl.E - e0)
            f = torch.empty((ne, 2 * wl.I, wl.H), dtype=torch.float32, device=dev)
            g.dev_normal_f32(wl.seed, g.STREAM_W1, e0 * 2 * wl.I * wl.H, f.numel(),
                             g.weight_sigma(wl.H), f.data_ptr(), sp)
            q, s = layer_cls.quantize_weights(f, stream, fmt=fmt)
            w1q[e0:e0 + ne].copy_(q)
            w1s[e0:e0 + ne].copy_(s)
            f = torch.empty((ne, wl.H, wl.I), dtype=torch.float32, device=dev)
            g.dev_normal_f32(wl.seed, g.STREAM_W2, e0 * wl.H * wl.I, f.numel(),
                             g.weight_sigma(wl.I), f.data_ptr(), sp)
            q, s = layer_cls.quantize_weights(f, stream, fmt=fmt)
            w2q[e0:e0 + ne].copy_(q)
            w2s[e0:e0 + ne].copy_(s)
            del f, q, s
    stream.synchronize()
    return w1q, w1s, w2q, w2s


def bind(layer, weights, fmt, stream):
    """bind the weights; a per-tensor layer also gets the workloads' static
    activation scales"""
    from gen import configs
    layer.bind_weights(*weights, stream)
    if fmt == "per_tensor":
        layer.set_activation_scales(float(configs.PT_X_SCALE), float(configs.PT_H_SCALE), stream)


def fmt_name(fmt):
    return {"mxfp8": "MXFP8: E4M3, E8M0 scale per 32 along K",
            "per_tensor": "E4M3, per-tensor scales (one per expert weight matrix; static x and h "
                          "scales 6/448 and 24/448)"}.get(fmt, "E4M3, 1x128 activation / 128x128 "
                                                              "weight scales")


def device_inputs(torch, g, wl, dev, stream):
    """x on the GPU from the device generator; routes from the host recipe."""
    x = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
    g.dev_normal_bf16(wl.seed, g.STREAM_X, 0, wl.T * wl.H, x.data_ptr(), stream.cuda_stream)
    idx_np, w_np = wl.make_routes()
    idx = torch.from_numpy(idx_np).to(dev)
    wts = torch.from_numpy(w_np).to(dev)
    flat = idx_np.ravel()
    counts = np.bincount(flat[flat >= 0], minlength=wl.E)
    return x, idx, wts, idx_np, w_np, counts


class StepTimer:
    """Device timing of whole forwards, the same way for every workload: two CUDA
    graph captures of the forward -- the timed one has no events between its
    kernels (each kernel after the first launches as a programmatic dependent
    of the previous one); the profiled one records an event before every
    kernel, which gives the per-kernel times.  L2 is flushed (a 256 MiB write on
    the stream, outside the timed span) before every step; each step is
    bracketed by CUDA events on the launching stream."""

    def __init__(self, torch, layer, x, idx, wts, stream, flush, use_graph):
        self.torch, self.layer, self.stream, self.flush = torch, layer, stream, flush
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)]
        self.t0 = torch.cuda.Event(enable_timing=True)
        self.t1 = torch.cuda.Event(enable_timing=True)
        self.fwd = lambda: layer.forward(x, idx, wts, stream=stream)
        with torch.cuda.stream(stream):
            self.fwd()
        stream.synchronize()
        st, bits = layer.read_status(stream)
        if st != 0:
            raise RuntimeError(f"forward reported device status {bits:#x}")
        self.graph = self._capture() if use_graph else None
        layer.set_profile_events(self.ev)
        self.graph_prof = self._capture() if use_graph else None
        layer.set_profile_events([])

    def _capture(self):
        torch = self.torch
        try:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=self.stream):
                self.fwd()
            self.stream.synchronize()
            return gr
        except Exception as e:  # fall back to direct launches
            print(f"# graph capture failed ({e}); timing direct launches", file=sys.stderr)
            return None

    def _step(self, profiled):
        torch = self.torch
        gr = self.graph_prof if profiled else self.graph
        if profiled:
            self.layer.set_profile_events(self.ev)
        with torch.cuda.stream(self.stream):
            if gr is not None:
                gr.replay()
            else:
                self.fwd()
        if profiled:
            self.layer.set_profile_events([])

    def steps(self, n, profiled=False, keep=None):
        """n flushed, event-timed steps -> (total ms, per-kernel ms summed)"""
        torch, s = self.torch, self.stream
        tot = 0.0
        per_kernel = {k: 0.0 for k in KERNELS}
        for _ in range(n):
            with torch.cuda.stream(s):
                self.flush.zero_()
                self.t0.record(s)
            self._step(profiled)
            with torch.cuda.stream(s):
                self.t1.record(s)
            s.synchronize()
            dt = self.t0.elapsed_time(self.t1)
            tot += dt
            if keep is not None:
                keep.append(dt)
            if profiled:
                for i, k in enumerate(KERNELS):
                    per_kernel[k] += self.ev[i].elapsed_time(self.ev[i + 1])
        return tot, per_kernel

    def l2_warm(self, n):
        """ms per step of the same capture replayed back to back, nothing flushed"""
        torch, s = self.torch, self.stream
        with torch.cuda.stream(s):
            self.flush.zero_()
            for _ in range(3):
                self._step(False)
            self.t0.record(s)
            for _ in range(n):
                self._step(False)
            self.t1.record(s)
        s.synchronize()
        return self.t0.elapsed_time(self.t1) / n

    def check_status(self, what):
        st, bits = self.layer.read_status(self.stream)
        if st != 0:
            raise RuntimeError(f"{what} reported device status {bits:#x}")


def kernel_times(layer, T, per_kernel, K):
    """per-kernel ms per step, named by what ran (one routing kernel or three)"""
    kern_ms = {k: v / K for k, v in per_kernel.items()}
    plan = layer.plan(T)
    if plan["route_kernels"] == 1:  # one cooperative routing kernel: its whole time is in the first span
        kern_ms["route_fused"] = kern_ms.pop("route_count")
        kern_ms.pop("route_scan")
        kern_ms.pop("route_scatter")
    return kern_ms, plan


def rooflines(wl, counts, kern_ms, ms_step):
    """The layer roofline and the dominant kernel's (FC1).  FP8 dense peak = 2 x
    the measured BF16 burst figure (the nominal FP8:BF16 ratio, 4.5 : 2.25): a
    forward is a kernel chain timed in isolation, so the burst figure is its
    denominator; the fraction of 2 x the sustained figure (measured back to
    back under the power cap) is reported beside it, never in its place."""
    hbm, bf16, bf16_sus, src = peaks()
    fp8 = 2.0 * bf16
    fp8_sus = 2.0 * bf16_sus if bf16_sus else None
    flops = wl.routed_flops
    b_alg, touched = algorithmic_bytes(wl, counts)
    t_fp8, t_hbm = flops / (fp8 * 1e12), b_alg / (hbm * 1e9)
    t_roof = max(t_fp8, t_hbm)
    tflops = flops / (ms_step * 1e-3) / 1e12
    layer = {"t_roof_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms_step,
             "bound": "fp8 tensor" if t_fp8 >= t_hbm else "hbm",
             "b_alg_bytes": b_alg, "experts_touched": touched,
             "fp8_peak_tflops": fp8, "fp8_peak": "2 x measured bf16 burst", "hbm_gbs": hbm,
             "fp8_peak_frac": tflops / fp8,
             "fp8_peak_frac_vs_sustained": (tflops / fp8_sus) if fp8_sus else None,
             "source": src}
    R = int(counts.sum())
    fc1_flops = 2 * R * wl.H * 2 * wl.I
    fc1_ms = kern_ms["fc1"]
    fc1_bytes = touched * (2 * wl.I * wl.H) + R * wl.H
    if fc1_flops / fc1_bytes >= fp8 * 1e12 / (hbm * 1e9):
        roof = {"bound": "tensor", "achieved": fc1_flops / (fc1_ms * 1e-3) / 1e12, "peak": fp8,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": fc1_bytes / (fc1_ms * 1e-3) / 1e9, "peak": hbm,
                "unit": "GB/s"}
    roof.update({"frac": roof["achieved"] / roof["peak"],
                 "traffic": recorded_traffic(wl.name, "fc1"), "kernel": "fc1",
                 "algorithmic_flops": fc1_flops, "algorithmic_bytes": fc1_bytes,
                 "peak_source": f"{src}: FP8 = 2 x bf16 burst" if roof["bound"] == "tensor"
                 else f"{src}: hbm copy"})
    return layer, roof, tflops


def tactic_str(layer, plan):
    t = layer.tactic()
    sw = plan.get("swap_ab_tokens", 0)
    return {"gemm": ("cta pairs" if t["gemm_pair"] else "single cta") + f" x{t['gemm_ctas']}"
                    + (f", token-as-N (tile {sw})" if sw else ""),
            "routing": "one cooperative kernel" if plan["route_kernels"] == 1 else "three kernels",
            "gemms": ("FC1 + FC2 in one persistent launch" if plan["gemm_launches"] == 1
                      else "two launches")
                     + (", combine folded into FC2" if plan.get("combine_in_fc2") else "")}


def l2_note(wl, b_alg):
    return ("flushed before every step (256 MiB write, untimed)"
            + (f"; the step also streams {b_alg / 1e9:.2f} GB of compulsory bytes, more than L2"
               if b_alg > L2_BYTES else ""))


def measure_record(torch, S, g, name, args, dev, stream, flush, weights_cache):
    """One workload of the per-workload record: the main line's device timing
    method (graph replay, L2 flushed before every step, W warm-up and K timed
    steps, per-kernel times from the profiled capture)."""
    from gen import configs
    wl = configs.WORKLOADS[name]
    key = (wl.H, wl.I, wl.E, wl.seed)
    if key not in weights_cache:
        weights_cache.clear()
        torch.cuda.empty_cache()
        weights_cache[key] = gpu_weights(torch, g, S.MegaMoELayer, wl, args.format, dev, stream)
    layer = S.MegaMoELayer(wl.H, wl.I, wl.E, wl.K, max_rows=wl.T, expected_m=wl.T,
                           fuse_fc1=not args.unfused, check_routes=True, gemm=args.gemm,
                           gemms=args.gemms, fmt=args.format, swap_ab=not args.no_swap,
                           combine_in_fc2=args.combine_in_fc2)
    bind(layer, weights_cache[key], args.format, stream)
    x, idx, wts, _, _, counts = device_inputs(torch, g, wl, dev, stream)
    torch.cuda.synchronize()
    timer = StepTimer(torch, layer, x, idx, wts, stream, flush, not args.no_graph)
    K = max(args.steps, 1)
    torch.cuda.synchronize()
    time.sleep(SETTLE_S)
    timer.steps(args.warmup)
    times = []
    total, _ = timer.steps(K, keep=times)
    timer.steps(min(args.warmup, 3), True)
    _, per_kernel = timer.steps(K, True)
    timer.check_status(f"{name} forwards")
    ms = total / K
    kern_ms, plan = kernel_times(layer, wl.T, per_kernel, K)
    lroof, roof, tflops = rooflines(wl, counts, kern_ms, ms)
    rec = {"workload": wl.name, "T": wl.T, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
           "step_ms": {"median": float(np.median(times)), "p10": float(np.percentile(times, 10)),
                       "p90": float(np.percentile(times, 90))},
           "tflops": tflops, "tokens_per_s": wl.T / (ms * 1e-3), "layer_roofline": lroof,
           "roofline": roof, "kernel_ms": kern_ms, **tactic_str(layer, plan),
           "l2": l2_note(wl, lroof["b_alg_bytes"])}
    del timer, layer, x, idx, wts
    torch.cuda.synchronize()
    return rec


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")

    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    from gen import configs, problem
    from gen import inputs as g

    wl = configs.WORKLOADS[args.config]
    if args.experts or args.tokens:
        from gen.configs import Workload
        E = args.experts or wl.E
        T = args.tokens or wl.T
        name = wl.name + (f"_E{E}" if args.experts else "") + (f"_T{T}" if args.tokens else "")
        wl = Workload(name, T, wl.H, wl.I, E, wl.K, wl.routing, wl.seed)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream()
    fused = not args.unfused

    layer = S.MegaMoELayer(wl.H, wl.I, wl.E, wl.K, max_rows=wl.T, expected_m=wl.T,
                           fuse_fc1=fused, check_routes=True, gemm=args.gemm,
                           gemms=args.gemms, fmt=args.format, swap_ab=not args.no_swap,
                           combine_in_fc2=args.combine_in_fc2)
    # weights: generated and quantised on the GPU, bound once; kept for the
    # per-workload record when workloads there share them (dsv3 prefill/decode)
    weights = gpu_weights(torch, g, S.MegaMoELayer, wl, args.format, dev, stream)
    bind(layer, weights, args.format, stream)
    weights_cache = {}
    if not (args.experts or args.tokens):
        weights_cache[(wl.H, wl.I, wl.E, wl.seed)] = weights
    del weights
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    x, idx, wts, idx_np, w_np, counts = device_inputs(torch, g, wl, dev, stream)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    if args.side_mlp:
        side_stream_sweep(args, torch, layer, x, idx, wts, wl, dev, flush)
        return
    if args.sm_budget:
        layer.set_sm_budget(args.sm_budget)

    timer = StepTimer(torch, layer, x, idx, wts, stream, flush, not args.no_graph)
    torch.cuda.synchronize()
    time.sleep(SETTLE_S)
    warm_ms, _ = timer.steps(args.warmup)
    if args.steps <= 0:
        # about a second of timed work (at least 20 steps, at most 5000)
        est = reduce_max(warm_ms / max(1, args.warmup), dev)
        args.steps = int(min(5000, max(20, math.ceil(1000.0 / max(est, 1e-3)))))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    step_times = []
    total_ms, _ = timer.steps(args.steps, keep=step_times)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = reduce_max(total_ms, dev)
    # beside the flushed figure: the same capture replayed back to back with
    # nothing flushed between steps (whatever of the working set L2 keeps)
    n_warm = min(L2_WARM_STEPS, args.steps)
    l2_warm_ms = reduce_max(timer.l2_warm(n_warm), dev)
    # per-kernel times: the same number of steps of the profiled capture
    timer.steps(min(args.warmup, 3), True)
    prof_ms, per_kernel = timer.steps(args.steps, True)
    timer.check_status("timed forwards")
    graph_used = timer.graph is not None
    del timer

    # ---------------------------------------------------------------- e2e
    # The public call a user makes with host buffers: every step copies its x
    # and routes from pinned host memory and reads its output back, all inside
    # the timed span.  Two figures: (1) serial -- copy in, forward, copy out,
    # one step after the other on one stream, L2 flushed before each step;
    # (2) pipelined, the way a serving loop runs it -- two device slots, copies
    # on their own streams, so step i+1's inputs and step i-1's output move
    # while step i computes; nothing is flushed between its steps (the value
    # says whether the step's compulsory bytes exceed L2).  The value is the
    # pipelined figure; the serial one is reported beside it.
    x_host = torch.from_numpy(problem.x_bits(wl).view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    idx_host = torch.from_numpy(idx_np).pin_memory()
    w_host = torch.from_numpy(w_np).pin_memory()
    out_host = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    idx_d = [torch.empty_like(idx) for _ in range(2)]
    w_d = [torch.empty_like(wts) for _ in range(2)]
    out_d = [layer.out, torch.empty_like(layer.out)]
    h2d = x_host.numel() * 2 + idx_host.numel() * 4 + w_host.numel() * 4
    d2h = out_host[0].numel() * 2
    layer.set_profile_events([])
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)

    def e2e_serial_step():
        with torch.cuda.stream(stream):
            x_d[0].copy_(x_host, non_blocking=True)
            idx_d[0].copy_(idx_host, non_blocking=True)
            w_d[0].copy_(w_host, non_blocking=True)
            out = layer.forward(x_d[0], idx_d[0], w_d[0], stream=stream)
            out_host[0].copy_(out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_serial_step()
    stream.synchronize()
    e2e_serial_ms = 0.0
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            flush.zero_()
            t_start.record(stream)
        e2e_serial_step()
        with torch.cuda.stream(stream):
            t_end.record(stream)
        stream.synchronize()
        e2e_serial_ms += t_start.elapsed_time(t_end)
    e2e_serial_ms = reduce_max(e2e_serial_ms, dev)

    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_fwd = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]

    def e2e_pipelined(n):
        for e in ev_fwd + ev_d2h:
            e.record(stream)
        for i in range(n):
            s = i & 1
            with torch.cuda.stream(h2d_stream):
                h2d_stream.wait_event(ev_fwd[s])      # the slot's previous forward has read it
                x_d[s].copy_(x_host, non_blocking=True)
                idx_d[s].copy_(idx_host, non_blocking=True)
                w_d[s].copy_(w_host, non_blocking=True)
                ev_h2d[s].record(h2d_stream)
            stream.wait_event(ev_h2d[s])
            stream.wait_event(ev_d2h[s])               # the slot's previous output is on the host
            layer.stage_output(out_d[s])
            layer.forward(x_d[s], idx_d[s], w_d[s], stream=stream)
            ev_fwd[s].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_fwd[s])
                out_host[s].copy_(out_d[s][:wl.T], non_blocking=True)
                ev_d2h[s].record(d2h_stream)
        stream.wait_event(ev_d2h[(n - 1) & 1])
        stream.wait_event(ev_d2h[n & 1])

    with torch.cuda.stream(stream):
        e2e_pipelined(max(2, args.warmup))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        flush.zero_()
        t_start.record(stream)
        e2e_pipelined(args.steps)
        t_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(t_start.elapsed_time(t_end), dev)
    layer.stage_output(out_d[0])
    st, bits = layer.read_status(stream)
    if st != 0:
        raise RuntimeError(f"e2e forwards reported device status {bits:#x}")
    if not torch.equal(out_host[0], out_host[1]):
        raise RuntimeError("pipelined end-to-end outputs differ between the two slots")

    # ---------------------------------------------------------------- report
    K = args.steps
    flops = wl.routed_flops
    ms_step = total_ms / K
    value = aggregate_rate(world, flops, K, total_ms) / 1e12
    e2e_value = aggregate_rate(world, flops, K, e2e_ms) / 1e12
    kern_ms, plan = kernel_times(layer, wl.T, per_kernel, K)
    lroof, roof, _ = rooflines(wl, counts, kern_ms, ms_step)
    big = lroof["b_alg_bytes"] > L2_BYTES
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "K": wl.K,
                   "fc1_epilogue": "fused" if fused else "unfused",
                   "format": fmt_name(args.format),
                   "l2": l2_note(wl, lroof["b_alg_bytes"]),
                   "launch": "cuda graph replay" if graph_used else "direct launches",
                   "timing": f"set-up, then {SETTLE_S:g} s idle, warm-up, timed steps (the burst "
                             "power regime; the part reaches its power limit after ~0.3 s of load)",
                   **tactic_str(layer, plan),
                   "sm_budget": args.sm_budget or None,
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": aggregate_rate(world, wl.T, K, total_ms),
        "layer_roofline": lroof,
        "roofline": roof,
        "step_ms": {"median": float(np.median(step_times)), "p10": float(np.percentile(step_times, 10)),
                    "p90": float(np.percentile(step_times, 90))},
        "l2_warm": {"ms_per_step": l2_warm_ms, "steps": n_warm,
                    "how": "the same capture replayed back to back, L2 not flushed (not the value)"},
        "kernel_ms": kern_ms,
        "kernel_ms_source": ("CUDA events before every kernel, a second capture of the same forward "
                             f"replayed for the same {K} steps right after the timed ones "
                             f"({prof_ms / K:.4f} ms per step with the events in place; FC1 and FC2 "
                             "run there as two launches of the same GEMM code)"),
        "gpu_launches": K * plan["kernels"],
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / K,
                "copies": "pipelined: two device slots; H2D and D2H on their own streams overlap the "
                          "neighbouring steps' forwards",
                "l2": ("not flushed between the pipelined steps; each step's compulsory bytes exceed L2"
                       if big else "not flushed between the pipelined steps (L2-warm)"),
                "serial": {"value": aggregate_rate(world, flops, K, e2e_serial_ms) / 1e12,
                           "ms_per_step": e2e_serial_ms / K,
                           "l2": "flushed before every step (untimed)"}},
    }
    del x_d, idx_d, w_d, out_d, layer
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_bits = x_host.view(torch.int16).numpy().view(np.uint16)
        line["cpu_baseline"] = oracle_bounded_run(wl, x_bits, idx_np, w_np, CPU_BASELINE_S,
                                                  np.random.default_rng(0))
    if world == 1 and not args.no_records:
        torch.cuda.empty_cache()
        names = [n for n in args.records.split(",") if n and configs.WORKLOADS[n].name != wl.name]
        clocks = ClockSampler(local)
        recs = {}
        for n in names:
            recs[n] = measure_record(torch, S, g, n, args, dev, stream, flush, weights_cache)
        line["per_workload"] = {
            "how": ("each workload as the main line times it (CUDA graph replay, L2 flushed before "
                    f"every step, {args.warmup} warm-up and {K} timed steps, per-kernel times "
                    "from the profiled capture), in this run, after the main line"),
            "clocks": clocks.stop(), "records": recs}
    weights_cache.clear()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
