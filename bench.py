"""Benchmark of the routed MoE expert FFN layer (MXFP4 weights, online FP8
activations) on GB300.

One step = one moe_forward over one batch of synthetic tokens (route, histogram +
scan + permute, FP8 quantisation, W13 grouped GEMM, SwiGLU + FP8 requantisation, W2
grouped GEMM, weighted top-k combine + shared-expert add).  Inputs are resident in
HBM when the timed region starts.  L2 between timed steps (--l2): "auto" (default)
flushes it with a 512 MiB write before every step, outside its CUDA-event pair, unless
one step streams at least 4x the L2 size of expert weights (decode, decode256,
prefill: 1.8-13.5 GB per step against a 126 MB L2), where no step's weights can be
L2-resident and the write-flush would only add its own dirty-line write-back to the
next step; such runs also report the write-flushed step time.  Prints one JSON line
on rank 0.

The default run (--workload decode) times the 7-token decode layer for the line's
headline value, and in the same invocation measures the 256-token decode layer, the
32K-token prefill chunk (each for >= 2 s, with its own clock samples) and the
grouped-GEMM shape sweep; those are reported under "workloads" and "sweep" in the same
line (--no-extra skips them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|decode256|prefill|tiny]
  python bench.py --workload sweep       (the grouped-GEMM sweep alone, every point)
  python bench.py --workload gemm --gemm w13|w2 --groups G --rows M [--weights nvfp4]
                                         (one grouped GEMM, e.g. for an ncu capture)
  python bench.py --workload prefill --options pair_tiles,...   (moe_forward_ex options)
  python bench.py --impl reference ...   (the CPU oracle on a bounded sample)

Multi-GPU: one independent replica per GPU (the layer is not sharded; no
collective); value = tokens processed by all ranks / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gen import inputs as gi  # noqa: E402

METRIC = "MoE-layer tokens/s"
WEIGHT_BYTES_PER_ELEM = 0.5 + 1.0 / 32.0  # E2M1 code + E8M0 scale per 32
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode",
                    choices=list(gi.WORKLOADS) + ["sweep", "gemm"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-flush", action="store_true", help="same as --l2 none")
    ap.add_argument("--l2", default="auto", choices=["auto", "flush", "none"])
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (a smaller layer of the same shape, for ncu captures)")
    ap.add_argument("--tokens", type=int, default=None, help="override T")
    ap.add_argument("--weights", default="mxfp4", choices=["mxfp4", "nvfp4"],
                    help="expert weight format of the measured layer")
    ap.add_argument("--no-extra", action="store_true",
                    help="decode only: skip the decode256 / prefill / sweep records")
    ap.add_argument("--options", default="",
                    help="comma list of moe_forward_ex options for the measured layer "
                         "(fuse_swiglu, fuse_combine, pair_tiles)")
    ap.add_argument("--gemm", default="w13", choices=["w13", "w2"],
                    help="--workload gemm: which grouped GEMM (sweep shapes)")
    ap.add_argument("--groups", type=int, default=64, help="--workload gemm: groups")
    ap.add_argument("--rows", type=int, default=2, help="--workload gemm: rows per group")
    return ap.parse_args()


def dist_init(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                return json.load(f), "measured"
        except Exception:
            pass
    return None, "fallback"


def hbm_peak_gbs():
    peaks, src = measured_peaks()
    if peaks:
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in peaks:
                v = peaks[key]
                if isinstance(v, dict):
                    v = v.get("burst", v.get("value"))
                try:
                    return float(v), "measured"
                except (TypeError, ValueError):
                    pass
    return FALLBACK_HBM_GBS, "fallback"


def fp8_tensor_peak_tflops(sustained=False):
    """Dense FP8 tensor peak: the measured bf16 cuBLAS peak x the nominal 2x FP8/bf16
    ratio (the burst figure, or with sustained=True the seconds-long loop's figure, for
    a kernel timed inside a long run of steps), else the fallback bf16 figure x 2."""
    peaks, _ = measured_peaks()
    if peaks:
        keys = ("bf16_tflops_sustained",) if sustained else ("bf16_tflops", "bf16")
        for key in keys:
            if key in peaks:
                try:
                    return 2.0 * float(peaks[key]), (
                        f"measured bf16 {'sustained' if sustained else 'burst'} x2 "
                        "(nominal fp8/bf16 ratio)")
                except (TypeError, ValueError):
                    pass
        if sustained:
            return fp8_tensor_peak_tflops(False)
    return 2.0 * FALLBACK_BF16_TFLOPS, "fallback bf16 x2 (nominal fp8/bf16 ratio)"


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per active weight group of
# one small-M W13 GEMM launch, from the committed ncu summary of the small-M W13 launch
# on the 7-token, 64-expert layer, keyed by the hash of the GEMM sources it was taken
# on.  A changed kernel reports traffic null until it is captured again.
NCU_SMALL_W13_TRAFFIC = {"src": "bf194fcfbaae33fc", "bytes_per_group": (964.70e6 + 4.00e6) / 41}


def gemm_src_hash():
    import hashlib
    csrc = os.path.join(ROOT, "moe_expert_ffn_scan_gb300", "csrc")
    digests = []
    for name in ("gemm.cu", "kernels.cuh", "common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            digests.append(hashlib.sha256(f.read()).hexdigest())
    return hashlib.sha256(("\n".join(digests) + "\n").encode()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running.

    `load()` brackets a region of GPU work (a context manager); `summary(tag)` reports
    only the samples whose nvidia-smi timestamps fall inside the regions marked with
    that tag, so idle time before and after them does not count."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")
        self.windows = []  # (tag, t0, t1) host wall-clock times

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    class _Load:
        def __init__(self, owner, tag):
            self.owner, self.tag = owner, tag

        def __enter__(self):
            self.t0 = datetime.datetime.now()
            return self

        def __exit__(self, *a):
            self.owner.windows.append((self.tag, self.t0, datetime.datetime.now()))

    def load(self, tag):
        return ClockSampler._Load(self, tag)

    def summary(self, tag=None):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        wins = [(a, b) for t, a, b in self.windows if tag is None or t == tag]
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        try:
            lines = open(self.path).read().splitlines()
        except OSError:
            lines = []
        for line in lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f")
                f_sm, f_max = float(p[2]), float(p[3])
            except ValueError:
                continue
            if wins and not any(a <= ts <= b for a, b in wins):
                continue
            sm.append(f_sm)
            smax.append(f_max)
            for n, v in zip(names, p[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def make_layer_for(args, workload, seed, dev):
    if args.experts is None and args.tokens is None:
        return gi.make_layer(workload, seed=seed, device=dev)
    import dataclasses
    d = gi.WORKLOADS[workload]
    d = dataclasses.replace(d, E=args.experts or d.E, T=args.tokens or d.T)
    return d, gi.custom_layer(d, seed=seed, device=dev, logits_kind=gi.LOGITS_KIND[workload])


def active_groups(counts, has_shared):
    return int((counts > 0).sum()) + (1 if has_shared else 0)


# ------------------------------------------------------------------ CPU oracle ------

def oracle_sample(d, t_host_fn, tokens, seed):
    """Times the oracle on `tokens` tokens of the workload (their experts only)."""
    from oracle import moe_oracle as o
    x, lg, w_get = t_host_fn()
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(d.T, size=min(tokens, d.T), replace=False))
    t0 = time.perf_counter()
    ridx, _ = o.route(lg[toks], d.k)
    experts = sorted(set(ridx.ravel().tolist()) | ({d.E} if d.has_shared else set()))
    w13, w13s, w2, w2s = w_get(experts)
    o.moe_forward_tokens(x, lg, d.k, w13, w13s, w2, w2s, d.has_shared, toks)
    dt = time.perf_counter() - t0
    return len(toks), dt


def host_view(d, t):
    """Callables giving the oracle numpy views of the layer inputs (weights copied to
    the host only for the experts a sample touches)."""
    x = t["x"].cpu().view(torch.int16).numpy().view(np.uint16)
    if t.get("wg") is not None:
        # logits that are the gate projection of x: the oracle projects them itself
        from oracle import moe_oracle as o
        lg = o.router_logits(x, t["wg"].cpu().numpy()).astype(np.float32)
    else:
        lg = t["logits"].cpu().numpy()

    def w_get(experts):
        shp = lambda n: (d.G,) + tuple(t[n].shape[1:])
        out = [np.zeros(shp(n), np.uint8) for n in ("w13", "w13_s", "w2", "w2_s")]
        for e in experts:
            for a, n in zip(out, ("w13", "w13_s", "w2", "w2_s")):
                a[e] = t[n][e].cpu().numpy()
        return out

    return lambda: (x, lg, w_get)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


# ------------------------------------------------------------------ arms ------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload in ("sweep", "gemm"):
        print(json.dumps({"impl": "reference", "unavailable": "the GEMM sweep has no CPU arm; "
                          "run a layer workload"}), flush=True)
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d, t = make_layer_for(args, args.workload, args.seed, dev)
    hv = host_view(d, t)
    # tokens per step: one, or more when one is quick, keeping the whole run at about
    # three minutes (the tiny layer runs in full every step)
    _, t1 = oracle_sample(d, hv, 1, args.seed)
    per_step = min(10.0, 180.0 / max(1, args.steps + args.warmup))
    tokens = max(1, min(d.T, int(per_step / max(t1, 1e-3))))
    times = []
    n_done = 0
    for i in range(args.warmup + args.steps):
        n, dt = oracle_sample(d, hv, tokens, args.seed + i)
        if i >= args.warmup:
            times.append(dt)
            n_done += n
    total = sum(times)
    value = n_done / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "T": d.T, "H": d.H, "I": d.I, "E": d.E,
                   "k": d.k, "shared_experts": d.has_shared},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"{tokens} token(s) per step"
                                   + (" (the whole layer)" if tokens == d.T else "")
                                   + f", their top-{d.k} experts"
                                   + (" and the shared expert" if d.has_shared else "")
                                   + ", full layer in float64 numpy"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bf16_tensor_peak_tflops(sustained=False):
    """Dense bf16 tensor peak (the NVFP4 path's kind::f16 MMAs): the measured cuBLAS
    bf16 burst figure (sustained=True: the seconds-long loop's), else the fallback."""
    peaks, _ = measured_peaks()
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    if peaks and key in peaks:
        try:
            return float(peaks[key]), f"measured bf16 (cuBLAS {'sustained' if sustained else 'burst'})"
        except (TypeError, ValueError):
            pass
    if sustained:
        return bf16_tensor_peak_tflops(False)
    return FALLBACK_BF16_TFLOPS, "fallback bf16"


WEIGHT_BYTES = {"mxfp4": 0.5 + 1.0 / 32.0, "nvfp4": 0.5 + 1.0 / 16.0}


def gemm_roofline(d, groups, t_ms, which, hbm, hbm_src, tpk, tpk_src, fmt="mxfp4",
                  tpk_burst=None):
    """Roofline of one grouped GEMM launch sequence (W13 or W2) of a layer step.
    Algorithmic bytes: the active groups' weight bytes (codes + scales) plus the packed
    FP8 rows and scales read and the bf16 rows written; flops: 2 x rows x N x K.  The
    bound is HBM when the flops per byte sit below the ridge point, else the tensor
    pipe (kind::mxf8f6f4 runs at the FP8 rate)."""
    Rs = d.R + (d.T if d.has_shared else 0)
    if which == "w13":
        N, K = 2 * d.I, d.H
    else:
        N, K = d.H, d.I
    wbytes = groups * N * K * WEIGHT_BYTES[fmt]
    # packed activation rows read (FP8 codes + scales, or bf16 values) + bf16 rows out
    abytes = Rs * ((K + K / 128) if fmt == "mxfp4" else 2 * K) + Rs * N * 2
    flops = 2.0 * Rs * N * K
    t = t_ms * 1e-3
    if flops / (wbytes + abytes) < (tpk * 1e12) / (hbm * 1e9):
        ach = (wbytes + abytes) / t / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "traffic": None, "peak_source": f"{hbm_src} HBM copy bandwidth",
                "algorithmic_bytes": wbytes + abytes}
    ach = flops / t / 1e12
    rec = {"bound": "tensor", "achieved": ach, "peak": tpk, "unit": "TFLOP/s",
           "frac": ach / tpk, "traffic": None, "peak_source": tpk_src,
           "algorithmic_flops": flops}
    if tpk_burst is not None and tpk_burst != tpk:
        rec["frac_of_burst_peak"] = ach / tpk_burst
        rec["burst_peak"] = tpk_burst
    return rec


def measure_layer(args, workload, steps, warmup, rank, world, local, clocks, *, soak_s=0.0,
                  e2e_steps=None, router=False, cpu=False, fmt="mxfp4", tag=None, options=(),
                  tune=False):
    """One workload: the layer step captured as a CUDA graph, timed over `steps` replays
    (each followed by an event-instrumented forward for the stage times), inside a
    clock-sampling window tagged `tag` (the workload's name).  fmt: the expert weight
    format (MXFP4, or NVFP4 drawn by gen.inputs.nvfp4_layer_weights).  Returns a dict."""
    import moe_expert_ffn_scan_gb300 as moe
    tag = tag or workload
    dev = torch.device("cuda", local)
    d, t = make_layer_for(args, workload, args.seed + rank, dev)
    if t["logits"] is None:  # logits are the gate projection of x: the library's router
        t["logits"] = torch.empty(d.T, d.E, dtype=torch.float32, device=dev)
        moe.moe_router_logits(t["x"], t["wg"], t["logits"])
    md = moe.dims(d.T, d.H, d.I, d.E, d.k, d.has_shared)
    if fmt == "nvfp4":
        for n in ("w13", "w13_s", "w2", "w2_s"):
            del t[n]
        t.update(gi.nvfp4_layer_weights(d, seed=args.seed + rank, device=dev))
    # --options applies to the headline layer only
    layer_opts = ({o_: True for o_ in args.options.split(",") if o_}
                  if tag == workload == args.workload else {})
    layer = moe.MoELayer(d.H, d.I, d.E, d.k, d.has_shared, t["w13"], t["w13_s"], t["w2"],
                         t["w2_s"], fmt=fmt, w13_gs=t.get("w13_gs"), w2_gs=t.get("w2_gs"),
                         **layer_opts)
    x, lg = t["x"], t["logits"]
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device=dev)
    ws = layer.workspace(d.T)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    # routing statistics (for the algorithmic byte / flop counts)
    dbg = {"counts": torch.empty(d.E, dtype=torch.int32, device=dev)}
    layer.forward(x, lg, out=out, debug=dbg)
    bits = moe.moe_check_status(ws)
    if bits:
        raise RuntimeError(f"device status bits {bits:#x}")
    counts = dbg["counts"].cpu().numpy()
    groups = active_groups(counts, d.has_shared)
    step_weight_bytes = groups * 3 * d.I * d.H * WEIGHT_BYTES[fmt]
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    policy = "none" if args.no_flush else args.l2
    do_flush = policy == "flush" or (policy == "auto" and step_weight_bytes < 4 * l2_bytes)
    if do_flush:
        l2_note = "flushed (512 MiB write) before each step"
    else:
        l2_note = (f"not flushed: each step streams {step_weight_bytes / 1e9:.2f} GB of expert "
                   f"weights ({step_weight_bytes / l2_bytes:.0f}x the {l2_bytes >> 20} MiB L2)")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(steps)]
    for row in evs:
        for e in row:
            e.record(stream)  # creates the event handles
    for _ in range(warmup):
        layer.forward(x, lg, out=out)
    torch.cuda.synchronize()
    # One step = one replay of the layer captured as a CUDA graph (every launch of the
    # path, PDL edges between them).  Stage times come from an event-instrumented
    # forward run right after it, inside the same timed region.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x, lg, out=out)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(steps)]

    with clocks.load(tag):
        if soak_s > 0:
            # back-to-back replays of the same graph right before the timed region, so
            # that the clock sampler sees the GPU under this load for a few seconds
            t_end = time.perf_counter() + soak_s
            while time.perf_counter() < t_end:
                for _ in range(64):
                    graph.replay()
                torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        for i in range(steps):
            if do_flush:
                flush.fill_(i & 0xFF)
            step_evs[i][0].record(stream)
            graph.replay()
            step_evs[i][1].record(stream)
            if do_flush:
                flush.fill_((i + 128) & 0xFF)
            layer.forward_timed(x, lg, out, evs[i])
        torch.cuda.synchronize()
        barrier(world)
    bits = moe.moe_check_status(ws)
    if bits:
        raise RuntimeError(f"device status bits {bits:#x}")
    stage_ms = {s_: [] for s_ in moe.STAGES}
    step_ms = [a_.elapsed_time(b_) for a_, b_ in step_evs]
    for row in evs:
        for j, s_ in enumerate(moe.STAGES):
            stage_ms[s_].append(row[j].elapsed_time(row[j + 1]))
    stream_step_ms = statistics.mean(row[0].elapsed_time(row[7]) for row in evs)
    flushed_ms = None
    if not do_flush:  # the same graph with the 512 MiB write-flush before each step
        n_f = min(steps, 50)
        fe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_f)]
        for i in range(n_f):
            flush.fill_(i & 0xFF)
            fe[i][0].record(stream)
            graph.replay()
            fe[i][1].record(stream)
        torch.cuda.synchronize()
        flushed_ms = max_over_ranks(statistics.mean(a_.elapsed_time(b_) for a_, b_ in fe), world)
    ms = statistics.mean(step_ms)
    qs = (statistics.quantiles(step_ms, n=10, method="inclusive") if len(step_ms) >= 2
          else [ms] * 9)
    pct = {"p10": qs[0], "p50": statistics.median(step_ms), "p90": qs[8]}
    ms_max = max_over_ranks(ms, world)
    stage_mean = {s_: statistics.mean(v) for s_, v in stage_ms.items()}

    hbm, hbm_src = hbm_peak_gbs()
    # a timed region of a second or more of back-to-back steps is a long run: the
    # tensor peak is then the measured sustained figure (the burst one is reported too)
    long_run = sum(step_ms) >= 1000.0
    peak_fn = fp8_tensor_peak_tflops if fmt == "mxfp4" else bf16_tensor_peak_tflops
    tpk_burst, _ = peak_fn(False)
    tpk, tpk_src = peak_fn(long_run)
    roof13 = gemm_roofline(d, groups, stage_mean["gemm_w13"], "w13", hbm, hbm_src, tpk, tpk_src,
                           fmt, tpk_burst)
    roof2 = gemm_roofline(d, groups, stage_mean["gemm_w2"], "w2", hbm, hbm_src, tpk, tpk_src,
                          fmt, tpk_burst)
    kname = "k_gemm_mx" if fmt == "mxfp4" else "k_gemm_nv"
    roof13["kernel"] = f"{kname} (W13 grouped GEMM)"
    roof2["kernel"] = f"{kname} (W2 grouped GEMM)"
    if fmt == "mxfp4" and roof13["bound"] == "hbm" and d.T <= 16 and \
            gemm_src_hash() == NCU_SMALL_W13_TRAFFIC["src"]:
        roof13["traffic"] = groups * NCU_SMALL_W13_TRAFFIC["bytes_per_group"]

    # end to end through the public API, host buffers, copies inside the timed region
    e2e = None
    if e2e_steps and fmt == "mxfp4":
        e2e = measure_e2e(layer, d, x, lg, out, e2e_steps, do_flush, flush, world)

    # the layer again with each option of moe_forward_ex (f1 SwiGLU in the W13 epilogue,
    # f2 combine in the W2 epilogue, SM-pair tiles), same inputs and weights: its step
    # time beside the default's, and whether its output equals the default's bit for bit
    opt_rec = {}
    if options and fmt == "mxfp4":
        out.zero_()
        layer.forward(x, lg, out=out)
        torch.cuda.synchronize()
        ref_out = out.clone()
        n_o = min(steps, 30)
        for opt in options:
            lo = moe.MoELayer(d.H, d.I, d.E, d.k, d.has_shared, t["w13"], t["w13_s"], t["w2"],
                              t["w2_s"], **{opt: True})
            o_out = torch.zeros_like(out)
            lo.forward(x, lg, out=o_out)
            torch.cuda.synchronize()
            o_bits = moe.moe_check_status(lo.workspace(d.T))
            same = bool(torch.equal(o_out, ref_out)) and o_bits == 0
            og = torch.cuda.CUDAGraph()
            with torch.cuda.graph(og):
                lo.forward(x, lg, out=o_out)
            for _ in range(warmup):
                og.replay()
            oe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(n_o)]
            for i in range(n_o):
                if do_flush:
                    flush.fill_(i & 0xFF)
                oe[i][0].record(stream)
                og.replay()
                oe[i][1].record(stream)
            torch.cuda.synchronize()
            o_ms = max_over_ranks(statistics.mean(a_.elapsed_time(b_) for a_, b_ in oe), world)
            opt_rec[opt] = {"ms_per_step": o_ms, "vs_default": o_ms / ms_max,
                            "output_identical_to_default": same, "steps": n_o}
            del og, lo, o_out
            torch.cuda.synchronize()
            torch.cuda.empty_cache()

    # exact-shape tuning of the tile plan on this batch's routing histogram: the chunk
    # size for groups above 64 rows (every candidate gives the same output bit for bit)
    tune_rec = None
    if tune and fmt == "mxfp4":
        best, times = layer.tune_chunk_rows(x, lg, steps=10, warmup=3)
        layer.large_chunk_rows = 0
        tune_rec = {"best_chunk_rows": best, "ms_per_candidate": times,
                    "default_chunk_rows": 224,
                    "gain_vs_default": times[224] / times[best] if 224 in times else None,
                    "how": "median of 10 forwards per candidate (CUDA events, not graphs)"}

    router_rec = None
    if router:
        # the router gate projection for this workload's T (outside the layer step: the
        # layer's boundary takes logits); W_g synthetic fp32 [E, H]
        wg = t["wg"] if t.get("wg") is not None else gi.gate_weight(d.E, d.H, args.seed, dev)
        rlg = torch.empty(d.T, d.E, dtype=torch.float32, device=dev)
        # above ROUTER_TC_MIN_T tokens the tensor-core form (W_g split once per weight
        # into three bf16 pieces, outside the timed region); below, the fp32 GEMV
        use_tc = d.T >= ROUTER_TC_MIN_T
        if use_tc:
            wg3 = moe.moe_router_split(wg)

            def router_call():
                moe.moe_router_logits_split(x, wg3, rlg)
        else:
            def router_call():
                moe.moe_router_logits(x, wg, rlg)
        for _ in range(3):
            router_call()
        n_r = min(steps, 20)
        r_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n_r)]
        for i in range(n_r):
            if do_flush:
                flush.fill_(i & 0xFF)
            r_ev[i][0].record(stream)
            router_call()
            r_ev[i][1].record(stream)
        torch.cuda.synchronize()
        r_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in r_ev)
        r_bytes = d.E * d.H * (6 if use_tc else 4) + d.T * d.H * 2 + d.T * d.E * 4
        r_flop = 2.0 * d.T * d.E * d.H
        router_rec = {"ms": r_ms, "gbs": r_bytes / (r_ms * 1e-3) / 1e9,
                      "tflops": r_flop / (r_ms * 1e-3) / 1e12,
                      "kernel": "k_router_tc" if use_tc else
                      ("k_router_gemv" if d.T <= 1024 else "k_router_tiled")}
        if use_tc:
            # three bf16 MMAs per product: the tensor pipe's work is 3x the projection's
            bpk, bpk_src = bf16_tensor_peak_tflops()
            router_rec["tensor_frac"] = 3.0 * r_flop / (r_ms * 1e-3) / 1e12 / bpk
            router_rec["tensor_peak"] = {"tflops": bpk, "source": bpk_src}

    cpu_rec = None
    if cpu and rank == 0:
        hv = host_view(d, t)
        # one token first; when that is quick, as many more as about 10 s of oracle
        # work allows (the tiny layer runs in full)
        n, dt = oracle_sample(d, hv, 1, args.seed)
        more = min(d.T, int(10.0 / max(dt, 1e-3)))
        if more > 1:
            n, dt = oracle_sample(d, hv, more, args.seed)
        whole = " (the whole layer)" if n == d.T else ""
        shared = " + shared expert" if d.has_shared else ""
        cpu_rec = {"value": n / dt, "unit": "tokens/s", "cores": blas_threads(),
                   "kind": "oracle",
                   "sample": f"{n} token(s) of the {workload} workload{whole}, their top-{d.k} "
                             f"experts{shared}, full layer in float64 numpy, {dt:.2f} s"}

    # per forward: prep / quant-scatter / SwiGLU / combine (T <= 128) or route, histogram,
    # scan, permute, quant-scatter, plan, SwiGLU, combine; per GEMM one launch per
    # variant a group of up to T rows can need (small, medium > 16, mid > 64, large > 128)
    gemm_variants = 1 + (d.T > 16) + (d.T > 64) + (d.T > 128)
    launches_per_step = (4 if d.T <= 128 else 8) + 2 * gemm_variants
    rec = {
        "workload": workload, "d": d, "value": world * d.T / (ms_max * 1e-3),
        "ms_per_step": ms_max, "steps": steps, "warmup": warmup,
        "config": {"workload": workload, "T": d.T, "H": d.H, "I": d.I, "E": d.E, "k": d.k,
                   "shared_experts": d.has_shared, "weights": fmt, "active_groups": groups,
                   "routed_rows": d.R, "l2": l2_note, "parallelism": f"replicas x{world}",
                   "options": sorted(layer_opts) or None},
        "roofline": roof13, "roofline_w2": roof2, "stage_ms": stage_mean,
        "stream_ms_per_step": stream_step_ms, "ms_per_step_l2_write_flushed": flushed_ms,
        "ms_per_step_percentiles": pct,
        "weight_gbs": groups * 3 * d.I * d.H * WEIGHT_BYTES[fmt] /
                      ((stage_mean["gemm_w13"] + stage_mean["gemm_w2"]) * 1e-3) / 1e9,
        "gemm_tflops": 2.0 * (d.R + (d.T if d.has_shared else 0)) * 3 * d.I * d.H /
                       ((stage_mean["gemm_w13"] + stage_mean["gemm_w2"]) * 1e-3) / 1e12,
        "router_gate": router_rec, "cpu_baseline": cpu_rec, "e2e": e2e,
        "gpu_launches": 2 * launches_per_step * steps,
        "clocks": clocks.summary(tag),
        "options": opt_rec or None,
        "plan_tuning": tune_rec,
    }
    del graph, layer, t, x, lg, out, ws, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def measure_e2e(layer, d, x, lg, out, steps, do_flush, flush, world):
    """The same layer end to end through the public API from and to pinned host
    buffers, copies inside the timed region."""
    # single step, serialised: one graph replay = two copies in, the layer, one out
    hg = layer.host_graph(d.T)  # pinned host buffers, one graph launch per step
    hg.x_host.copy_(x.cpu())
    hg.logits_host.copy_(lg.cpu())
    for _ in range(3):
        hg.replay()
    torch.cuda.synchronize()
    e_ms = []
    for i in range(steps):
        if do_flush:
            flush.fill_(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        hg.replay()  # copies in, the layer, copy out
        torch.cuda.synchronize()
        e_ms.append((time.perf_counter() - t0) * 1e3)
    layer.forward(x, lg, out=out)
    torch.cuda.synchronize()
    out_ref = out.cpu()
    if not torch.equal(hg.out_host, out_ref):
        raise RuntimeError("host-buffer forward differs from the device forward")
    xh, lgh, oh = hg.x_host, hg.logits_host, hg.out_host
    single_ms = max_over_ranks(statistics.mean(e_ms), world)
    e2e = {"h2d_bytes_per_step": int(xh.numel() * 2 + lgh.numel() * 4),
           "d2h_bytes_per_step": int(oh.numel() * 2), "single_step_ms": single_ms}
    del hg
    if do_flush:
        # L2 flushed between steps: steps cannot overlap, the serialised form stands
        e2e.update(value=world * d.T / (single_ms * 1e-3), unit="tokens/s",
                   ms_per_step=single_ms, steps=steps,
                   api="MoELayer.host_graph(T).replay(): moe_forward_host captured as "
                       "one CUDA graph over pinned host buffers, one step at a time")
        return e2e
    # steps through the native host-buffer pipeline: step i's copies overlap the
    # kernels of steps i-1 and i+1; every step still copies its inputs in and its output
    # out; the first copy-in and last copy-out are in the time
    depth = 2
    pipe = layer.host_pipeline(d.T, depth)
    pxh = [xh.clone().pin_memory() for _ in range(depth)]
    plh = [lgh.clone().pin_memory() for _ in range(depth)]
    poh = [torch.empty_like(oh).pin_memory() for _ in range(depth)]
    for i in range(2 * depth):
        pipe.submit(pxh[i % depth], plh[i % depth], poh[i % depth])
    pipe.sync()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        pipe.submit(pxh[i % depth], plh[i % depth], poh[i % depth])
    pipe.sync()
    pipe_ms = (time.perf_counter() - t0) * 1e3 / steps
    for j in range(depth):
        if not torch.equal(poh[j], out_ref):
            raise RuntimeError("pipelined host-buffer forward differs from the device forward")
    pipe.close()
    em = max_over_ranks(pipe_ms, world)
    e2e.update(value=world * d.T / (em * 1e-3), unit="tokens/s", ms_per_step=em, steps=steps,
               api=f"MoELayer.host_pipeline(T, depth={depth}).submit() x steps + sync(): "
                   "moe_host_pipeline_*, pinned host buffers, copies on their own streams "
                   "overlapping neighbouring steps' kernels")
    return e2e


def sub_record(rec):
    """The compact form of a workload's measurement carried inside the headline line."""
    keep = ("value", "ms_per_step", "steps", "config", "roofline", "roofline_w2", "stage_ms",
            "ms_per_step_l2_write_flushed", "ms_per_step_percentiles", "weight_gbs",
            "gemm_tflops", "router_gate", "e2e", "clocks", "options", "plan_tuning")
    out = {k: rec[k] for k in keep}
    out["unit"] = "tokens/s"
    return out


# Steps of the extra workloads the default run measures beside the headline line:
# enough that each timed region lasts >= 2 s (>= 10 clock samples at 200 ms).
EXTRA_STEPS = {"decode256": 600, "prefill": 60, "decode_nvfp4": 3000}
# token count from which the router timing uses the tensor-core projection (measured
# faster from ~256 tokens; the fp32 GEMV wins for decode-sized batches)
ROUTER_TC_MIN_T = 256
EXTRA_E2E_STEPS = {"decode256": 50, "prefill": 20}
# moe_forward_ex options timed beside the default layer (decode, decode256, prefill)
OPTIONS = ("fuse_swiglu", "fuse_combine", "pair_tiles")


def run_ours(args, rank, world, local):
    import moe_expert_ffn_scan_gb300 as moe
    moe.lib()
    clocks = ClockSampler(local)
    with clocks:
        head = measure_layer(args, args.workload, args.steps, args.warmup, rank, world, local,
                             clocks, soak_s=2.5, e2e_steps=None if args.no_e2e else args.steps,
                             router=True, cpu=not args.no_cpu_baseline, fmt=args.weights,
                             options=() if (args.no_extra or args.options) else OPTIONS)
        extras = {}
        sweep = None
        if args.workload == "decode" and args.weights == "mxfp4" and not args.no_extra \
                and args.experts is None and args.tokens is None and not args.options:
            for wl in ("decode256", "prefill"):
                extras[wl] = sub_record(measure_layer(
                    args, wl, EXTRA_STEPS[wl], args.warmup, rank, world, local, clocks,
                    e2e_steps=None if args.no_e2e else EXTRA_E2E_STEPS[wl],
                    router=(wl == "prefill"), options=OPTIONS, tune=True))
            # the decode layer again with NVFP4 expert weights (f3)
            extras["decode_nvfp4"] = sub_record(measure_layer(
                args, "decode", EXTRA_STEPS["decode_nvfp4"], args.warmup, rank, world, local,
                clocks, fmt="nvfp4", tag="decode_nvfp4"))
            with clocks.load("sweep"):
                pts = sweep_points(args, local, steps=5, warmup=3)
            sweep = {"points": [{"gemm": p_["gemm"], "M": p_["M"], "ms": p_["ms"],
                                 "bound": "hbm" if p_["hbm_frac"] >= p_["tensor_frac"]
                                 else "tensor", "frac": p_["roofline_frac"]} for p_ in pts],
                     "steps_per_point": 5, "l2": "flushed before each call",
                     "clocks": clocks.summary("sweep")}
    if rank == 0:
        d = head["d"]
        clk = head["clocks"]
        clk["window"] = ("the timed region and 2.5 s of back-to-back replays of the same "
                         "step graph right before it")
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "mxfp4xfp8->f32" if args.weights == "mxfp4" else "nvfp4xfp8(bf16 mma)->f32",
            "data": "synthetic",
            "config": head["config"],
            "roofline": head["roofline"],
            "roofline_w2": head["roofline_w2"],
            "stage_ms": head["stage_ms"],
            "stream_ms_per_step": head["stream_ms_per_step"],
            "ms_per_step_l2_write_flushed": head["ms_per_step_l2_write_flushed"],
            "ms_per_step_percentiles": head["ms_per_step_percentiles"],
            "weight_gbs": head["weight_gbs"],
            "gemm_tflops": head["gemm_tflops"],
            "router_gate": head["router_gate"],
            "cpu_baseline": head["cpu_baseline"],
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "clocks": clk,
            "options": head["options"],
        }
        if extras:
            line["workloads"] = extras
        if sweep:
            line["sweep"] = sweep
        print(json.dumps(line), flush=True)


def sweep_points(args, local, steps, warmup, ms=None):
    """Grouped-GEMM shape sweep points: W13 (N=6144, K=7168) and W2 (N=7168, K=3072), G
    groups of M rows each (G*M ~ 32768 for M >= 64, else G = 64).  Activations bf16
    N(0,1), quantised by the library's FP8 quantiser; L2 flushed before each call."""
    import moe_expert_ffn_scan_gb300 as moe
    dev = torch.device("cuda", local)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    hbm, _ = hbm_peak_gbs()
    tpk, _ = fp8_tensor_peak_tflops()
    points = []
    for which in ("w13", "w2"):
        N, K = gi.SWEEP_SHAPES[which]
        for M in (ms or gi.SWEEP_M):
            x, offsets, w, ws_ = gi.sweep_point(which, M, seed=args.seed, device=dev)
            rows, G = x.shape[0], offsets.numel() - 1
            q = torch.empty(rows, K, dtype=torch.uint8, device=dev)
            qs = torch.empty(rows, K // 128, dtype=torch.uint8, device=dev)
            moe.moe_quant_act(x, q, qs)
            del x
            y = torch.empty(rows, N, dtype=torch.bfloat16, device=dev)
            if which == "w13":
                d = moe.dims(rows, K, N // 2, G, 1, 0)
            else:
                d = moe.dims(rows, N, K, G, 1, 0)
            wsp = moe.alloc_workspace(moe.gemm_workspace_size(d), dev)

            def call():
                if which == "w13":
                    moe.moe_grouped_gemm_w13(d, q, qs, None, offsets, w, ws_, y, wsp)
                else:
                    moe.moe_grouped_gemm_w2(d, q, qs, offsets, w, ws_, y, wsp)
            for _ in range(warmup):
                call()
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]
            for i in range(steps):
                flush.fill_(i & 0xFF)
                evs[i][0].record()
                call()
                evs[i][1].record()
            torch.cuda.synchronize()
            bits = moe.moe_check_status(wsp)
            if bits:
                raise RuntimeError(f"device status bits {bits:#x}")
            ms_ = statistics.median(a.elapsed_time(b) for a, b in evs)
            wbytes = G * N * K * WEIGHT_BYTES_PER_ELEM
            flops = 2.0 * rows * N * K
            gbs = wbytes / (ms_ * 1e-3) / 1e9
            tfl = flops / (ms_ * 1e-3) / 1e12
            points.append({"gemm": which, "M": M, "G": G, "ms": ms_, "weight_gbs": gbs,
                           "tflops": tfl, "hbm_frac": gbs / hbm, "tensor_frac": tfl / tpk,
                           "roofline_frac": max(gbs / hbm, tfl / tpk)})
            del q, qs, y, w, ws_, wsp
            torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return points


def run_gemm_point(args, rank, world, local):
    """One grouped GEMM of the sweep shapes (--gemm, --groups G, --rows M, --weights):
    the W13 or W2 call alone, L2 flushed before each call; for ncu captures of one
    kernel variant."""
    import moe_expert_ffn_scan_gb300 as moe
    moe.lib()
    dev = torch.device("cuda", local)
    which, G, M, fmt = args.gemm, args.groups, args.rows, args.weights
    N, K = gi.SWEEP_SHAPES[which]
    x, offsets, w, ws_ = gi.sweep_point(which, M, seed=args.seed, device=dev, G=G)
    rows = x.shape[0]
    q = torch.empty(rows, K, dtype=torch.uint8, device=dev)
    qs = torch.empty(rows, K // 128, dtype=torch.uint8, device=dev)
    moe.moe_quant_act(x, q, qs)
    y = torch.empty(rows, N, dtype=torch.bfloat16, device=dev)
    d = moe.dims(rows, K, N // 2, G, 1, 0) if which == "w13" else moe.dims(rows, N, K, G, 1, 0)
    if fmt == "nvfp4":
        w, wsn, gs = gi.nvfp4_weights(G, N, K, args.seed, dev,
                                      segments=2 if which == "w13" else 1)
        wsp = moe.alloc_workspace(moe.gemm_workspace_size_nvfp4(d), dev)

        def call():
            if which == "w13":
                moe.moe_grouped_gemm_w13_nvfp4(d, q, qs, None, offsets, w, wsn, gs, y, wsp)
            else:
                moe.moe_grouped_gemm_w2_nvfp4(d, q, qs, offsets, w, wsn, gs.reshape(-1), y, wsp)
    else:
        wsp = moe.alloc_workspace(moe.gemm_workspace_size(d), dev)

        def call():
            if which == "w13":
                moe.moe_grouped_gemm_w13(d, q, qs, None, offsets, w, ws_, y, wsp)
            else:
                moe.moe_grouped_gemm_w2(d, q, qs, offsets, w, ws_, y, wsp)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record()
        call()
        evs[i][1].record()
    torch.cuda.synchronize()
    bits = moe.moe_check_status(wsp)
    if bits:
        raise RuntimeError(f"device status bits {bits:#x}")
    ms_ = statistics.median(a.elapsed_time(b) for a, b in evs) if evs else 0.0
    wbytes = G * N * K * WEIGHT_BYTES[fmt]
    if rank == 0:
        hbm, hbm_src = hbm_peak_gbs()
        print(json.dumps({
            "metric": "grouped-GEMM weight GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms": ms_, "unit": "GB/s",
            "value": wbytes / (ms_ * 1e-3) / 1e9 if ms_ else None,
            "hbm_frac": wbytes / (ms_ * 1e-3) / 1e9 / hbm if ms_ else None,
            "hbm_peak_source": hbm_src, "tflops": 2.0 * rows * N * K / (ms_ * 1e-3) / 1e12
            if ms_ else None, "data": "synthetic",
            "config": {"workload": "gemm", "gemm": which, "groups": G, "rows_per_group": M,
                       "N": N, "K": K, "weights": fmt, "l2": "flushed before each call"}}),
            flush=True)


def run_sweep(args, rank, world, local):
    """The grouped-GEMM sweep on its own: one JSON line with every point."""
    import moe_expert_ffn_scan_gb300 as moe
    moe.lib()
    hbm, hbm_src = hbm_peak_gbs()
    tpk, tpk_src = fp8_tensor_peak_tflops()
    points = sweep_points(args, local, args.steps, args.warmup)
    if rank == 0:
        line = {"metric": "grouped-GEMM sweep (weight GB/s, TFLOP/s per M)",
                "value": statistics.mean(p["roofline_frac"] for p in points),
                "unit": "mean roofline fraction", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "higher_is_better": True, "data": "synthetic",
                "dtype": "mxfp4xfp8->f32",
                "config": {"workload": "sweep", "l2": "flushed before each call",
                           "hbm_peak_gbs": hbm, "hbm_peak_source": hbm_src,
                           "fp8_peak_tflops": tpk, "fp8_peak_source": tpk_src},
                "points": points}
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_init(args)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.workload == "sweep":
            run_sweep(args, rank, world, local)
        elif args.workload == "gemm":
            run_gemm_point(args, rank, world, local)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
