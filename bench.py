#!/usr/bin/env python
"""Throughput of one routed MoE layer forward on GB300 (routed tokens/s).

A step is one moe_forward (route -> dispatch -> grouped expert FFN ->
combine) over one batch of synthetic tokens already resident in HBM. The
default workload is the largest layer that fits one GPU: the fine-grained
skewed layer (T=16384, d=7168, E=256, top-8, f=2048, bf16, Zipf(1.1) expert
popularity). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

`value` comes from K steps of moe_forward bracketed by two CUDA events and
nothing else in between: the layer's kernels use programmatic dependent
launch, and an event recorded between two kernels stops the next one from
being scheduled early. Per-kernel times (the `kernels` table and the roofline
`achieved`) come from a second pass of K steps right after it, with events
at every kernel boundary (moe_forward_with_events) on the launching stream.
The per-step working set
(expert weights, 15 GB for the default layer) is larger than the 129 MB L2,
so no L2 flush is needed between steps; --flush-l2 adds one anyway.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed tokens/s per MoE layer fwd at 1 GB300"
UNIT = "tokens/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the moe_forward_with_events slots; "w1_prologue" runs no kernel (the FP8
# payload is expanded to bf16 inside the W1 GEMM) and is left out of the table
STAGES = ["route", "dispatch", "w1_prologue", "gemm_w1_silu", "gemm_w2", "quantize_out",
          "combine"]


def parse():
    from workloads import CONFIG_ORDER, VARIANTS
    p = argparse.ArgumentParser(
        description="Routed tokens/s of one MoE layer forward: one JSON line on rank 0.")
    p.add_argument("--gpus", type=int, default=1,
                   help="replicas, one process per GPU (launched by torch.distributed.run)")
    p.add_argument("--steps", type=int, default=20, help="timed forwards")
    p.add_argument("--warmup", type=int, default=5, help="untimed forwards first (at least 3)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"],
                   help="ours: the CUDA library; reference: the fp64 CPU oracle")
    p.add_argument("--config", default=None,
                   help="layer name (default: the 256-expert layer); one of "
                   + ", ".join(list(CONFIG_ORDER) + list(VARIANTS)))
    p.add_argument("--flush-l2", action="store_true",
                   help="write a buffer twice the L2 before every timed forward")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle timing")
    p.add_argument("--no-e2e", action="store_true",
                   help="skip the end-to-end timing with host buffers")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="CPU oracle baseline: run 16-token chunks until this much time has passed")
    p.add_argument("--backward", action="store_true",
                   help="also time moe_backward (adds a 'backward' object to the line): after "
                        "a forward that keeps the pre-activation Z (keep_z, timed too), or, "
                        "with --recompute-z, after the plain forward, recomputing Z")
    p.add_argument("--recompute-z", action="store_true",
                   help="with --backward: the backward recomputes Z instead of reading it")
    p.add_argument("--x-perm-mode", type=int, default=None, choices=[0, 1, 2],
                   help="0 the library's choice, 1 packed rows, 2 rows gathered by the W1 GEMM")
    p.add_argument("--gemm-tile-n", type=int, default=None, choices=[0, 256, 512],
                   help="expert GEMM pair-tile width (0: the library's choice)")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {k: d[k] for k in PEAKS_FALLBACK}, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ---------------------------------------------------------------- algorithmic work
def stage_work(cfg, counts, gathered=False):
    """Algorithmic bytes and flops per launch of each stage: only what the
    method must move (weights of experts that received rows, each operand
    read once, each result written once). `gathered`: the W1 GEMM reads each
    routed row from x itself and the dispatch writes only the layout."""
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    R = T * k
    b = 4 if cfg.dtype == "f32" else 2
    pb = 1 if cfg.payload_fp8 else b
    active = sum(1 for c in counts if c > 0)
    w = {}
    soft = getattr(cfg, "router", 0) == 3
    # soft gating also reads its Gumbel samples; its dispatch writes only the
    # layout, and its W1 GEMM reads x itself (once per expert from L2: x once
    # from HBM)
    w["route"] = (T * d * b + d * E * b + E * 4 + R * 8 + (T * E * 4 if soft else 0),
                  2.0 * T * d * E)
    # soft gating: the layout only; gathered rows: ids read, the layout written
    w["dispatch"] = ((R * 8 + E * 8) if soft else (R * 12 + E * 8) if gathered else
                     (T * d * b + R * d * pb + R * 12 + (R * 4 if cfg.payload_fp8 else 0)), 0.0)
    w["w1_prologue"] = (0, 0.0)
    a_bytes = T * d * b if soft else R * d * pb
    w["gemm_w1_silu"] = (active * d * f * b + a_bytes + R * f * b, 2.0 * R * d * f)
    w["gemm_w2"] = (active * f * d * b + R * f * b + R * d * 4, 2.0 * R * f * d)
    ofp8 = getattr(cfg, "output_fp8", 0)
    # FP8 expert outputs: read Y once, write the E4M3 rows, scale and zero
    w["quantize_out"] = ((R * d * 4 + R * d + R * 8) if ofp8 else 0, 0.0)
    w["combine"] = (R * d * (1 if ofp8 else 4) + R * 8 + (R * 8 if ofp8 else 0) + T * d * b,
                    2.0 * R * d)
    return w


def source_sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def ncu_traffic(workload_stage):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current source of the kernel (the entry names its file and hash);
    else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        ent = json.load(open(path)).get(workload_stage)
        if not ent:
            return None
        src = os.path.join(ROOT, "mixture_experts_routed_gb300", "csrc", ent["file"])
        if os.path.exists(src) and ent.get("source_sha") == source_sha(src):
            return ent.get("dram_bytes_per_launch")
    except Exception:
        return None
    return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi every 100 ms, each sample time-stamped; the summary keeps
    the samples inside the window the caller marks (the GPU-busy steps)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 100

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def mark(self, t0, t1):
        """The busy window, host wall-clock datetimes."""
        self.window = (t0, t1)

    @staticmethod
    def _summary(rows):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for parts in rows:
            try:
                sm.append(float(parts[2]))
                mx = float(parts[3])
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        import datetime
        rows, inside = [], []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            rows.append(parts)
            if self.window is not None:
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                except ValueError:
                    continue
                if self.window[0] <= ts <= self.window[1]:
                    inside.append(parts)
        out = self._summary(inside)
        if out is not None:
            out["window"] = "samples taken while the timed steps and the per-kernel pass ran"
            out["window_ms"] = round((self.window[1] - self.window[0]).total_seconds() * 1e3, 1)
            return out
        out = self._summary(rows)
        if out is not None:
            out["window"] = ("no sample fell inside the busy window; every sample of the run "
                             "(before, during and after the timed steps)")
        return out


# ---------------------------------------------------------------- CPU oracle timing
def cpu_oracle_run(cfg, host, tokens):
    import oracle
    t0 = time.perf_counter()
    oracle.forward_tokens(cfg, host, tokens)
    return time.perf_counter() - t0


def host_inputs(inp):
    """The oracle's host inputs (outside any timed region): fp64 arrays of x,
    W_g, bias (and the Gumbel samples), CPU copies of the expert weights,
    which the oracle upcasts one expert at a time."""
    import oracle
    return oracle.inputs_to_numpy({k: v.detach().cpu() for k, v in inp.items()})


def cpu_oracle_sample(cfg, host, seconds, chunk=16):
    """The oracle over consecutive chunks of `chunk` tokens from token 0 until
    `seconds` have passed (or the batch is done): (tokens, wall seconds)."""
    done, t = 0, 0.0
    while done < cfg.T and (done == 0 or t < seconds):
        n = min(chunk, cfg.T - done)
        t += cpu_oracle_run(cfg, host, list(range(done, done + n)))
        done += n
    return done, t


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- ranks
def max_over_ranks(value, dist, device):
    """The largest of every rank's value (a replicated job is as slow as its
    slowest rank); on one process (dist None) the value itself."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def error_on_any_rank(bad, dist, device):
    """True on every rank when any rank saw a device error (a collective, so
    that all ranks raise together and none is left waiting in the next one)."""
    return max_over_ranks(1.0 if bad else 0.0, dist, device) > 0.0


# ---------------------------------------------------------------- reference arm
def reference_sample_tokens(cfg):
    """Tokens the reference arm runs per step: about 128 routed rows, so that
    one step stays around a second or two of host work even on the layers
    whose oracle upcasts many experts' weights."""
    return max(1, min(cfg.T, 128 // cfg.k))


def run_reference(args, cfg):
    import numpy as np
    import torch
    from workloads import make_inputs
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # the draws are made on the GPU when there is one (the CPU generator takes
    # minutes for the 15 GB of expert weights) and copied to host memory; the
    # oracle itself runs on the host cores only
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(cfg, device=gen_dev)
    host = host_inputs(inp)
    del inp
    if gen_dev == "cuda":
        torch.cuda.empty_cache()
    S = reference_sample_tokens(cfg)
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        cpu_oracle_run(cfg, host, np.sort(rng.choice(cfg.T, S, replace=False)))
    t = 0.0
    for _ in range(args.steps):
        t += cpu_oracle_run(cfg, host, np.sort(rng.choice(cfg.T, S, replace=False)))
    per_step = t / args.steps
    value = S / per_step
    sample = (f"{S} random tokens of the {cfg.T}-token batch per step: gate, router, the FFN "
              f"of every chosen expert (its weights upcast to fp64 as the oracle does) and the "
              f"combine, numpy fp64; inputs drawn on {gen_dev}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg, args):
    router = {0: "renorm", 1: "prek_softmax",
              2: f"group_limited(n_group={cfg.n_group}, topk_group={cfg.topk_group})",
              3: f"soft_gumbel(tau={cfg.tau:g}), all {cfg.E} experts"}
    payload = {0: cfg.dtype, 1: "fp8_e4m3 (per-token absmax scale)",
               2: f"fp8_e4m3 (static scale {cfg.payload_scale:.6g})"}
    return {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "f": cfg.f,
            "router": router[cfg.router], "pre_k": cfg.pre_k,
            "payload": payload[int(cfg.payload_fp8)],
            "x_perm_mode": {0: "library's choice", 1: "packed", 2: "gathered"}[cfg.x_perm_mode],
            "gemm_tile_n": cfg.gemm_tile_n or "library's choice",
            "expert_output": ("fp8_e4m3 (per-row min/max affine)" if cfg.output_fp8
                              else "fp32"), "seed": cfg.seed,
            "parallelism": f"replicas x{args.gpus}",
            "l2": ("flushed between steps" if args.flush_l2 else
                   "not flushed: per-step working set (expert weights) exceeds the 129 MB L2")}


# ---------------------------------------------------------------- our arm
def run_ours(args, cfg):
    import numpy as np
    import torch
    import mixture_experts_routed_gb300 as moe
    from mixture_experts_routed_gb300.stats import load_stats
    from workloads import make_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    inp = make_inputs(cfg, device=dev)
    ws = moe.alloc_workspace(cfg, device=dev)
    out = torch.empty((cfg.T, cfg.d), dtype=cfg.torch_dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = None
    if args.flush_l2:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def step(events=None):
        if flush is not None:
            flush.fill_(1)
        moe.forward(cfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws,
                    out=out, events=events, noise=inp.get("gumbel"), stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if error_on_any_rank(moe.get_device_error(ws) != moe.MOE_OK, dist, dev):
        raise RuntimeError("device error during warm-up")

    # ---- timed region: K steps, no event between kernels
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_NUM_EVENTS)]
           for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if world == 1 else local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    import datetime
    busy_from = datetime.datetime.now()
    t_start.record(stream)
    for i in range(K):
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    # ---- per-kernel pass: K more steps with events at every kernel boundary
    for i in range(K):
        step(evs[i])
    torch.cuda.synchronize(dev)
    clocks.mark(busy_from, datetime.datetime.now())
    clk = clocks.stop() if rank == 0 else None
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    if error_on_any_rank(moe.get_device_error(ws) != moe.MOE_OK, dist, dev):
        raise RuntimeError("device error in the timed steps")
    ms_per_step = total_ms / K
    value = cfg.T * world / (ms_per_step / 1e3)

    # per-kernel averages (event i -> i+1 brackets one stage)
    stage_ms = {}
    for si, name in enumerate(STAGES):
        stage_ms[name] = sum(evs[i][si].elapsed_time(evs[i][si + 1]) for i in range(K)) / K

    views = moe.forward_views(cfg, ws)
    counts = views["counts"].cpu().tolist()
    gathered = views["x_perm"] is None and cfg.router != 3
    work = stage_work(cfg, counts, gathered)
    peaks, peak_src = load_peaks()
    kernels = {}
    for name in STAGES:
        by, fl = work[name]
        t = stage_ms[name] / 1e3
        if by == 0 and fl == 0:
            continue
        gbs = by / t / 1e9 if t > 0 else 0.0
        tfl = fl / t / 1e12 if t > 0 else 0.0
        kernels[name] = {"us": stage_ms[name] * 1e3, "bytes": by, "flops": fl, "GB_s": gbs,
                         "TFLOP_s": tfl, "hbm_frac": gbs / peaks["hbm_gbs"],
                         "tensor_frac": (tfl / peaks["bf16_tflops"]) if name.startswith("gemm")
                         else None,
                         "tensor_frac_sustained": (tfl / peaks["bf16_tflops_sustained"])
                         if name.startswith("gemm") else None}
    dom = max(kernels, key=lambda n: kernels[n]["us"])
    kd = kernels[dom]
    by, fl = work[dom]
    is_tensor = dom.startswith("gemm") and cfg.dtype == "bf16" and \
        fl / (peaks["bf16_tflops"] * 1e12) > by / (peaks["hbm_gbs"] * 1e9)
    traffic = ncu_traffic(f"{cfg.name}:{dom}")
    if is_tensor:
        # the dominant GEMM runs inside K back-to-back forwards: when the
        # power cap engaged during them, the peak it can reach is the
        # sustained one (measured under the cap), else the burst one
        capped = bool(clk) and "sw_power_cap" in clk.get("reasons", [])
        tpeak = peaks["bf16_tflops_sustained"] if capped else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": kd["TFLOP_s"], "peak": tpeak,
                "unit": "TFLOP/s", "frac": kd["TFLOP_s"] / tpeak,
                "frac_of_burst_peak": kd["TFLOP_s"] / peaks["bf16_tflops"],
                "traffic": traffic,
                "peak_source": f"{peak_src} bf16, " + (
                    "sustained (sw_power_cap active during the timed steps)" if capped
                    else "burst")}
    else:
        roof = {"bound": "hbm", "achieved": kd["GB_s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": kd["GB_s"] / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": f"{peak_src} HBM copy"}
    roof["kernel"] = dom
    roof["algorithmic_bytes"] = by
    roof["algorithmic_flops"] = fl

    # ---- end to end through the public API with host buffers. Every step
    # copies its batch (x, and soft gating's Gumbel samples) from pinned
    # host memory to the GPU, runs moe_forward and copies the output back.
    # The copies run on their own streams with double-buffered device
    # tensors, so step i + 1's upload and step i - 1's download overlap
    # step i's forward (a streaming caller's pipeline); the timed region
    # runs from before the first upload to after the last download.
    e2e = None
    if not args.no_e2e:
        x_host = inp["x"].cpu().pin_memory()
        # soft gating's Gumbel samples are a per-step input too
        g_host = inp["gumbel"].cpu().pin_memory() if "gumbel" in inp else None
        nb = 2
        x_dev = [torch.empty_like(inp["x"]) for _ in range(nb)]
        g_dev = [torch.empty_like(inp["gumbel"]) if g_host is not None else None
                 for _ in range(nb)]
        o_dev = [torch.empty((cfg.T, cfg.d), dtype=cfg.torch_dtype, device=dev)
                 for _ in range(nb)]
        o_host = [torch.empty((cfg.T, cfg.d), dtype=cfg.torch_dtype).pin_memory()
                  for _ in range(nb)]
        up = torch.cuda.Stream(dev)
        down = torch.cuda.Stream(dev)
        ev_up = [torch.cuda.Event() for _ in range(nb)]
        ev_fwd = [torch.cuda.Event() for _ in range(nb)]
        ev_down = [torch.cuda.Event() for _ in range(nb)]

        def e2e_step(i, m=None):
            b = i % nb
            # upload into buffer b once the forward two steps back has read it
            if i >= nb:
                up.wait_event(ev_fwd[b])
            with torch.cuda.stream(up):
                if m is not None:
                    m[0].record(up)
                x_dev[b].copy_(x_host, non_blocking=True)
                if g_host is not None:
                    g_dev[b].copy_(g_host, non_blocking=True)
                if m is not None:
                    m[1].record(up)
                ev_up[b].record(up)
            stream.wait_event(ev_up[b])
            if i >= nb:
                stream.wait_event(ev_down[b])   # o_dev[b] downloaded two steps back
            moe.forward(cfg, x_dev[b], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], ws=ws,
                        out=o_dev[b], noise=g_dev[b], stream=stream)
            ev_fwd[b].record(stream)
            down.wait_event(ev_fwd[b])
            with torch.cuda.stream(down):
                if m is not None:
                    m[2].record(down)
                o_host[b].copy_(o_dev[b], non_blocking=True)
                if m is not None:
                    m[3].record(down)
                ev_down[b].record(down)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b_ev = torch.cuda.Event(enable_timing=True)
        # copy start / end events of every timed step (the copy streams'
        # own time, so a slow host link shows in the line)
        cp = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        a.record(stream)
        up.wait_event(a)
        for i in range(K):
            e2e_step(i, cp[i])
        stream.wait_event(ev_down[(K - 1) % nb])
        b_ev.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(a.elapsed_time(b_ev), dist, dev)
        h2d_ms = sum(m[0].elapsed_time(m[1]) for m in cp) / K
        d2h_ms = sum(m[2].elapsed_time(m[3]) for m in cp) / K
        e2e = {"value": cfg.T * world / (e_ms / K / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": x_host.numel() * x_host.element_size() + (
                   g_host.numel() * g_host.element_size() if g_host is not None else 0),
               "d2h_bytes_per_step": o_host[0].numel() * o_host[0].element_size(),
               "h2d_ms_per_step": h2d_ms, "d2h_ms_per_step": d2h_ms,
               "pipelining": "uploads and downloads on two copy streams, double-buffered, "
                             "overlapping the neighbouring steps' forwards"}

    # ---- backward (optional): K steps of moe_backward after the forward above
    bwd = None
    if args.backward and not (cfg.payload_fp8 or getattr(cfg, "output_fp8", 0)):
        # training form: the forward keeps Z (keep_z) and the backward reads
        # it; --recompute-z: the plain forward, the backward recomputes Z
        kept = not args.recompute_z
        bcfg = cfg.with_(keep_z=1) if kept else cfg
        fws = moe.alloc_workspace(bcfg) if kept else ws
        bws = moe.alloc_workspace(bcfg, "backward")
        gen = torch.Generator(device=dev)
        gen.manual_seed(5)
        dout = torch.randn((cfg.T, cfg.d), generator=gen, device=dev).to(cfg.torch_dtype)
        fwd_z_ms = None
        if kept:
            fout = torch.empty((cfg.T, cfg.d), dtype=cfg.torch_dtype, device=dev)

            def fwd_z_step():
                moe.forward(bcfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"],
                            ws=fws, out=fout, noise=inp.get("gumbel"), stream=stream)

            for _ in range(max(1, args.warmup)):
                fwd_z_step()
            torch.cuda.synchronize(dev)
            if dist:
                dist.barrier()
            fa = torch.cuda.Event(enable_timing=True)
            fb = torch.cuda.Event(enable_timing=True)
            fa.record(stream)
            for _ in range(K):
                fwd_z_step()
            fb.record(stream)
            torch.cuda.synchronize(dev)
            fwd_z_ms = max_over_ranks(fa.elapsed_time(fb), dist, dev) / K
            if error_on_any_rank(moe.get_device_error(fws) != moe.MOE_OK, dist, dev):
                raise RuntimeError("device error in the forward steps keeping Z")

        def bwd_step():
            moe.backward(bcfg, inp["x"], inp["Wg"], inp["bias"], inp["W1"], inp["W2"], dout,
                         fwd_ws=fws, ws=bws, noise=inp.get("gumbel"), stream=stream)

        for _ in range(max(1, args.warmup)):
            bwd_step()
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            bwd_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        b_ms = max_over_ranks(a.elapsed_time(b), dist, dev) / K
        if error_on_any_rank(moe.get_device_error(bws) != moe.MOE_OK, dist, dev):
            raise RuntimeError("device error in the backward steps")
        R = cfg.T * cfg.k
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        gate = 4.0 * cfg.T * cfg.d * cfg.E  # dx_gate and dW_g (fp32 FMA)
        # Z = X W1 is one 2Rdf GEMM of the backward unless the forward kept it
        nz = 0.0 if kept else 2.0
        if cfg.dtype == "f32":
            # every GEMM in fp32 FMA: (Z,) dH, dX_perm, dW2, dW1 and the gate's
            simt = (8.0 + nz) * R * cfg.d * cfg.f + gate
            # fp32 FMA peak from unit counts: SMs x 128 fp32 lanes x 2 flop x clock
            fp32_peak = sms * 128 * 2 * (clk or {}).get("sm_max_mhz", 2070.0) * 1e6 / 1e12
            broof = {"bound": "alu", "achieved": simt / (b_ms / 1e3) / 1e12, "peak": fp32_peak,
                    "unit": "TFLOP/s", "frac": simt / (b_ms / 1e3) / 1e12 / fp32_peak,
                    "peak_source": "derived: SMs x 128 fp32 FMA lanes x 2 x max SM clock",
                    "flops": simt}
            note = "achieved = every GEMM's fp32 FMA work over the whole backward time"
        else:
            # the method's own work: four expert GEMMs (and Z, when it is
            # recomputed), 2Rdf each. The tensor cores execute more: each of
            # the three GEMMs with an fp32 operand (dY or w H for dW2, dZ for
            # dX_perm and dW1) runs on its bf16 split hi + lo, which doubles
            # it; dH reads the bf16 dout rows with the routing weight applied
            # after the sum (14Rdf executed, 16Rdf with Z recomputed)
            algo = (8.0 + nz) * R * cfg.d * cfg.f
            executed = (14.0 + nz) * R * cfg.d * cfg.f
            t_s = b_ms / 1e3
            broof = {"bound": "tensor", "achieved": algo / t_s / 1e12,
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": algo / t_s / 1e12 / peaks["bf16_tflops"],
                    "peak_source": "measured bf16 (burst)", "flops": algo,
                    "executed_flops": executed,
                    "executed_tflops": executed / t_s / 1e12,
                    "executed_frac": executed / t_s / 1e12 / peaks["bf16_tflops"]}
            note = ("achieved = the method's expert-GEMM flops (" +
                    ("8 R d f: dH, dX_perm, dW1, dW2; Z kept by the forward" if kept else
                     "10 R d f: Z recomputed, dH, dX_perm, dW1, dW2") +
                    ") over the whole backward time; executed_* count the tensor-core flops "
                    "actually run (the hi/lo operand split doubles three GEMMs: " +
                    ("14" if kept else "16") + " R d f); the gate's fp32 FMA work is simt_flops")
        bwd = {"ms_per_step": b_ms, "tokens_per_s": cfg.T * world / (b_ms / 1e3),
               "z": "kept by the forward (keep_z)" if kept else "recomputed",
               "forward_keep_z_ms_per_step": fwd_z_ms,
               "training_step_ms": (fwd_z_ms + b_ms) if kept else (ms_per_step + b_ms),
               "roofline": broof, "simt_flops": gate if cfg.dtype != "f32" else None,
               "note": note}

    if dist:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return 0

    # ---- CPU oracle on a bounded sample (rank 0 only, N = 1 only)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        host = host_inputs(inp)
        S, t = cpu_oracle_sample(cfg, host, args.cpu_seconds)
        cpu = {"value": S / t, "unit": UNIT, "cores": cores(), "kind": "oracle",
               "sample": f"the first {S} tokens of the {cfg.T}-token batch in chunks of 16 "
                         f"(run until {args.cpu_seconds:g} s had passed), whole layer (gate, "
                         f"router, FFN of every chosen expert incl. its fp64 weight upcast, "
                         f"combine) in numpy fp64; {t:.1f} s"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
            "config": dict(workload_config(cfg, args),
                           rows=("x itself, read by every expert (soft gating)"
                                 if cfg.router == 3 else
                                 "gathered by the W1 GEMM from x (no packed copy)" if gathered
                                 else "packed by the dispatch")),
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": e2e, "gpu_launches": moe.kernel_count(cfg) * K, "clocks": clk,
            "kernel_times": "CUDA events at every kernel boundary, in a second pass of K steps "
                            "after the timed one (events between kernels would stop their "
                            "programmatic dependent launch)",
            "kernels": kernels, "grouped_gemm_tflops":
                (work["gemm_w1_silu"][1] + work["gemm_w2"][1]) /
                ((stage_ms["gemm_w1_silu"] + stage_ms["gemm_w2"]) / 1e3) / 1e12,
            "load": load_stats(counts), "peaks": peaks}
    if bwd is not None:
        line["backward"] = bwd
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    from workloads import get_config, BENCH_CONFIG
    cfg = get_config(args.config or BENCH_CONFIG)
    if args.x_perm_mode is not None:
        cfg = cfg.with_(x_perm_mode=args.x_perm_mode)
    if args.gemm_tile_n is not None:
        cfg = cfg.with_(gemm_tile_n=args.gemm_tile_n)
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
