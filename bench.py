"""Benchmark of the Interleaved Head Attention forward pass on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one pass of the whole hot path over one batch of synthetic input:
projection + pseudo-head mixing into the stacked layout (the library's route for the
shape: the head projections with the mixing in the GEMM epilogue, or fold alpha into W
then project) -> attention
over the stacked sequence -> R contraction, launched through the library's step
entry points on one stream, each kernel bracketed by CUDA events on that stream.
L2 is flushed (256 MiB write) between steps, outside the timed events.
Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica of the workload (weak scaling; the forward pass has no
cross-sample exchange), and the step time is the max over ranks.

--impl reference times the fp64 CPU oracle (the only other implementation of
the method: the pages ship no code) on the host cores, on a bounded sample of
the same workload, and prints the same JSON line with "impl": "reference".
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import iha_inputs as gi  # noqa: E402

METRIC = "IHA fwd pseudo-tokens/s and TFLOP/s (% of GB300 dense BF16 peak), 1 GPU"
UNIT = "pseudo-tokens/s"
DEFAULT_WORKLOAD = "bf16_causal_p4_n8192"
DATA = ("synthetic: seeded SplitMix64 + Box-Muller; X~N(0,1), W~N(0,1/D), alpha~N(0,1/H), "
        "R~N(0,1/(H*P)); random-init weights, bf16-rounded")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return dict(hbm=m["hbm_gbs"], bf16=m["bf16_tflops"], bf16_sustained=m["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------
# work accounting (algorithmic, per step)
# ---------------------------------------------------------------------------

def token_pairs(w) -> int:
    """Readable (query token, key token) pairs of one sequence under the mask."""
    N = w.N
    if w.mask_mode == gi.MASK_NONE:
        return N * N
    if w.mask_mode == gi.MASK_CAUSAL or w.window >= N:
        return N * (N + 1) // 2
    ww = w.window
    # sum_t min(t + 1, w)
    return ww * (ww + 1) // 2 + (N - ww) * ww


def work(w):
    B, N, H, d, P, D = w.B, w.N, w.H, w.d, w.P, w.D
    pairs = B * H * P * P * token_pairs(w)              # readable pseudo-token pairs
    attn = 4.0 * d * pairs                              # QK^T and PV, 2 flops per MAC
    proj_folded = 2.0 * B * N * D * (3 * H * P * d)     # executed GEMM
    proj_heads = 2.0 * B * N * D * 3 * D                # X W^(m), all heads, Q/K/V
    mixing = 2.0 * B * N * 3 * (H * P) * D              # sum over m of alpha * (X W^(m))
    contract = 2.0 * B * N * (H * P) * D                # R contraction
    es = 2
    bytes_contract = es * (B * N * H * P * d + B * N * D)
    bytes_fold = es * (3 * D * D + 3 * H * P * d * D)
    bytes_slice = es * 2 * 3 * D * D                            # read W_Q/W_K/W_V, write them slice-major
    return dict(pairs=pairs, attn=attn, proj_folded=proj_folded, proj_heads=proj_heads,
                algorithmic=proj_heads + mixing + attn + contract,
                executed_folded=proj_folded + attn + contract, executed_unfolded=proj_heads + mixing + attn + contract,
                bytes_contract=bytes_contract, bytes_fold=bytes_fold, bytes_slice=bytes_slice, pseudo_tokens=B * P * N)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_rows(w, n_tokens):
    """n_tokens query tokens of batch element 0, evenly spaced over [0, N), so the
    sample's average cost per token is the workload's."""
    n = min(n_tokens, w.N)
    toks = sorted({int(round((i + 0.5) * w.N / n)) for i in range(n)})
    return [t for t in toks if t < w.N]


def time_oracle(w, inp_f64, n_tokens):
    import oracle
    rows = oracle_sample_rows(w, n_tokens)
    f = inp_f64
    t0 = time.perf_counter()
    oracle.forward(f["X"][:1], f["W_Q"], f["W_K"], f["W_V"], f["alpha_Q"], f["alpha_K"], f["alpha_V"], f["R"],
                   H=w.H, d=w.d, P=w.P, mask_mode=w.mask_mode, window=w.window, rows=rows, projection="numpy")
    dt = time.perf_counter() - t0
    return w.P * len(rows) / dt, dt, len(rows)


def oracle_sample_desc(w, n):
    return (f"batch element 0, {n} query tokens evenly spaced over N={w.N} (all P={w.P} pseudo-rows each, "
            f"every head); projections of the tokens they read by float64 BLAS matmul, the rest in C")


# ---------------------------------------------------------------------------
# distributed setup (torchrun); every rank is an independent replica
# ---------------------------------------------------------------------------

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def max_over_ranks(x: float, dist, device):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, pseudo_tokens_per_rank: int, step_ms: float) -> float:
    """Whole-job throughput: every rank processes its own replica of the workload, so the
    job handles world x pseudo_tokens_per_rank per step of step_ms (max over ranks)."""
    return world * pseudo_tokens_per_rank / (step_ms * 1e-3)


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, w):
    rank, world, local, dist = dist_setup(args.gpus)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    import oracle
    oracle.build()
    f = gi.as_f64(gi.make_inputs(w))
    per_step_tokens = args.ref_tokens
    times, vals = [], []
    for i in range(args.warmup + args.steps):
        v, dt, n = time_oracle(w, f, per_step_tokens)
        if i >= args.warmup:
            times.append(dt)
            vals.append(v)
    value = w.P * n * len(times) / sum(times)
    cores = oracle.default_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": config_of(w, l2="host memory"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": oracle_sample_desc(w, n) + " per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def config_of(w, l2):
    return {"workload": w.name, "B": w.B, "N": w.N, "D": w.D, "H": w.H, "d": w.d, "P": w.P,
            "stacked_length": w.PN, "mask": ["none", "causal", "causal+window"][w.mask_mode],
            "window": w.window if w.mask_mode == gi.MASK_WINDOW else None, "l2": l2}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class ForwardStep:
    """One forward step of workload w through the library's step entry points, on one
    stream: the route's steps 1+2 (project heads then mix, or fold then project), the
    attention, the contraction; each kernel bracketed by CUDA events on that stream."""

    def __init__(self, iha, w, host, dev, stream):
        self.iha, self.w, self.dev, self.stream = iha, w, dev, stream
        self.dt = iha.IHA_DTYPE_BF16 if w.dtype == "bf16" else iha.IHA_DTYPE_F32
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.d = {k: v.to(dev).contiguous() for k, v in host.items()}
        self.route = iha.iha_projection_route(w.H, w.d, w.P, self.dt)
        if self.route == 1:   # slice-major weights
            self.Wt = torch.empty(iha.iha_sliced_weights_bytes(w.H, w.d, self.dt), dtype=torch.uint8, device=dev)
        else:                 # folded weights
            self.Wt = torch.empty(3 * w.H * w.P * w.d, w.D, dtype=tdt, device=dev)
        self.QKV = torch.empty(3, w.B, w.H, w.N * w.P, w.d, dtype=tdt, device=dev)
        self.Pbar = torch.empty(w.B, w.N, w.H, w.P, w.d, dtype=tdt, device=dev)
        self.out = torch.empty(w.B, w.N, w.D, dtype=tdt, device=dev)
        self.names = (["slice_weights", "project_mix", "attention", "contract"] if self.route == 1
                      else ["fold", "project", "attention", "contract"])

    def launches(self):
        iha, w, d, dt, s = self.iha, self.w, self.d, self.dt, self.stream
        if self.route == 1:
            yield lambda: iha.check(iha.iha_slice_weights(d["W_Q"], d["W_K"], d["W_V"], w.H, w.d, dt, self.Wt, s),
                                    "slice_weights")
            yield lambda: iha.check(iha.iha_project_mix(d["X"], self.Wt, d["alpha_Q"], d["alpha_K"], d["alpha_V"],
                                                        w.B, w.N, w.H, w.d, w.P, dt, self.QKV, s), "project_mix")
        else:
            yield lambda: iha.check(iha.iha_fold_weights(d["W_Q"], d["W_K"], d["W_V"], d["alpha_Q"], d["alpha_K"],
                                                         d["alpha_V"], w.H, w.d, w.P, dt, self.Wt, s), "fold")
            yield lambda: iha.check(iha.iha_project(d["X"], self.Wt, w.B, w.N, w.H, w.d, w.P, dt, self.QKV, s),
                                    "project")
        yield lambda: iha.check(iha.iha_attention(self.QKV, w.B, w.N, w.H, w.d, w.P, w.mask_mode, w.window, dt,
                                                  self.Pbar, s), "attention")
        yield lambda: iha.check(iha.iha_contract(self.Pbar, d["R"], w.B, w.N, w.H, w.d, w.P, dt, self.out, s),
                                "contract")

    def run(self, ev=None):
        for j, launch in enumerate(self.launches()):
            if ev is not None:
                ev[j].record(self.stream)
            launch()
        if ev is not None:
            ev[len(self.names)].record(self.stream)

    def time(self, steps, warmup, flush, dist=None, clocks=None):
        """Warm-up, then `steps` timed steps with L2 flushed between them (outside the events).
        Returns (mean step ms, {kernel: mean ms}, wall seconds of the timed region)."""
        iha, stream, dev = self.iha, self.stream, self.dev
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                flush.fill_(1)
                self.run()
        torch.cuda.synchronize(dev)
        rc, code = iha.iha_check_device_status(stream)
        iha.check(rc, f"device status after warm-up ({code:#x})")
        n = len(self.names)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
        barrier(dist)
        torch.cuda.synchronize(dev)
        with (clocks if clocks is not None else _NoClock()):
            t_wall0 = time.perf_counter()
            with torch.cuda.stream(stream):
                for i in range(steps):
                    flush.fill_(i & 0xFF)          # evict L2 between steps (outside the events)
                    self.run(events[i])
            torch.cuda.synchronize(dev)
            t_wall = time.perf_counter() - t_wall0
        barrier(dist)
        rc, code = iha.iha_check_device_status(stream)
        iha.check(rc, f"device status after timed steps ({code:#x})")
        k_ms = {nm: sum(ev[j].elapsed_time(ev[j + 1]) for ev in events) / steps for j, nm in enumerate(self.names)}
        step_ms = sum(ev[0].elapsed_time(ev[n]) for ev in events) / steps
        return step_ms, k_ms, t_wall


class _NoClock:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


# the other workloads of the target, timed in the same run (ms per step, kernel times and
# the attention kernel's fraction of peak), beside the headline workload's line
SIDE_WORKLOADS = ["bf16_causal_n1024", "bf16_window1024_n4096", "bf16_window4096_n16384"]


def side_workloads(iha, args, dev, stream, flush, peaks, skip):
    res = {}
    for name in SIDE_WORKLOADS:
        if name == skip:
            continue
        w = gi.WORKLOADS[name]
        fs = ForwardStep(iha, w, gi.make_inputs(w), dev, stream)
        ms, k_ms, _ = fs.time(args.steps, args.warmup, flush)
        wk = work(w)
        tf = wk["attn"] / (k_ms["attention"] * 1e-3) / 1e12
        res[name] = {"value": wk["pseudo_tokens"] / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "kernel_ms": k_ms,
                     "attention_tflops_exact_pairs": tf, "attention_frac": tf / peaks["bf16"],
                     "forward_tflops_algorithmic": wk["algorithmic"] / (ms * 1e-3) / 1e12,
                     "steps": args.steps, "config": config_of(w, "flushed between steps")}
        del fs
        torch.cuda.empty_cache()
    return res


def run_gpu(args, w):
    rank, world, local, dist = dist_setup(args.gpus)
    import transformer_attention_variant_gb300 as iha
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    wk = work(w)
    dt = iha.IHA_DTYPE_BF16 if w.dtype == "bf16" else iha.IHA_DTYPE_F32
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    host = gi.make_inputs(w)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    fs = ForwardStep(iha, w, host, dev, stream)
    route, names = fs.route, fs.names
    clk = ClockSampler(local)
    mean_step, kmean, t_wall = fs.time(args.steps, args.warmup, flush, dist=dist, clocks=clk)
    mean_step = max_over_ranks(mean_step, dist, dev)
    value = job_value(world, wk["pseudo_tokens"], mean_step)

    # roofline of the dominant kernel
    dom = max(kmean, key=kmean.get)
    if dom == "attention":
        ach = wk["attn"] / (kmean[dom] * 1e-3) / 1e12
        roof = {"kernel": "attn_fwd_tc", "bound": "tensor", "achieved": ach, "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16"],
                "frac_of_sustained": ach / peaks["bf16_sustained"],
                "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
                else "fallback 1.9 PFLOP/s"}
        traffic_key = "attention"
    elif dom in ("project", "project_mix"):
        ach = (wk["proj_folded"] if dom == "project" else wk["proj_heads"]) / (kmean[dom] * 1e-3) / 1e12
        roof = {"kernel": "proj_gemm_tc", "bound": "tensor", "achieved": ach, "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16"],
                "frac_of_sustained": ach / peaks["bf16_sustained"], "peak_source": peaks["source"]}
        traffic_key = dom
    else:
        b = {"contract": wk["bytes_contract"], "fold": wk["bytes_fold"], "slice_weights": wk["bytes_slice"]}[dom]
        ach = b / (kmean[dom] * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": ach / peaks["hbm"], "peak_source": peaks["source"]}
        traffic_key = dom
    roof["traffic"] = traffic_per_launch(w.name, traffic_key)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": DATA,
        "config": config_of(w, "flushed between steps (256 MiB write outside the timed events)"),
        "tflops": {
            "attention_exact_pairs": wk["attn"] / (kmean["attention"] * 1e-3) / 1e12,
            "forward_algorithmic": wk["algorithmic"] / (mean_step * 1e-3) / 1e12,
            "forward_executed": (wk["executed_unfolded"] if route == 1 else wk["executed_folded"])
            / (mean_step * 1e-3) / 1e12,
            "projection_gemm": (wk["proj_heads"] / (kmean["project_mix"] * 1e-3) if route == 1
                                else wk["proj_folded"] / (kmean["project"] * 1e-3)) / 1e12,
        },
        "kernel_ms": kmean,
        "projection_route": ("head projections with the mixing in the GEMM epilogue" if route == 1
                             else "fold alpha into W + project"),
        "roofline": roof,
        "gpu_launches": len(names) * args.steps,
        "wall_s_timed_region": t_wall,
        "clocks": clk.summary(),
    }

    # end to end through the host-buffer entry point (pinned host inputs, copies in the timed region)
    if not args.no_e2e:
        hin = {k: v.contiguous().pin_memory() for k, v in host.items()}
        hout = torch.empty(w.B, w.N, w.D, dtype=tdt).pin_memory()
        nbytes = iha.iha_host_buffer_bytes(w.B, w.N, w.H, w.d, w.P, dt)
        del fs
        torch.cuda.empty_cache()
        dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        h2d = sum(v.numel() * v.element_size() for v in hin.values())
        d2h = hout.numel() * hout.element_size()

        def e2e_call():
            rc = iha.iha_forward_host(hin["X"], hin["W_Q"], hin["W_K"], hin["W_V"], hin["alpha_Q"], hin["alpha_K"],
                                      hin["alpha_V"], hin["R"], w.B, w.N, w.H, w.d, w.P, w.mask_mode, w.window,
                                      hout, dt, stream, dbuf, nbytes)
            iha.check(rc, "iha_forward_host")

        for _ in range(max(1, args.warmup)):
            e2e_call()
        n_e2e = max(3, min(args.steps, 50))
        t = []
        for _ in range(n_e2e):
            flush.fill_(0)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            e2e_call()
            t.append(time.perf_counter() - t0)
        e2e_s = max_over_ranks(sum(t) / len(t), dist, dev)
        line["e2e"] = {"value": job_value(world, wk["pseudo_tokens"], e2e_s * 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3, "steps": n_e2e,
                       "call": "iha_forward_host (pinned host buffers, preallocated device buffer)"}

    if args.side_workloads and world == 1 and args.workload == DEFAULT_WORKLOAD and args.N is None:
        if not args.no_e2e:
            del dbuf
            torch.cuda.empty_cache()
        line["workloads"] = side_workloads(iha, args, dev, stream, flush, peaks, skip=w.name)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        f = gi.as_f64(host)
        v, secs, n = time_oracle(w, f, args.cpu_tokens)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
                                "sample": oracle_sample_desc(w, n), "seconds": secs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_stack(args, w):
    """The layer stack of the pages' appendix C on workload w's shape: four sliding-window
    IHA layers (P = w.P, window N/(2P^2) tokens) and one global layer (P = 1, causal), timed
    through iha_forward_stack.  Its own JSON line; value = tokens through the stack / s."""
    rank, world, local, dist = dist_setup(args.gpus)
    import transformer_attention_variant_gb300 as iha
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    sched = gi.local_global_schedule(w.N, w.P)
    host = gi.make_stack_inputs(w.B, w.N, w.H, w.d, w.dtype, w.seed, sched)
    keys = ("W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")
    layers = []
    for L in host:
        dl = {k: L[k].to(dev).contiguous() for k in keys}
        dl.update(P=L["P"], mask_mode=L["mask_mode"], window=L["window"])
        layers.append(dl)
    X = host[0]["X"].to(dev).contiguous()
    out = torch.empty_like(X)
    dt = iha.IHA_DTYPE_BF16 if w.dtype == "bf16" else iha.IHA_DTYPE_F32
    ws_bytes = iha.iha_stack_workspace_bytes([L["P"] for L in layers], w.B, w.N, w.H, w.d, dt)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flops = sum(work(L["workload"])["algorithmic"] for L in host)

    def step():
        iha.check(iha.iha_forward_stack(X, layers, w.B, w.N, w.H, w.d, dt, out, stream, ws, ws_bytes), "stack")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            step()
    torch.cuda.synchronize()
    barrier(dist)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(i & 0xFF)          # evict L2 between steps (outside the events)
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status(stream)
    iha.check(rc, f"device status after timed steps ({code:#x})")
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    ms = max_over_ranks(ms, dist, dev)
    barrier(dist)
    if rank == 0:
        line = {
            "metric": "IHA layer stack (4 sliding-window layers + 1 global layer) tokens/s, 1 GPU per replica",
            "value": job_value(world, w.B * w.N, ms), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": DATA,
            "config": {"workload": f"stack4x1_{w.name}", "B": w.B, "N": w.N, "H": w.H, "d": w.d,
                       "layers": [{"P": L["P"], "mask": ["none", "causal", "causal+window"][L["mask_mode"]],
                                   "window": L["window"] or None} for L in layers],
                       "l2": "flushed between steps (256 MiB write outside the timed events)"},
            "tflops_algorithmic": flops / (ms * 1e-3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": peaks["bf16"],
                         "unit": "TFLOP/s", "frac": flops / (ms * 1e-3) / 1e12 / peaks["bf16"], "traffic": None,
                         "note": "whole stack: the layers' algorithmic flops over the stack's time"},
            "gpu_launches": 4 * len(layers) * args.steps, "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_decode(args, w):
    """One decoding step at position N-1 over a full cache of workload w's shape (B
    sequences, N cached tokens, P pseudo-heads): HBM-bound, so reported against the copy
    bandwidth.  Algorithmic bytes per step: W_Q, W_K, W_V once (3 D^2 bf16) + the readable
    cached pseudo-keys and values + the new token's rows; the cache holds random values."""
    rank, world, local, dist = dist_setup(args.gpus)
    import transformer_attention_variant_gb300 as iha
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    B, N, H, d, P = w.B, w.N, w.H, w.d, w.P
    host = gi.make_inputs(w.with_(N=1, name=w.name + "@decode"))
    dd = {k: v.to(dev).contiguous() for k, v in host.items()}
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    Kc = torch.randn(B, H, N * P, d, generator=g, device=dev).to(torch.bfloat16)
    Vc = torch.randn(B, H, N * P, d, generator=g, device=dev).to(torch.float16)
    x = dd["X"].reshape(B, w.D).contiguous()
    out = torch.empty(B, w.D, dtype=torch.bfloat16, device=dev)
    ws_bytes = iha.iha_decode_workspace_bytes(B, H, d, P)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    t = N - 1
    lo = max(0, (t - w.window + 1) * P) if w.mask_mode == gi.MASK_WINDOW else 0
    rows = (t + 1) * P - lo
    nbytes = 3 * w.D * w.D * 2 + B * H * rows * d * 2 * 2 + B * w.D * 2 * 2

    def step():
        iha.check(iha.iha_decode_step(x, dd["W_Q"], dd["W_K"], dd["W_V"], dd["alpha_Q"], dd["alpha_K"], dd["alpha_V"],
                                      dd["R"], B, H, d, P, w.mask_mode, w.window, Kc, Vc, N, t, out,
                                      iha.IHA_DTYPE_BF16, stream, ws, ws_bytes), "decode")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            step()
    torch.cuda.synchronize()
    barrier(dist)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status(stream)
    iha.check(rc, f"device status after timed steps ({code:#x})")
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    ms = max_over_ranks(ms, dist, dev)
    barrier(dist)
    if rank == 0:
        gbs = nbytes / (ms * 1e-3) / 1e9
        line = {
            "metric": "IHA decode step tokens/s (one new token per sequence over a full pseudo-token cache)",
            "value": job_value(world, B, ms), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": DATA + "; cache filled with N(0,1) values",
            "config": {"workload": f"decode_{w.name}", "B": B, "cached_tokens": N, "H": H, "d": d, "P": P,
                       "mask": ["none", "causal", "causal+window"][w.mask_mode], "window": w.window or None,
                       "l2": "flushed between steps (256 MiB write outside the timed events)"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"], "bytes_per_step": nbytes, "traffic": None},
            "gpu_launches": 4 * args.steps, "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_backward(args, w):
    """One backward pass of the layer (iha_backward, forward pieces recomputed inside) on
    workload w; reports gradient passes per second and the algorithmic TFLOP/s (the
    backward's flops: twice the forward's projections and mixing, 2.5x its attention
    pairs, the contraction and token reductions)."""
    rank, world, local, dist = dist_setup(args.gpus)
    import transformer_attention_variant_gb300 as iha
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    B, N, H, d, P, D = w.B, w.N, w.H, w.d, w.P, w.D
    host = gi.make_inputs(w)
    dd = {k: v.to(dev).contiguous() for k, v in host.items()}
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    dO = torch.randn(B, N, D, generator=g, device=dev).to(torch.bfloat16)
    keys = ("X", "W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")
    outs = [torch.empty_like(dd[k]) for k in keys]
    ws_bytes = iha.iha_backward_workspace_bytes(B, N, H, d, P, iha.IHA_DTYPE_BF16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    wk = work(w)
    # gradients: projections (dX and dW: 2x the head projections), mixing and contraction
    # (2x each), attention (QK^T, dP, dS K, dS^T Q, P^T dO: 10 d flops per pair, 2.5x forward)
    flops = 2 * wk["proj_heads"] + 2 * (wk["algorithmic"] - wk["proj_heads"] - wk["attn"]) + 2.5 * wk["attn"]

    def step():
        iha.check(iha.iha_backward(*(dd[k] for k in keys), B, N, H, d, P, w.mask_mode, w.window, dO, *outs,
                                   iha.IHA_DTYPE_BF16, stream, ws, ws_bytes), "backward")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    barrier(dist)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status(stream)
    iha.check(rc, f"device status after timed steps ({code:#x})")
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    ms = max_over_ranks(ms, dist, dev)
    barrier(dist)
    if rank == 0:
        tf = flops / (ms * 1e-3) / 1e12
        line = {
            "metric": "IHA backward (all input gradients) pseudo-tokens/s and TFLOP/s, 1 GPU per replica",
            "value": job_value(world, wk["pseudo_tokens"], ms), "unit": "pseudo-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": DATA,
            "config": config_of(w, "flushed between steps (256 MiB write outside the timed events)"),
            "tflops_algorithmic": tf,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16"], "traffic": None,
                         "note": "whole backward (forward recomputed inside counts as overhead, not work)"},
            "gpu_launches": None, "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_train(args, w):
    """One training step of the layer on workload w without recomputation: iha_forward_train
    (the forward, leaving its pieces in the backward workspace) then iha_backward_saved (every
    input gradient from them).  Reports steps/s as pseudo-tokens/s, the algorithmic TFLOP/s of
    forward + backward, and each half's time (CUDA events between the two calls)."""
    rank, world, local, dist = dist_setup(args.gpus)
    import transformer_attention_variant_gb300 as iha
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    B, N, H, d, P, D = w.B, w.N, w.H, w.d, w.P, w.D
    host = gi.make_inputs(w)
    dd = {k: v.to(dev).contiguous() for k, v in host.items()}
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    dO = torch.randn(B, N, D, generator=g, device=dev).to(torch.bfloat16)
    keys = ("X", "W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")
    grads = [torch.empty_like(dd[k]) for k in keys]
    out = torch.empty(B, N, D, dtype=torch.bfloat16, device=dev)
    ws_bytes = iha.iha_backward_workspace_bytes(B, N, H, d, P, iha.IHA_DTYPE_BF16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    wk = work(w)
    fwd_flops = wk["algorithmic"]
    bwd_flops = 2 * wk["proj_heads"] + 2 * (wk["algorithmic"] - wk["proj_heads"] - wk["attn"]) + 2.5 * wk["attn"]
    args_in = [dd[k] for k in keys] + [B, N, H, d, P, w.mask_mode, w.window]

    def fwd():
        iha.check(iha.iha_forward_train(*args_in, out, iha.IHA_DTYPE_BF16, stream, ws, ws_bytes), "forward_train")

    def bwd():
        iha.check(iha.iha_backward_saved(*args_in, dO, *grads, iha.IHA_DTYPE_BF16, stream, ws, ws_bytes),
                  "backward_saved")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            fwd()
            bwd()
    torch.cuda.synchronize()
    barrier(dist)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                ev[i][0].record(stream)
                fwd()
                ev[i][1].record(stream)
                bwd()
                ev[i][2].record(stream)
        torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status(stream)
    iha.check(rc, f"device status after timed steps ({code:#x})")
    ms_f = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    ms_b = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    ms = max_over_ranks(ms_f + ms_b, dist, dev)
    barrier(dist)
    if rank == 0:
        tf = (fwd_flops + bwd_flops) / (ms * 1e-3) / 1e12
        line = {
            "metric": "IHA training step (forward + all input gradients, no recomputation) pseudo-tokens/s, 1 GPU "
                      "per replica",
            "value": job_value(world, wk["pseudo_tokens"], ms), "unit": "pseudo-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": DATA,
            "config": config_of(w, "flushed between steps (256 MiB write outside the timed events)"),
            "forward_train_ms": ms_f, "backward_saved_ms": ms_b, "tflops_algorithmic": tf,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16"], "traffic": None},
            "gpu_launches": None, "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def traffic_per_launch(workload, kernel):
    """DRAM bytes (read + write) per launch recorded from ncu in profiles/dram_traffic.txt,
    provided the kernel's source is unchanged since that capture; None otherwise."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        f = line.split()
        if len(f) < 6 or f[0].startswith("#") or f[0] != workload or f[1] != kernel:
            continue
        src = os.path.join(ROOT, "transformer_attention_variant_gb300", "csrc", f[2])
        if not os.path.exists(src):
            return None
        if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != f[3]:
            return None
        return int(f[4]) + int(f[5])
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=gi.WORKLOAD_ORDER)
    ap.add_argument("--cpu-tokens", type=int, default=768, help="oracle sample size for cpu_baseline (about 10-15 s)")
    ap.add_argument("--ref-tokens", type=int, default=48, help="oracle sample size per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end host-buffer measurement")
    ap.add_argument("--no-side-workloads", dest="side_workloads", action="store_false",
                    help="do not time the other target workloads (the 'workloads' object of the line)")
    ap.add_argument("--stack", action="store_true",
                    help="time the four-local + one-global layer stack on the workload's shape instead")
    ap.add_argument("--decode", action="store_true",
                    help="time one decoding step over a full cache of the workload's shape instead")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (iha_backward) on the workload instead")
    ap.add_argument("--train", action="store_true",
                    help="time a training step (iha_forward_train + iha_backward_saved) on the workload instead")
    ap.add_argument("--N", type=int, default=None,
                    help="shrink the workload's sequence length (smaller cases for profiler captures); "
                         "the window stays N/(2P) for windowed workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = gi.WORKLOADS[args.workload]
    if args.N is not None:
        w = w.with_(N=args.N, name=f"{w.name}@N={args.N}",
                    window=args.N // (2 * w.P) if w.mask_mode == gi.MASK_WINDOW else w.window)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.stack:
        run_stack(args, w)
    elif args.decode:
        run_decode(args, w)
    elif args.backward:
        run_backward(args, w)
    elif args.train:
        run_train(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
