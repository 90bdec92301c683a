#!/usr/bin/env python
"""Decode benchmark: decode tokens/s of a hybrid Gated-DeltaNet / GQA / MoE
model on one GB300, and achieved HBM GB/s as a fraction of the measured peak.

Workloads (--workload), seeded synthetic weights and inputs of the configs'
shapes:
  dense4b (default)  dense 4B-shaped hybrid (32 layers, 3:1 DeltaNet:GQA, hidden
                     2560, FFN 9216, vocab 151936), bf16, random 4096-token
                     prompt, then --steps greedy steps (one CUDA-graph launch
                     each, the argmax fed back on the device);
  dense4b-32k        the same at context 32768 (seeded cache fill), with the
                     split-KV sweep and tokens/s per 32-token window;
  moe35b             MoE 35B-A3B-shaped hybrid, bf16, 2048-token prompt;
  moe35b-q4-b8       its 4-bit form at batch 8, ragged contexts 1024..16384
                     (seeded cache fill), seeded tokens per sequence and step;
  tiny               the 2-layer test model.

One JSON line on rank 0.  `--impl reference` times the FP64 CPU oracle on the
same metric and config instead.  With torchrun (N > 1) every rank runs an
independent replica (the decode step has no cross-GPU exchange).  On one GPU,
the default workload's line also carries `other_workloads`: the same
measurement of dense4b-32k, moe35b and moe35b-q4-b8, each run after the main
one in a process of its own (--no-other-workloads skips them).
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tokens/s; achieved HBM GB/s as fraction of GB300 peak"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REFERENCE_BUDGET_S = 120.0
SYNTHETIC_FILL_ABOVE = 8192  # longer prompts: seeded synthetic cache fill instead of a token-by-token prefill
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="dense4b")
    ap.add_argument("--splits", type=int, default=0, help="split-KV chunks per kv head (0 = automatic)")
    ap.add_argument("--layers", type=int, default=0, help="truncate depth (profiling captures only)")
    ap.add_argument("--prompt", type=int, default=-1, help="override the prompt length (profiling captures only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernel-timing", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="no programmatic dependent launch between kernels")
    ap.add_argument("--kernel-table", action="store_true",
                    help="time every decode kernel kind on its own (CUDA graphs over every layer's own buffers) and "
                         "print one JSON line of rows instead of the benchmark line")
    ap.add_argument("--paged", action="store_true", help="batch workloads: a paged KV cache sized to the contexts")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="default workload on one GPU: skip the runs of the other workloads")
    return ap.parse_args(argv)


OTHER_WORKLOADS = ("dense4b-32k", "moe35b", "moe35b-q4-b8")
OTHER_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "config", "roofline", "step_roofline", "timing",
              "split_sweep_tokens_per_s", "prefill", "e2e", "gpu_launches", "kernels_per_step", "clocks")


def other_workloads(args):
    """The other decode workloads, each measured by this script in a process
    of its own (same steps and warm-up, no CPU baseline), after the main run
    has released the GPU; their lines, trimmed to the measurement keys."""
    out = {}
    for wl in OTHER_WORKLOADS:
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", wl, "--steps", str(args.steps),
               "--warmup", str(args.warmup), "--no-cpu-baseline", "--no-other-workloads"]
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, env=dict(os.environ))
            lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
            if r.returncode != 0 or not lines:
                out[wl] = {"error": f"exit {r.returncode}: {(r.stderr or '').strip().splitlines()[-1:]}"}
                continue
            d = json.loads(lines[-1])
            out[wl] = {k: d[k] for k in OTHER_KEYS if k in d}
        except (subprocess.TimeoutExpired, OSError, ValueError) as e:
            out[wl] = {"error": f"{type(e).__name__}: {e}"}
    return out


def workload_of(args):
    from synth import workloads
    w = workloads.WORKLOADS[args.workload]
    shape = w.shape
    if args.layers:
        shape = dataclasses.replace(shape, name=f"{shape.name}-l{args.layers}", n_layers=args.layers,
                                    attn_layers=tuple(l for l in shape.attn_layers if l < args.layers))
    prompt = w.prompt_len if args.prompt < 0 else args.prompt
    return w, shape, prompt


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if any."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for ln in f:
            parts = ln.split()
            if len(parts) >= 3 and not ln.startswith("#") and parts[0] == kernel and parts[1] == workload:
                return int(parts[2])
    return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        for ln in out.strip().splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(REASONS, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(seconds: float, dist, device) -> float:
    """The slowest rank's time (every rank gets it); `dist` None: this rank's."""
    if dist is None:
        return seconds
    import torch
    tt = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(n_ranks: int, units_per_rank: int, seconds: float) -> float:
    """Whole-job units per second: every rank processed units_per_rank in at most
    `seconds` (weak scaling: independent replicas, no exchange)."""
    return max(n_ranks, 1) * units_per_rank / seconds


# ---------------------------------------------------------------- CPU oracle

def oracle_decode_sample(shape, context: int, budget_s: float, max_tokens: int, host_w=None, warm=True):
    """Time full-depth oracle decode tokens at position `context` from a seeded
    synthetic cache (random K/V rows and recurrent state: the prompt itself is
    not replayed on the CPU).  Returns (tokens/s, threads, tokens, seconds)."""
    import numpy as np

    from oracle import oracle as orc
    from synth import gen, workloads
    if host_w is None:
        host_w = workloads.host_weights(shape)
    o = orc.Oracle(shape, host_w, context + max_tokens + 2)
    rng = np.random.default_rng(1234)
    n_attn = sum(1 for l in range(shape.n_layers) if shape.is_attn(l))
    for a in range(n_attn):
        K, V = o.kv_cache(a)
        K[:, :context] = gen.f32_to_bf16_bits(rng.standard_normal((shape.attn_kv_heads, context, shape.head_dim))
                                              .astype(np.float32))
        V[:, :context] = gen.f32_to_bf16_bits(rng.standard_normal((shape.attn_kv_heads, context, shape.head_dim))
                                              .astype(np.float32) * 0.1)
    for gi in range(shape.n_layers - n_attn):
        S = o.gdn_state(gi)
        S[:] = (rng.standard_normal(S.shape) * 0.01).astype(np.float32)
    o.cache.len = context
    tok = 17
    n = max_tokens
    if warm:  # one untimed token, which also sizes the sample to the budget
        t0 = time.perf_counter()
        o.forward(tok, want_hidden=False)
        t1 = time.perf_counter() - t0
        n = max(1, min(max_tokens, int(math.ceil(budget_s / max(t1, 1e-3)))))
    t0 = time.perf_counter()
    for i in range(n):
        tok = int(orc.argmax(o.forward(tok, want_hidden=False)["logits"]))
    dt = time.perf_counter() - t0
    return n / dt, orc.threads(), n, dt


def cpu_baseline_obj(shape, context: int, what: str):
    """The oracle on this host's cores (all of them, ~12 s) and on one core (one
    token), at `context` from a seeded synthetic cache."""
    from oracle import oracle as orc
    from synth import workloads
    host_w = workloads.host_weights(shape)
    tps, cores, ntok, dt = oracle_decode_sample(shape, context, budget_s=12.0, max_tokens=16, host_w=host_w)
    orc.set_threads(1)
    try:
        tps1, _, ntok1, dt1 = oracle_decode_sample(shape, context, budget_s=0.0, max_tokens=1, host_w=host_w,
                                                   warm=False)
    finally:
        orc.set_threads(cores)
    return {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "oracle": "FP64 throughout, the DeltaNet step with its explicit dk x dk matrix",
            "cpu_model": cpu_model(),
            "value_1_core": tps1,
            "sample": f"{ntok} full-depth FP64 oracle decode tokens{' ' + what if what else ''} at context {context} "
                      f"from a seeded "
                      f"synthetic cache ({dt:.1f} s on {cores} threads; {ntok1} token on 1 thread, {dt1:.1f} s)"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w, shape, prompt = workload_of(args)
    from synth import workloads
    host_w = workloads.host_weights(shape)
    import numpy as np  # noqa: F401

    from oracle import oracle as orc
    o_warm = max(args.warmup, 0)
    # warm-up tokens are part of the same sampler run; up to W + K tokens,
    # bounded to about two minutes of CPU work
    if w.batch > 1:  # the oracle runs one sequence at a time: sample one at the batch's mean context
        ctx = [int(c) for c in workloads.ragged_contexts(w)]
        prompt = int(round(sum(ctx) / len(ctx)))
    tps, cores, n, dt = oracle_decode_sample(shape, prompt, budget_s=REFERENCE_BUDGET_S,
                                             max_tokens=o_warm + args.steps, host_w=host_w)
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000.0 / tps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "context": prompt, "batch": w.batch},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "oracle": "FP64 throughout, the DeltaNet step with its explicit dk x dk matrix",
                         "sample": f"{n} full-depth FP64 oracle decode tokens ({dt:.1f} s) at context {prompt} from a "
                                   f"seeded synthetic cache (prompt not replayed on the CPU)"},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    del orc
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch

    from bandwidth_bound_hybrid_gb300 import accounting as acc
    from bandwidth_bound_hybrid_gb300 import build as hb
    from bandwidth_bound_hybrid_gb300.model import HybridModel
    from synth import workloads

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
        torch.cuda.set_device(0)
    if rank == 0:
        hb.build()
    if dist:
        dist.barrier()

    w, shape, prompt = workload_of(args)
    if w.batch > 1:
        return run_ours_batch(args, w, shape, dist, ws, rank, local)
    peak, peak_kind = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream()

    weights = workloads.device_weights(shape)
    cap = prompt + args.warmup + 2 * args.steps + 16
    from bandwidth_bound_hybrid_gb300 import capi as _capi
    flags = _capi.HY_FLAG_NO_PDL if args.no_pdl else 0
    model = HybridModel(shape, weights, [cap], splits=args.splits, flags=flags)
    toks = torch.from_numpy(workloads.prompt_ids(w, n=prompt)).to(dev) if prompt else None
    ids = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)  # the step returns logits and the greedy id
    synthetic_fill = prompt > SYNTHETIC_FILL_ABOVE
    pre = None
    if synthetic_fill:  # a step's cost depends on the context length, not on what the cache holds
        model.fill_synthetic(0, prompt, seed=1)
        ids.copy_(toks[-1:])
    elif prompt:
        pre = timed_prefill(model, toks, shape, logits)
        ids.copy_(toks[-1:])
    for _ in range(args.warmup):
        model.decode_step(0, ids, ids, logits)
    torch.cuda.synchronize()
    assert model.check_device() == 0, "device guard fired during warm-up"
    ctx0 = model.seq_len(0)

    # ---- timed region: K graph launches, inputs resident in HBM
    depth_window = 32 if w.splits else 0  # the long-context workload: tokens/s per 32-token window
    t, clk, windows, win = timed_region(args, dist, local, st, lambda: model.decode_step(0, ids, ids, logits),
                                        window=depth_window, warm=False)
    assert model.check_device() == 0, "device guard fired in the timed region"
    n = max(ws, 1)
    value = job_throughput(n, args.steps, t)
    mid_ctx = ctx0 + args.steps // 2
    sb = acc.step_bytes(shape, mid_ctx, logits=True)
    step_gbs = sb.total * args.steps / t / 1e9

    # ---- dominant kernel: the gate/up SwiGLU GEMV.  One CUDA graph launches
    # it once per layer over that layer's weights (every launch streams fresh
    # weights from HBM); average launch duration = graph time / launches.
    roof = None
    if not args.no_kernel_timing and shape.ffn > 0:
        from bandwidth_bound_hybrid_gb300 import capi
        L = capi.lib()
        x = torch.randn(shape.hidden, device=dev)
        g = torch.ones(shape.hidden, device=dev)
        h = torch.empty(shape.ffn, device=dev)
        side = torch.cuda.Stream()

        def sweep_layers(stream):
            for l in range(shape.n_layers):
                capi.check(L.hy_op_gemv_swiglu(weights[f"l{l}.w_gate"].data_ptr(), weights[f"l{l}.w_up"].data_ptr(),
                                               shape.ffn, shape.hidden, x.data_ptr(), g.data_ptr(), 1e-6, h.data_ptr(),
                                               stream.cuda_stream), "gemv_swiglu")

        with torch.cuda.stream(side):
            sweep_layers(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            sweep_layers(side)
        graph.replay()
        torch.cuda.synchronize()
        reps = 5
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            graph.replay()
        b.record(st)
        torch.cuda.synchronize()
        launch_s = a.elapsed_time(b) / 1e3 / (reps * shape.n_layers)
        bytes_launch = acc.gemv_swiglu_bytes(shape.ffn, shape.hidden)
        achieved = bytes_launch / launch_s / 1e9
        roof = {"bound": "hbm", "kernel": "gemv gate/up + SwiGLU (k_gemv, dense rows, SwiGLU epilogue)", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": load_traffic("gemv_swiglu", args.workload),
                "bytes_per_launch": bytes_launch, "launch_us_mean": launch_s * 1e6,
                "launches_timed": reps * shape.n_layers, "peak_source": f"{peak_kind} hbm_gbs"}
        del graph

    # ---- split-KV sweep (workloads that name split counts): same timed region per count
    sweep = None
    if w.splits and not args.splits and args.layers == 0:
        sweep = {}
        for sp in w.splits:
            m2 = HybridModel(shape, weights, [cap], splits=sp, flags=flags)
            m2.fill_synthetic(0, ctx0, seed=1)
            ids2 = ids.clone()
            t2 = timed_region(args, dist, local, st, lambda: m2.decode_step(0, ids2, ids2, logits))[0]
            assert m2.check_device() == 0
            sweep[str(sp)] = max(ws, 1) * args.steps / t2
            m2.close()

    if not args.no_kernel_timing and shape.ffn == 0:
        roof = moe_gateup_roofline(shape, weights, peak, peak_kind, args.workload)

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    tok_h = torch.zeros(1, dtype=torch.int32).pin_memory()
    ids_h = torch.zeros(1, dtype=torch.int32).pin_memory()
    tok_h[0] = int(ids.item())
    e2e_steps = args.steps
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        model.decode_step_host(0, tok_h, ids_h)
        tok_h[0] = ids_h[0]
    e2e_t = time.perf_counter() - t0
    e2e_t = max_over_ranks(e2e_t, dist, dev)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_obj(shape, mid_ctx, "")

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "shape": shape.name, "batch": 1, "prompt": prompt,
                       "context_timed": [ctx0, ctx0 + args.steps], "weights": "bf16",
                       "kv": "int8 + FP32 scale per vector" if getattr(shape, "kv_format", 0) else "bf16",
                       "outputs": "FP32 logits [V] and the greedy id per step",
                       "context_fill": "seeded synthetic KV rows and recurrent state (no prompt replay)"
                       if synthetic_fill else "prefill of the prompt",
                       "splits": model.step_splits(0), "parallelism": f"replicas x{n}",
                       "l2": "inputs larger than L2: every step streams all weights (GBs) through the 129 MB L2"},
            "roofline": roof,
            "step_roofline": {"bound": "hbm", "bytes_per_step": sb.total, "achieved": step_gbs, "peak": peak,
                              "unit": "GB/s", "frac": step_gbs / peak},
            "timing": window_stats(windows, win, args.steps),
            "depth_curve": [{"context_start": ctx0 + i * win, "tokens_per_s": n * win / wt}
                            for i, wt in enumerate(windows) if (i + 1) * win <= args.steps] if depth_window else None,
            "split_sweep_tokens_per_s": sweep,
            "prefill": pre,
            "cpu_baseline": cpu,
            "e2e": {"value": n * e2e_steps / e2e_t, "unit": "tokens/s", "h2d_bytes_per_step": 4,
                    "d2h_bytes_per_step": 4},
            "gpu_launches": model.step_kernels() * args.steps,
            "kernels_per_step": model.step_kernels(),
            "graph_launches_per_token": 1,
            "clocks": clk,
        }
    model.close()
    if rank == 0:
        if ws == 1 and args.workload == "dense4b" and not args.no_other_workloads and not args.layers \
                and args.prompt < 0:
            del model, weights
            torch.cuda.empty_cache()
            line["other_workloads"] = other_workloads(args)
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def timed_region(args, dist, local, st, step, window=0, before_timing=None, warm=True):
    """W warm-up steps, then K timed steps between barriers and device
    synchronisations, with the clocks sampled meanwhile.  Events are also
    recorded every `window` steps (default: K / 7) inside the timed region (no
    synchronisation between them).  Returns (seconds, max over ranks; clock
    record; per-window seconds of this rank)."""
    import torch
    for _ in range(args.warmup if warm else 0):
        step()
    torch.cuda.synchronize()
    if before_timing:
        before_timing()
    win = window if window > 0 else max(1, args.steps // 7)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps // win + 2)]
    clocks = Clocks(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    evs[0].record(st)
    n_ev = 1
    for i in range(args.steps):
        step()
        if (i + 1) % win == 0 and (i + 1) < args.steps:
            evs[n_ev].record(st)
            n_ev += 1
    evs[n_ev].record(st)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    t = evs[0].elapsed_time(evs[n_ev]) / 1e3
    windows = [evs[i].elapsed_time(evs[i + 1]) / 1e3 for i in range(n_ev)]
    t = max_over_ranks(t, dist, torch.device("cuda", local))
    return t, clk, windows, win


def window_stats(windows, win, steps):
    """Mean ms per step over the full windows, their coefficient of variation
    and a Student-t 95% interval of the mean."""
    full = [w / win * 1e3 for i, w in enumerate(windows) if (i + 1) * win <= steps]
    n = len(full)
    if n < 2:
        return None
    m = statistics.mean(full)
    sd = statistics.stdev(full)
    tq = {2: 12.71, 3: 4.303, 4: 3.182, 5: 2.776, 6: 2.571, 7: 2.447, 8: 2.365, 9: 2.306, 10: 2.262}.get(n, 2.0)
    h = tq * sd / math.sqrt(n)
    return {"windows": n, "steps_per_window": win, "ms_per_step_mean": m, "cv": sd / m if m else None,
            "ci95_ms_per_step": [m - h, m + h], "cv_over_5pct": (sd / m) > 0.05 if m else None}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part", "hardware")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def gemv_in_roofline(shape, weights, peak, peak_kind, workload):
    """The batch-1 GEMV (k_gemv) timed alone with RMSNorm fused: one graph
    launches it once per layer over that layer's input projection (every
    launch streams a fresh bf16 matrix from HBM); average launch duration =
    graph time / launches."""
    import torch

    from bandwidth_bound_hybrid_gb300 import accounting as acc
    from bandwidth_bound_hybrid_gb300 import capi
    L = capi.lib()
    H = shape.hidden
    x = torch.randn(H, device="cuda")
    g = torch.ones(H, device="cuda")
    layers = [l for l in range(shape.n_layers) if not shape.is_attn(l)]  # one launch shape: the DeltaNet layers'
    R = shape.gdn_in_rows
    y = torch.empty(R, device="cuda")
    side = torch.cuda.Stream()

    def sweep(stream):
        for l in layers:
            capi.check(L.hy_op_gemv(weights[f"l{l}.w_in"].data_ptr(), R, H, x.data_ptr(), g.data_ptr(), 1e-6,
                                    y.data_ptr(), 0, stream.cuda_stream), "gemv")

    with torch.cuda.stream(side):
        sweep(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        sweep(side)
    graph.replay()
    torch.cuda.synchronize()
    reps = 5
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        graph.replay()
    b.record(st)
    torch.cuda.synchronize()
    launch_s = a.elapsed_time(b) / 1e3 / (reps * len(layers))
    bytes_launch = acc.linear_bytes(R, H, 0) + (H + R) * acc.F32
    achieved = bytes_launch / launch_s / 1e9
    del graph
    return {"bound": "hbm", "kernel": f"gemv with fused RMSNorm (k_gemv), DeltaNet input projections [{R}, {H}]",
            "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": load_traffic("gemv_in", workload), "bytes_per_launch": bytes_launch,
            "launch_us_mean": launch_s * 1e6, "launches_timed": reps * len(layers),
            "peak_source": f"{peak_kind} hbm_gbs"}


def load_tensor_peak():
    """Measured dense bf16 tensor throughput (TFLOP/s): (burst, sustained, kind)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return 1900.0, 1700.0, "fallback"


def timed_prefill(model, toks, shape, logits):
    """The prompt through hy_prefill, timed with CUDA events on the launching
    stream: time to the first token's logits, tokens/s, and FLOP rates
    (prompt GEMMs at bf16 hi + lo on the tensor cores, the rest on the CUDA
    cores) against the measured sustained bf16 tensor peak."""
    import torch

    from bandwidth_bound_hybrid_gb300 import accounting as acc
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(st)
    model.prefill(0, toks, logits)
    b.record(st)
    torch.cuda.synchronize()
    t = a.elapsed_time(b) / 1e3
    n = int(toks.numel())
    fl = acc.prefill_flops(shape, n)
    _, sustained, kind = load_tensor_peak()
    chunked = getattr(shape, "weight_format", 0) == 0 and getattr(shape, "kv_format", 0) == 0
    gemms = ("tcgen05 GEMMs (the experts as grouped GEMMs over the tokens that picked them)" if shape.is_moe
             else "tcgen05 GEMMs")
    return {"tokens": n, "ttft_ms": t * 1e3, "tokens_per_s": n / t,
            "path": f"chunks of up to 2048 tokens: {gemms} + prompt mixer kernels" if chunked
            else "token by token through the decode step",
            "flops_total": fl["total"], "tflops_total": fl["total"] / t / 1e12,
            "tensor_tflops_executed": fl["tensor_executed"] / t / 1e12, "peak_tflops_sustained": sustained,
            "frac_of_tensor_peak_whole_prefill": fl["tensor_executed"] / t / 1e12 / sustained,
            "peak_source": f"{kind} bf16_tflops_sustained"}


def graph_us_per_launch(launches, reps=5):
    """Mean microseconds per launch of one CUDA graph that makes every call of
    `launches` (functions of a stream handle) once, replayed `reps` times."""
    import torch
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        for f in launches:
            f(side.cuda_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for f in launches:
            f(side.cuda_stream)
    graph.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        graph.replay()
    b.record(st)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (reps * len(launches))
    del graph
    return us


def moe_gateup_roofline(shape, weights, peak, peak_kind, workload):
    """The MoE step's dominant kernel timed alone: the expert gate/up + SwiGLU
    (k_gemv over the routed experts' rows, routing in every CTA), one graph
    launching it once per layer over that layer's expert tensors from fixed
    router logits (top_k + 1 slots of Fe gate and up rows each launch: fresh
    weights from HBM every launch); average launch duration = graph time /
    launches."""
    import torch

    from bandwidth_bound_hybrid_gb300 import capi
    L = capi.lib()
    H, E, K, Fe = shape.hidden, shape.n_experts, shape.top_k, shape.expert_ffn
    gen = torch.Generator(device="cuda").manual_seed(5)
    rl = torch.randn(E + 1, device="cuda", generator=gen)
    x = torch.randn(H, device="cuda", generator=gen)
    g = torch.ones(H, device="cuda")
    h = torch.empty((K + 1) * Fe, device="cuda")
    ids = torch.empty(K, dtype=torch.int32, device="cuda")
    wts = torch.empty(K + 1, device="cuda")

    def one(l):
        return lambda s: capi.check(L.hy_op_moe_gateup(
            weights[f"l{l}.exp_gate"].data_ptr(), weights[f"l{l}.exp_up"].data_ptr(),
            weights[f"l{l}.sh_gate"].data_ptr(), weights[f"l{l}.sh_up"].data_ptr(), E, K, Fe, H, rl.data_ptr(),
            x.data_ptr(), g.data_ptr(), 1e-6, h.data_ptr(), ids.data_ptr(), wts.data_ptr(), s), "moe_gateup")

    layers = list(range(shape.n_layers))
    us = graph_us_per_launch([one(l) for l in layers])
    bytes_launch = (K + 1) * 2 * Fe * H * 2 + (E + 1 + 2 * H + (K + 1) * Fe) * 4
    achieved = bytes_launch / (us * 1e-6) / 1e9
    return {"bound": "hbm", "kernel": f"expert gate/up + SwiGLU with in-kernel top-{K} routing (k_gemv, expert rows), "
                                      f"{K} routed + 1 shared experts x 2 x [{Fe}, {H}]",
            "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": load_traffic("moe_gateup", workload), "bytes_per_launch": bytes_launch,
            "launch_us_mean": us, "launches_timed": 5 * len(layers), "peak_source": f"{peak_kind} hbm_gbs"}


def kernel_table(args):
    """Every decode kernel kind of the workload timed on its own: one CUDA
    graph launches it once per layer over that layer's own weights, states or
    caches (distinct buffers cycled so that no launch finds its bytes in L2),
    replayed 5 times; bytes are the algorithmic bytes of one launch.  Plus the
    prompt GEMM (tcgen05) on a 2048-token chunk, in executed TFLOP/s."""
    import torch

    from bandwidth_bound_hybrid_gb300 import accounting as acc
    from bandwidth_bound_hybrid_gb300 import build as hb
    from bandwidth_bound_hybrid_gb300 import capi
    from synth import workloads
    torch.cuda.set_device(0)
    hb.build()
    L = capi.lib()
    w, shape, prompt = workload_of(args)
    peak, peak_kind = load_peaks()
    burst, sustained, tkind = load_tensor_peak()
    weights = workloads.device_weights(shape)
    H, F4 = shape.hidden, acc.F32
    gen = torch.Generator(device="cuda").manual_seed(3)
    rows = []
    gdn_l = [l for l in range(shape.n_layers) if not shape.is_attn(l)]
    att_l = [l for l in range(shape.n_layers) if shape.is_attn(l)]
    x = torch.randn(max(H, 16384), device="cuda", generator=gen)
    g = torch.ones(max(H, 16384), device="cuda")
    y = torch.empty(200000, device="cuda")

    def add(name, kernel, launches, nbytes, note=""):
        us = graph_us_per_launch(launches)
        gbs = nbytes / (us * 1e-6) / 1e9
        rows.append({"kernel": name, "impl": kernel, "launches_in_graph": len(launches), "bytes_per_launch": nbytes,
                     "us_per_launch": us, "gbs": gbs, "frac": gbs / peak, "note": note})

    def gemv(l, name, R, C, norm, acc_):
        return lambda s: capi.check(L.hy_op_gemv(weights[f"l{l}.{name}"].data_ptr(), R, C, x.data_ptr(),
                                                 g.data_ptr() if norm else None, 1e-6, y.data_ptr(), acc_, s), "gemv")

    R = shape.gdn_in_rows
    add(f"input projection, DeltaNet layers [{R}, {H}]", "k_gemv (RMSNorm prologue)",
        [gemv(l, "w_in", R, H, True, 0) for l in gdn_l], acc.linear_bytes(R, H, 0) + (2 * H + R) * F4)
    Ra = (shape.attn_q_heads + 2 * shape.attn_kv_heads) * shape.head_dim
    add(f"input projection, attention layers [{Ra}, {H}]", "k_gemv (RMSNorm prologue)",
        [gemv(l, "w_in", Ra, H, True, 0) for l in att_l], acc.linear_bytes(Ra, H, 0) + (2 * H + Ra) * F4)
    Cg = shape.gdn_heads * shape.gdn_dv
    add(f"output projection + residual, DeltaNet layers [{H}, {Cg}]", "k_gemv (residual epilogue)",
        [gemv(l, "w_o", H, Cg, False, 1) for l in gdn_l], acc.linear_bytes(H, Cg, 0) + (Cg + 2 * H) * F4)
    Ca = shape.attn_q_heads * shape.head_dim
    add(f"output projection + residual, attention layers [{H}, {Ca}]", "k_gemv (residual epilogue)",
        [gemv(l, "w_o", H, Ca, False, 1) for l in att_l], acc.linear_bytes(H, Ca, 0) + (Ca + 2 * H) * F4)
    if shape.ffn > 0:
        Fd = shape.ffn
        hbuf = torch.empty(Fd, device="cuda")

        def gu(l):
            return lambda s: capi.check(L.hy_op_gemv_swiglu(weights[f"l{l}.w_gate"].data_ptr(),
                                                            weights[f"l{l}.w_up"].data_ptr(), Fd, H, x.data_ptr(),
                                                            g.data_ptr(), 1e-6, hbuf.data_ptr(), s), "swiglu")
        lay = list(range(shape.n_layers))
        add(f"RMSNorm + gate/up + SwiGLU 2 x [{Fd}, {H}]", "k_gemv (SwiGLU epilogue)", [gu(l) for l in lay],
            acc.gemv_swiglu_bytes(Fd, H))
        add(f"down projection + residual [{H}, {Fd}]", "k_gemv (residual epilogue)",
            [gemv(l, "w_down", H, Fd, False, 1) for l in lay], acc.linear_bytes(H, Fd, 0) + (Fd + 2 * H) * F4)
    else:
        E, K, Fe = shape.n_experts, shape.top_k, shape.expert_ffn
        lay = list(range(shape.n_layers))
        add(f"router logits [{E + 1}, {H}]", "k_gemv (RMSNorm prologue)",
            [gemv(l, "router", E + 1, H, True, 0) for l in lay], (E + 1) * H * 2 + (2 * H + E + 1) * F4)
        roof = moe_gateup_roofline(shape, weights, peak, peak_kind, args.workload)
        rows.append({"kernel": f"expert gate/up + SwiGLU, {K} routed + shared x 2 x [{Fe}, {H}]",
                     "impl": "k_gemv (expert rows, in-kernel top-k)", "launches_in_graph": len(lay),
                     "bytes_per_launch": roof["bytes_per_launch"], "us_per_launch": roof["launch_us_mean"],
                     "gbs": roof["achieved"], "frac": roof["frac"], "note": ""})
        rl = torch.randn(E + 1, device="cuda", generator=gen)
        hb_ = torch.randn((K + 1) * Fe, device="cuda", generator=gen)
        ids = torch.empty(K, dtype=torch.int32, device="cuda")
        wts = torch.empty(K + 1, device="cuda")
        capi.check(L.hy_op_moe_gateup(weights["l0.exp_gate"].data_ptr(), weights["l0.exp_up"].data_ptr(),
                                      weights["l0.sh_gate"].data_ptr(), weights["l0.sh_up"].data_ptr(), E, K, Fe, H,
                                      rl.data_ptr(), x.data_ptr(), g.data_ptr(), 1e-6, hb_.data_ptr(), ids.data_ptr(),
                                      wts.data_ptr(), None), "moe_gateup")

        def dn(l):
            return lambda s: capi.check(L.hy_op_moe_down(weights[f"l{l}.exp_down"].data_ptr(),
                                                         weights[f"l{l}.sh_down"].data_ptr(), E, K, Fe, H,
                                                         ids.data_ptr(), wts.data_ptr(), hb_.data_ptr(),
                                                         y.data_ptr(), s), "moe_down")
        add(f"expert down + weighted sum + residual, {K} routed + shared x [{H}, {Fe}]",
            "k_gemv (expert segments)", [dn(l) for l in lay],
            (K + 1) * H * Fe * 2 + ((K + 1) * Fe + K + 1 + 2 * H) * F4)
    ws = torch.zeros(L.hy_op_argmax_workspace(), dtype=torch.uint8, device="cuda")
    lg = torch.empty(shape.vocab, device="cuda")
    oid = torch.empty(1, dtype=torch.int32, device="cuda")
    head = lambda s: capi.check(L.hy_op_gemv_argmax(weights["lm_head"].data_ptr(), shape.vocab, H, x.data_ptr(),  # noqa
                                                    g.data_ptr(), 1e-6, lg.data_ptr(), oid.data_ptr(),
                                                    ws.data_ptr(), s), "argmax")
    add(f"final RMSNorm + LM head [{shape.vocab}, {H}] + argmax", "k_gemv (argmax epilogue)", [head] * 4,
        acc.linear_bytes(shape.vocab, H, 0) + (2 * H + shape.vocab) * F4)
    # DeltaNet update: 160 distinct states, more than L2 holds
    nh, dk, dv, K4 = shape.gdn_heads, shape.gdn_dk, shape.gdn_dv, shape.conv_k
    CC = 2 * nh * dk + nh * dv
    ns = max(8, (160 << 20) // (nh * dv * dk * 4))
    S = torch.randn((ns, nh, dv, dk), device="cuda", generator=gen) * 0.01
    ring = torch.zeros((ns, K4, CC), device="cuda")
    cw = weights[f"l{gdn_l[0]}.conv_w"]
    yg = torch.randn(CC + 2 * nh, device="cuda", generator=gen)
    og = torch.empty(nh * dv, device="cuda")
    pos = torch.tensor([5], dtype=torch.int32, device="cuda")

    def gd(i):
        return lambda s: capi.check(L.hy_op_gdn_step(yg.data_ptr(), cw.data_ptr(), ring[i].data_ptr(),
                                                     S[i].data_ptr(), og.data_ptr(), nh, dk, dv, K4, pos.data_ptr(),
                                                     s), "gdn")
    add(f"DeltaNet conv + gates + in-place delta rule, {nh} x {dv} x {dk} FP32 state", "k_gdn",
        [gd(i) for i in range(ns)],
        2 * nh * dv * dk * 4 + (K4 - 1) * CC * 4 + CC * 4 + CC * K4 * 2 + (CC + 2 * nh + nh * dv) * 4)
    del S, ring
    # attention at the workload's context: distinct caches, more than L2 holds
    nq, nkv, hd = shape.attn_q_heads, shape.attn_kv_heads, shape.head_dim
    T = max(prompt, 1)
    cap = T + 8
    per = nkv * cap * hd * 2
    nc = max(4, min(64, (400 << 20) // (2 * per)))
    Kc = torch.randn((nc, nkv, cap, hd), device="cuda", generator=gen).to(torch.bfloat16)
    Vc = torch.randn((nc, nkv, cap, hd), device="cuda", generator=gen).to(torch.bfloat16)
    table = torch.empty((cap, hd // 2, 2), device="cuda")
    capi.check(L.hy_op_rope_table(table.data_ptr(), cap, hd, 1e4, None), "rope")
    ya = torch.randn((nq + 2 * nkv) * hd, device="cuda", generator=gen)
    oa = torch.empty(nq * hd, device="cuda")
    ln = torch.tensor([T], dtype=torch.int32, device="cuda")
    wsa = torch.zeros(L.hy_op_attention_workspace(nq, nkv, hd, args.splits), dtype=torch.uint8, device="cuda")

    def at(i):
        return lambda s: capi.check(L.hy_op_attention(ya.data_ptr(), Kc[i].data_ptr(), Vc[i].data_ptr(), cap, nq, nkv,
                                                      hd, ln.data_ptr(), table.data_ptr(), args.splits, oa.data_ptr(),
                                                      wsa.data_ptr(), s), "attention")
    add(f"split-KV GQA attention {nq}/{nkv} x {hd} at context {T} (RoPE, bf16 KV append, LSE combine)", "k_attn",
        [at(i) for i in range(nc)], 2 * nkv * (T + 1) * hd * 2 + ((nq + 2 * nkv) * hd + nq * hd) * 4)
    del Kc, Vc
    # the prompt GEMM on a 2048-token chunk: the largest projection of the model
    M = 2048
    if shape.ffn > 0:
        N, Kd = shape.ffn, H
        hh = torch.empty((M, N), dtype=torch.int16, device="cuda")
        hl = torch.empty((M, N), dtype=torch.int16, device="cuda")
        xm = torch.randn((M, Kd), device="cuda", generator=gen)
        wsg = torch.empty(L.hy_op_gemm_workspace(M, Kd), dtype=torch.uint8, device="cuda")
        lay = list(range(shape.n_layers))

        def gm(l):
            return lambda s: capi.check(L.hy_op_gemm_swiglu(weights[f"l{l}.w_gate"].data_ptr(),
                                                            weights[f"l{l}.w_up"].data_ptr(), N, Kd, M, xm.data_ptr(),
                                                            Kd, g.data_ptr(), 1e-6, hh.data_ptr(), hl.data_ptr(), N,
                                                            wsg.data_ptr(), s), "gemm")
        us = graph_us_per_launch([gm(l) for l in lay])
        alg = 2.0 * M * (2 * N) * Kd
        rows.append({"kernel": f"prompt GEMM, RMSNorm + gate/up + SwiGLU, {M} tokens x 2 x [{N}, {Kd}] "
                               f"(plus the norm/split pass of the chunk)",
                     "impl": "k_norm_split + k_gemm (tcgen05, TMEM accumulator, TMA tiles)",
                     "launches_in_graph": len(lay), "us_per_launch": us, "tflops_algorithmic": alg / us / 1e6,
                     "tflops_executed": 2 * alg / us / 1e6, "frac_executed_of_sustained": 2 * alg / us / 1e6 / sustained,
                     "note": "activations as bf16 hi + lo parts: the tensor pipe executes twice the algorithmic FLOPs"})
    print(json.dumps({"kernel_table": rows, "workload": w.name, "hbm_peak_gbs": peak, "hbm_peak_source": peak_kind,
                      "bf16_tflops_sustained": sustained, "tensor_peak_source": tkind}), flush=True)
    return 0


def gemv_batch_roofline(shape, weights, B, peak, peak_kind, workload):
    """The batched tensor-core GEMV (k_bgemv) timed alone on the batch step's
    largest launch: MoE shapes, the expert gate/up + SwiGLU over the expected
    union of the batch's picks (round(E (1 - (1 - k/E)^B)) + 1 experts of Fe
    rows, as one dense view of consecutive experts of each layer's tensors);
    dense shapes, the input projections.  One graph launches it once per layer
    (every launch streams fresh weights from HBM); average launch duration =
    graph time / launches."""
    import torch

    from bandwidth_bound_hybrid_gb300 import accounting as acc
    from bandwidth_bound_hybrid_gb300 import capi
    from bandwidth_bound_hybrid_gb300.model import _tensor
    L = capi.lib()
    fmt = getattr(shape, "weight_format", 0)
    H = shape.hidden
    x = torch.randn((B, H), device="cuda")
    g = torch.ones(H, device="cuda")
    if shape.ffn == 0:
        u = int(round(acc.expected_union(shape.n_experts, shape.top_k, B))) + 1
        R = u * shape.expert_ffn
        layers = list(range(shape.n_layers))
        pairs = [(_tensor(weights[f"l{l}.exp_gate"]), _tensor(weights[f"l{l}.exp_up"])) for l in layers]
        what = f"expert gate/up + SwiGLU over {u} experts, [{R}, {H}] x 2"
        bytes_launch = 2 * acc.linear_bytes(R, H, fmt) + B * (H + R) * acc.F32
    else:
        layers = [l for l in range(shape.n_layers) if not shape.is_attn(l)]
        R = shape.gdn_in_rows
        pairs = [(_tensor(weights[f"l{l}.w_in"]), None) for l in layers]
        what = f"DeltaNet input projections [{R}, {H}]"
        bytes_launch = acc.gemv_batch_bytes(R, H, B, fmt)
    y = torch.empty((B, R), device="cuda")
    side = torch.cuda.Stream()

    def sweep(stream):
        for w, wu in pairs:
            capi.check(L.hy_op_gemv_batch(ctypes.byref(w), ctypes.byref(wu) if wu is not None else None, fmt, R, H, B,
                                          x.data_ptr(), H, g.data_ptr(), 1e-6, y.data_ptr(), R, 0, stream.cuda_stream),
                       "gemv_batch")

    with torch.cuda.stream(side):
        sweep(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        sweep(side)
    graph.replay()
    torch.cuda.synchronize()
    reps = 5
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        graph.replay()
    b.record(st)
    torch.cuda.synchronize()
    launch_s = a.elapsed_time(b) / 1e3 / (reps * len(pairs))
    achieved = bytes_launch / launch_s / 1e9
    del graph
    return {"bound": "hbm", "kernel": f"batched tensor-core GEMV (k_bgemv<{fmt}>), {what}, batch {B}",
            "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": load_traffic("gemv_batch", workload), "bytes_per_launch": bytes_launch,
            "launch_us_mean": launch_s * 1e6, "launches_timed": reps * len(pairs),
            "peak_source": f"{peak_kind} hbm_gbs"}


def run_ours_batch(args, w, shape, dist, ws, rank, local):
    """Batch decode: len(contexts) sequences with ragged cached contexts (a
    seeded synthetic cache fill: a step's cost depends on the lengths, not on
    the contents), one step = one token for every sequence."""
    import torch

    from bandwidth_bound_hybrid_gb300 import accounting as acc
    from bandwidth_bound_hybrid_gb300 import capi
    from bandwidth_bound_hybrid_gb300.model import HybridModel
    from synth import workloads
    peak, peak_kind = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream()
    ctx = [int(c) for c in workloads.ragged_contexts(w)]
    B = len(ctx)
    weights = workloads.device_weights(shape)
    caps = [c + args.warmup + 2 * args.steps + 16 for c in ctx]
    flags = capi.HY_FLAG_NO_PDL if args.no_pdl else 0
    pages = None
    if args.paged:  # a pool of 128-token pages holding what the contexts and steps need, not B maximal slabs
        pool = sum((c + args.warmup + 2 * args.steps + 127) // 128 for c in ctx)
        pages = (128, pool)
    model = HybridModel(shape, weights, caps, splits=args.splits, flags=flags, pages=pages)
    for s, c in enumerate(ctx):
        model.fill_synthetic(s, c, seed=s + 1)
    seqs = list(range(B))
    # Each sequence is fed its own seeded uniform token every step (teacher
    # forcing): with synthetic weights, feeding back the greedy ids makes the
    # sequences converge on one token stream, so the batch would route
    # identically and read 8 experts per layer instead of a real batch's
    # union.  A step's work is otherwise the same whichever tokens it gets.
    n_tok = args.warmup + 2 * args.steps
    tok_np = workloads.host.uniform_ids(w.prompt_seed, workloads.PROMPT_TID, n_tok * B, shape.vocab).reshape(n_tok, B)
    tok_dev = torch.from_numpy(tok_np).to(dev)
    ids = torch.empty(B, dtype=torch.int32, device=dev)
    cursor = [0]

    def step():
        model.decode_batch(seqs, tok_dev[cursor[0]], ids)
        cursor[0] += 1

    t, clk, windows, win = timed_region(args, dist, local, st, step, before_timing=model.experts_read)
    # distinct routed experts the timed steps read per layer (the union of the batch's picks)
    moe_layers = shape.n_layers if shape.ffn == 0 else 0
    realised = model.experts_read() / (moe_layers * args.steps) if moe_layers else None
    assert model.check_device() == 0, "device guard fired"
    n = max(ws, 1)
    value = job_throughput(n, B * args.steps, t)
    mid = [c + args.warmup + args.steps // 2 for c in ctx]
    sb = acc.batch_step_bytes(shape, mid, realised)
    step_gbs = sb.total * args.steps / t / 1e9

    roof = None if args.no_kernel_timing else gemv_batch_roofline(shape, weights, B, peak, peak_kind, args.workload)

    tok_h = torch.from_numpy(tok_np[args.warmup + args.steps:].copy()).pin_memory()  # the next K steps' tokens
    ids_h = torch.zeros(B, dtype=torch.int32).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        model.decode_batch_host(seqs, tok_h[i], ids_h)
    e2e_t = time.perf_counter() - t0
    e2e_t = max_over_ranks(e2e_t, dist, dev)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        c0 = int(round(sum(mid) / B))
        cpu = cpu_baseline_obj(shape, c0, "of one sequence (the oracle runs sequences one at a time) at the batch's "
                                          "mean context")
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "shape": shape.name, "batch": B, "contexts": ctx,
                       "context_fill": "seeded synthetic KV rows and recurrent state (no prompt replay)",
                       "tokens": "seeded uniform ids per sequence and step (teacher forcing)",
                       "weights": "4-bit blocks of 32 + fp16 scale" if getattr(shape, "weight_format", 0) else "bf16",
                       "kv": "bf16", "parallelism": f"replicas x{n}",
                       "kv_layout": f"paged: {pages[1]} pages of 128 positions shared by the batch" if pages
                       else "one slab of its capacity per sequence",
                       "l2": "inputs larger than L2: every step streams GBs of weights and KV through the 129 MB L2"},
            "roofline": roof,
            "step_roofline": {"bound": "hbm", "bytes_per_step": sb.total, "achieved": step_gbs, "peak": peak,
                              "unit": "GB/s", "frac": step_gbs / peak, "experts_per_layer": realised,
                              "experts_per_layer_expected": acc.expected_union(shape.n_experts, shape.top_k, B)
                              if shape.ffn == 0 else None},
            "timing": window_stats(windows, win, args.steps),
            "cpu_baseline": cpu,
            "e2e": {"value": n * B * args.steps / e2e_t, "unit": "tokens/s", "h2d_bytes_per_step": 4 * B,
                    "d2h_bytes_per_step": 4 * B},
            "gpu_launches": model.step_kernels() * args.steps,
            "kernels_per_step": model.step_kernels(),
            "graph_launches_per_token": 1.0 / B,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    model.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel_table:
        return kernel_table(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
