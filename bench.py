#!/usr/bin/env python
"""SFI decode-attention benchmark on GB300.

One bench "step" is one whole SFI decode run of the workload (default: the Llama-3-8B-
shaped layer, batch 4, 32K context, 256 decode steps with boundary-triggered slow steps):
every hot-path row runs inside it (append, dense attention + evidence, Selector, packing,
sparse attention, scheduler). The run is issued by the native driver and replayed as one
CUDA graph. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU: units never exchange data, so N GPUs run N independent replicas (no collective
on the data path); value = all tokens / slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SFI decode-attn tokens/s (slow/fast mix) at 32K/128K; % of HBM roofline"
DATA = "synthetic (seeded counter-based generator, Zipf(1.1) key-norm boost)"
NOMINAL_HBM_GBS = 7900.0     # GB300 HBM3e, nominal
BYTES_PER_ROW = 512          # one K row + one V row of 128 bf16
LOGIT_BYTES = 16             # the slow step's fp32 logits (4 heads) written per position


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama8b_ctx32k_b4")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the dense-only/fast-only modes, the CPU baseline and the other "
                         "workloads")
    ap.add_argument("--also", default="llama8b_ctx128k_l32,ragged_paged_b32,longcot_ctx128k_b8_l32,"
                                      "llama8b_ctx32k_b4_tok",
                    help="comma-separated workloads measured after the headline one")
    return ap.parse_args()


# ----------------------------------------------------------------------------- utilities

class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        time.sleep(0.15)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_record(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on this workload
    and the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, "sparse_long_context_sfi_gb300", "csrc", "attn.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec if rec.get("attn_cu_sha256_16") == h and rec.get("workload") == workload else None


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if n_gpus > 0 else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, world: int) -> float:
    """Slowest rank's value (timing is taken as the max over ranks)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(world: int, tokens_per_step: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput of N independent replicas: every rank's tokens over the slowest
    rank's time."""
    return world * tokens_per_step * steps / (ms_max / 1000.0)


def bytes_model(wl, slow, sel_rows):
    """Algorithmic bytes of every step's attention kernel: dense = KV rows + logits; sparse
    (the fused fast step) = packed rows + window rows (each 512 B of K+V) + the appended row
    (512 B read from the new-token buffer, 512 B written to the cache), plus q/out (small)."""
    cfg = wl.cfg
    per_unit_q = cfg.group * 256 + cfg.group * 128 * 2
    units_per_seq = cfg.n_layers * cfg.n_kv_heads
    dense, sparse = [], []
    for t in range(slow.shape[0]):
        L = wl.len0 + t + 1
        if slow[t].any():
            rows = (L * slow[t]).sum() * units_per_seq
            dense.append(rows * (BYTES_PER_ROW + LOGIT_BYTES) +
                         slow[t].sum() * units_per_seq * per_unit_q)
        else:
            dense.append(0)
        fast = ~slow[t].astype(bool)
        if fast.any():
            n_s = np.minimum(cfg.n_sink, L)
            win = L - np.maximum(n_s, L - cfg.n_window)
            rows = ((sel_rows + win) * fast).sum() * units_per_seq
            sparse.append(rows * BYTES_PER_ROW +
                          fast.sum() * units_per_seq * (per_unit_q + 2 * BYTES_PER_ROW))
        else:
            sparse.append(0)
    return np.array(dense, float), np.array(sparse, float)


# ------------------------------------------------------------------------- reference arm

def oracle_cycle(wl):
    """A bounded sample of the workload for the CPU oracle: one SFI cycle of every unit -- a
    slow decode step, then the fast steps that reuse its selection, as many as the run's own
    schedule has per slow step on average (15 on the 32K batch-4 workload: 16 slow of 256).
    Returns (prepared rows, forced step types [B][steps], steps)."""
    from oracle import decode as odecode
    cfg = wl.cfg
    frac = float(odecode.schedule(wl).mean())
    steps = 1 + max(0, int(round(1.0 / frac)) - 1)
    forced = np.zeros((cfg.batch, steps), np.uint8)
    forced[:, 0] = 1
    return odecode.prepare(wl, steps), forced, steps


def time_oracle_cycles(wl, n_min: int, seconds_min: float = 0.0):
    """Run the oracle cycle at least n_min times and until seconds_min have passed; returns
    the per-cycle seconds and the tokens of one cycle."""
    from oracle import decode as odecode
    prepared, forced, steps = oracle_cycle(wl)
    secs = []
    while len(secs) < n_min or sum(secs) < seconds_min:
        r = odecode.run(wl, steps=steps, prepared=prepared, slow=forced)
        secs.append(float(r["seconds"].sum()))
    return secs, wl.cfg.batch * steps, steps


def run_reference(args, world, rank):
    """The CPU oracle, as it stands, on the host cores. One step = one timed SFI cycle of
    every unit (oracle_cycle): value = tokens of the timed cycles / their seconds."""
    if rank != 0:
        return
    from oracle import decode as odecode
    from synth.configs import WORKLOADS
    from synth.workload import HostWorkload
    wl = HostWorkload(WORKLOADS[args.workload])
    cfg = wl.cfg
    time_oracle_cycles(wl, args.warmup)
    secs, tokens, steps = time_oracle_cycles(wl, args.steps)
    v = tokens * len(secs) / sum(secs)
    cores = os.cpu_count()
    sample = (f"per step: decode steps 0..{steps - 1} of all {wl.n_units} units, step 0 slow and "
              f"{steps - 1} fast (the run's slow:fast mix), {tokens} tokens; "
              f"{len(secs)} timed steps took {sum(secs):.2f} s")
    slow_full = odecode.schedule(wl)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * sum(secs) / len(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": dict(workload_config(wl, int(slow_full.any(axis=0).sum())),
                       parallelism="replicas" if world > 1 else "single"),
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "seconds": sum(secs)},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ------------------------------------------------------------------------------- our arm

def cpu_baseline(wl):
    """The oracle on the host cores over about 10 s of SFI cycles (see oracle_cycle)."""
    secs, tokens, steps = time_oracle_cycles(wl, 2, seconds_min=10.0)
    return {"value": tokens * len(secs) / sum(secs), "unit": "tokens/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{len(secs)} SFI cycles of all {wl.n_units} units (decode steps "
                      f"0..{steps - 1}: step 0 slow, the rest fast), {tokens} tokens each",
            "seconds": float(sum(secs))}


def measure(wl, args, world, dev, stream, k_steps, warmup, extras, clock_index=None,
            dense_only_runs=0, pipeline_runs=0, cold_fast=False, concurrent_runs=0):
    """Time whole decode runs of one workload (CUDA-graph replays), the per-kernel durations
    (event-instrumented replays), and optionally the dense-only / fast-only modes and the
    end-to-end run with host buffers."""
    import torch
    from synth import device as sdev
    cfg = wl.cfg
    st = sdev.make_state(wl, device=dev)
    ins = sdev.DeviceInputs(wl, cfg.steps, dev)
    slow = sdev.schedule(wl, st)                       # [steps][B]
    out = torch.empty((cfg.steps, cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim),
                      dtype=torch.bfloat16, device=dev)
    len0 = st.seq_len.clone()

    def capture(run):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            st.seq_len.copy_(len0)
            run.issue(stream)                      # eager warm-up: builds maps, checks args
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            st.seq_len.copy_(len0)
            run.issue(stream)
        return g

    def run_of(sl, **kw):
        return sdev.DriftingRun(wl, st, sl, ins.q, ins.k_new, ins.v_new, out, ins.model,
                                out_fp32=False, **kw)

    def time_graph(g, k, w):
        with torch.cuda.stream(stream):
            for _ in range(w):
                g.replay()
            torch.cuda.synchronize()
            barrier(world)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(k):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
        barrier(world)
        return allreduce_max(e0.elapsed_time(e1), world)

    res = {}
    tokens_per_run = cfg.batch * cfg.steps
    g_mix = capture(run_of(slow))
    clk = Clocks(clock_index) if clock_index is not None else None
    if clk:
        clk.__enter__()
    ms = time_graph(g_mix, k_steps, warmup)
    if clk:
        clk.__exit__()
        res["clocks"] = clk.summary()
    res["value"] = aggregate_tokens_per_s(world, tokens_per_run, k_steps, ms)
    res["ms_per_run"] = ms / k_steps
    res["tokens_per_run"] = tokens_per_run
    res["slow_steps"] = int(slow.any(axis=1).sum())
    # slow step: dense (with the append fused in), the evidence pass (computed inside the
    # Selector when it runs clustered), select, compact; fast step: one fused kernel
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def slow_launches(n_slow):
        units = cfg.n_layers * n_slow * cfg.n_kv_heads
        bound = int(wl.len0.max()) + cfg.steps - cfg.n_window - cfg.n_sink
        clustered = cfg.group == 4 and -(-bound // 4) <= 33280 and units * 4 <= 2 * sms
        return 3 + (0 if clustered else 1)
    res["launches_per_run"] = int(sum((slow_launches(int(r.sum())) if r.any() else 0) +
                                      (0 if r.all() else 1) for r in slow))
    sel_rows = (st.rows.view(cfg.n_layers, cfg.batch, cfg.n_kv_heads).float().mean(dim=(0, 2))
                .cpu().numpy())

    # live kernel timing: the same run with external event nodes around each slow step's
    # dense kernel, and around each maximal stretch of consecutive fast steps (whose fused
    # fast-step kernels run back to back, overlapped by programmatic dependent launch; the
    # stretch's time divided by its launches is their average duration there)
    is_slow = slow.any(axis=1)
    events = [None] * (2 * cfg.steps)
    groups = []                                    # (first, last) step of each fast stretch
    t = 0
    while t < cfg.steps:
        if is_slow[t]:
            events[2 * t] = torch.cuda.Event(enable_timing=True)
            events[2 * t + 1] = torch.cuda.Event(enable_timing=True)
            t += 1
            continue
        t1 = t
        while t1 + 1 < cfg.steps and not is_slow[t1 + 1]:
            t1 += 1
        events[2 * t] = torch.cuda.Event(enable_timing=True)
        events[2 * t1 + 1] = torch.cuda.Event(enable_timing=True)
        groups.append((t, t1))
        t = t1 + 1
    g_ev = capture(run_of(slow, events=events, concurrent=False))
    reps = 3
    d_dense, d_sparse = [], []                     # (steps, seconds)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g_ev.replay()
            torch.cuda.synchronize()
            for t in np.nonzero(is_slow)[0]:
                d_dense.append(([int(t)], events[2 * t].elapsed_time(events[2 * t + 1]) * 1e-3))
            for a, b in groups:
                d_sparse.append((list(range(a, b + 1)),
                                 events[2 * a].elapsed_time(events[2 * b + 1]) * 1e-3))
    bd, bs = bytes_model(wl, slow.astype(bool), sel_rows)
    peak, _ = measured_peaks()

    def kstats(d, bytes_per):
        if not d:
            return None
        n = sum(len(x[0]) for x in d)
        secs = float(sum(x[1] for x in d))
        byt = float(sum(bytes_per[i] for x in d for i in x[0]))
        avg = secs / n
        gbs = byt / secs / 1e9
        return {"launches_per_run": n // reps, "avg_us": avg * 1e6, "bytes_per_launch": byt / n,
                "achieved_gbs": gbs, "frac_of_peak": gbs / peak,
                "total_us_per_run": secs / reps * 1e6}

    res["kernels"] = {"sfi_dense_decode_attn": kstats(d_dense, bd),
                      "sfi_sparse_decode_attn": kstats(d_sparse, bs)}
    del g_ev

    if extras:
        # end to end through the public API with host buffers
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        hq, hk, hv, ho = pin(ins.q), pin(ins.k_new), pin(ins.v_new), pin(out)
        hq.copy_(ins.q.cpu())
        hk.copy_(ins.k_new.cpu())
        hv.copy_(ins.v_new.cpu())
        h2d = (hq.numel() + hk.numel() + hv.numel()) * 2
        with torch.cuda.stream(stream):
            for i in range(warmup + k_steps):
                if i == warmup:
                    torch.cuda.synchronize()
                    barrier(world)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                ins.q.copy_(hq, non_blocking=True)
                ins.k_new.copy_(hk, non_blocking=True)
                ins.v_new.copy_(hv, non_blocking=True)
                g_mix.replay()
                ho.copy_(out, non_blocking=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record()
            torch.cuda.synchronize()
        ms_e2e = allreduce_max(e0.elapsed_time(e1), world)
        res["e2e"] = {"value": world * tokens_per_run * k_steps / (ms_e2e / 1000.0),
                      "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                      "d2h_bytes_per_step": int(ho.numel() * 2), "ms_per_step": ms_e2e / k_steps}
        # dense-only (the full-KV baseline) and fast-only
        k2 = max(3, k_steps // 4)
        g_dense = capture(run_of(slow, dense_only=True))
        ms_d = time_graph(g_dense, k2, 2)
        del g_dense
        fast_only = np.zeros_like(slow)
        fast_only[0] = 1
        g_fast = capture(run_of(fast_only))
        ms_f = time_graph(g_fast, k2, 2)
        del g_fast
        res["modes"] = {
            "sfi_mix": {"tokens_per_s": res["value"], "ms_per_run": res["ms_per_run"],
                        "slow_steps": res["slow_steps"]},
            "dense_only": {"tokens_per_s": world * tokens_per_run * k2 / (ms_d / 1000.0),
                           "ms_per_run": ms_d / k2},
            "fast_only": {"tokens_per_s": world * tokens_per_run * k2 / (ms_f / 1000.0),
                          "ms_per_run": ms_f / k2, "note": "one slow step at t=0"},
        }
        res["modes"]["sfi_vs_dense_speedup"] = (res["modes"]["sfi_mix"]["tokens_per_s"] /
                                                res["modes"]["dense_only"]["tokens_per_s"])
    if extras:
        # Selector refinements (Soft-NMS, cross-head exclusivity, key-norm prior term) on the
        # last slow step's evidence, timed with events on the stream
        import sparse_long_context_sfi_gb300 as sfi
        st.kv.max_len = int(wl.len0.max()) + cfg.steps
        norms = torch.zeros_like(st.scores)
        refined = torch.empty_like(st.scores)
        bud = sfi.SfiBudget(n_sink=cfg.n_sink, n_window=cfg.n_window, n_select=cfg.n_select,
                            prior_tau=cfg.prior_tau, lambda_=cfg.lam, nms_radius=2,
                            nms_gamma=0.5, excl_mu=0.3, norm_nu=float(1.5 * cfg.head_dim ** 0.5))
        with torch.cuda.stream(stream):
            reps = 10
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            sfi.sfi_key_norms(st.kv, norms, stream=stream)
            sfi.sfi_refine_scores(st.kv, st.scores, norms, bud, refined, stream=stream)
            torch.cuda.synchronize()
            ev[0].record()
            for _ in range(reps):
                sfi.sfi_key_norms(st.kv, norms, stream=stream)
            ev[1].record()
            for _ in range(reps):
                sfi.sfi_refine_scores(st.kv, st.scores, norms, bud, refined, stream=stream)
            ev[2].record()
            torch.cuda.synchronize()
        n_pos = float(sum(int(x) + cfg.steps for x in wl.len0)) * cfg.n_layers * cfg.n_kv_heads
        res["refinements"] = {
            "key_norms_us": ev[0].elapsed_time(ev[1]) * 1e3 / reps,
            "refine_us": ev[1].elapsed_time(ev[2]) * 1e3 / reps,
            "options": "nms_radius 2, nms_gamma 0.5, excl_mu 0.3, norm_nu 1.5 sqrt(D)",
            "key_norms_gbs": n_pos * 256 / (ev[0].elapsed_time(ev[1]) * 1e-3 / reps) / 1e9}
    if dense_only_runs:
        g_dense = capture(run_of(slow, dense_only=True))
        ms_d = time_graph(g_dense, dense_only_runs, 1)
        del g_dense
        res["dense_only"] = {"tokens_per_s": world * tokens_per_run * dense_only_runs / (ms_d / 1000.0),
                             "ms_per_run": ms_d / dense_only_runs}
    if pipeline_runs:
        # the layer-wise asynchronous pipeline: slow steps group of layers by group, the
        # Selector and compaction of each group on a side stream beside the next group's
        # attention; measured for several group sizes (layers per dense launch)
        res["layer_pipeline"] = {}
        for grp in (1, 4, 8):
            if grp > cfg.n_layers:
                continue
            g_pipe = capture(run_of(slow, pipeline=True, pipeline_group=grp))
            ms_p = time_graph(g_pipe, pipeline_runs, 1)
            del g_pipe
            res["layer_pipeline"][f"group_{grp}"] = {
                "tokens_per_s": world * tokens_per_run * pipeline_runs / (ms_p / 1000.0),
                "ms_per_run": ms_p / pipeline_runs, "layers_per_dense_launch": grp}
    mixed_steps = int(sum(1 for r in slow if r.any() and not r.all()))
    if concurrent_runs and mixed_steps:
        # the timed runs issue the fast step of a mixed step's fast sequences on a side stream
        # beside the slow sequences' chain; the same runs on one stream, for comparison
        g_seq = capture(run_of(slow, concurrent=False))
        ms_s = time_graph(g_seq, concurrent_runs, 1)
        del g_seq
        res["one_stream"] = {
            "tokens_per_s": world * tokens_per_run * concurrent_runs / (ms_s / 1000.0),
            "ms_per_run": ms_s / concurrent_runs, "mixed_steps": mixed_steps}
    if cold_fast:
        res["fast_cold"] = fast_step_cold(wl, st, ins, stream, dev, world)
    if extras:
        res["dense_isolated"] = dense_isolated(wl, st, ins, stream, world)
    torch.cuda.synchronize()
    res["device_error"] = int(st.err[0])
    del g_mix
    return res


def dense_isolated(wl, st, ins, stream, world, n=4, k=5, w=2):
    """The dense kernel alone (no evidence), n launches back to back per graph replay on the
    state the timed runs left (every sequence at its final length). In the run each dense
    launch is bracketed by event nodes, which cost it its programmatic-launch overlap; this
    is the kernel's own rate. The cache is far larger than L2, so every launch reads HBM."""
    import torch
    from sparse_long_context_sfi_gb300 import sfi_dense_decode_attn
    cfg = wl.cfg
    out = torch.empty((cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim),
                      dtype=torch.bfloat16, device=st.k.device)
    st.kv.max_len = st.capacity

    def issue():
        for _ in range(n):
            sfi_dense_decode_attn(st.kv, ins.q[0], out, False, None, st.ws, st.ws_bytes,
                                  stream=stream)
    with torch.cuda.stream(stream):
        issue()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        issue()
    with torch.cuda.stream(stream):
        for _ in range(w):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(k):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
    ms = allreduce_max(e0.elapsed_time(e1), world)
    L = st.seq_len.double().cpu().numpy()
    per_unit_q = cfg.group * 256 + cfg.group * 128 * 2
    byt = float(L.sum() * cfg.n_layers * cfg.n_kv_heads * BYTES_PER_ROW +
                cfg.n_layers * cfg.batch * cfg.n_kv_heads * per_unit_q)
    avg = ms * 1e-3 / (k * n)
    peak, _ = measured_peaks()
    del g
    return {"avg_us": avg * 1e6, "bytes_per_launch": byt, "achieved_gbs": byt / avg / 1e9,
            "frac_of_peak": byt / avg / 1e9 / peak,
            "how": f"{n} dense launches (no evidence) back to back per graph replay, {k} replays"}


def fast_step_cold(wl, st, ins, stream, dev, world, per_replica=8, k=10, w=3):
    """The fused fast step with a cold L2. Its working set (packed rows + window) fits in L2
    for small workloads, so consecutive fast steps of one run hit in L2 (the in-run, warm
    figure). Here R copies of the decode state (cache and packed memory, as the timed runs
    left them) take the launches in turn, R chosen so that their per-launch working sets
    together exceed 2x L2: every launch then reads its rows from HBM, as the fast step of
    one layer among many would. Lengths restart 8 positions past the prefill."""
    import math

    import torch
    from sparse_long_context_sfi_gb300 import sfi_fast_decode_step
    from sparse_long_context_sfi_gb300.engine import SfiState
    cfg = wl.cfg
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    len_start = wl.len0.astype(np.int64) + 8
    rows = st.rows.view(cfg.n_layers, cfg.batch, cfg.n_kv_heads).double().cpu().numpy()
    per_unit_q = cfg.group * 256 + cfg.group * 128 * 2

    def launch_bytes(L):                     # L: lengths before the launch's append
        Ln = L + 1
        win = Ln - np.maximum(np.minimum(cfg.n_sink, Ln), Ln - cfg.n_window)
        return float(((rows + win[None, :, None]) * BYTES_PER_ROW).sum() +
                     rows.size * (per_unit_q + 2 * BYTES_PER_ROW))

    per_launch = launch_bytes(len_start)
    R = max(4, math.ceil(2 * l2 / per_launch) + 1)
    reps = [st]
    for _ in range(R - 1):
        r = SfiState(cfg, wl.len0, device=dev, page_table=wl.table, n_pages=wl.n_pages)
        for name in ("k", "v", "kc", "vc", "sel_idx", "sel_cnt", "rows"):
            getattr(r, name).copy_(getattr(st, name))
        reps.append(r)
    start = torch.from_numpy(len_start.astype(np.int32)).to(dev)
    for r in reps:
        r.seq_len.copy_(start)
        r.kv.max_len = r.capacity - 1        # host bound on every length these launches see
    out = torch.empty((cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim),
                      dtype=torch.bfloat16, device=dev)
    n = R * per_replica

    def issue():
        for i in range(n):
            r = reps[i % R]
            t = i % ins.q.shape[0]
            sfi_fast_decode_step(r.kv, r.mem, r.budget, ins.k_new[t], ins.v_new[t], ins.q[t], out,
                                 False, r.ws, r.ws_bytes, stream=stream)

    with torch.cuda.stream(stream):
        issue()                               # eager: builds the maps, checks the arguments
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        issue()
    with torch.cuda.stream(stream):
        for _ in range(w):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(k):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
    ms = allreduce_max(e0.elapsed_time(e1), world)
    err = max(int(r.err[0]) for r in reps)
    # lengths grew by one per launch on each replica; bytes of the middle launch stand in
    mid = launch_bytes(len_start + per_replica * (1 + w + k // 2))
    avg = ms * 1e-3 / (k * n)
    peak, _ = measured_peaks()
    del g, reps
    torch.cuda.empty_cache()
    return {"avg_us": avg * 1e6, "bytes_per_launch": mid, "achieved_gbs": mid / avg / 1e9,
            "frac_of_peak": mid / avg / 1e9 / peak, "replicas": R,
            "working_set_bytes_all_replicas": per_launch * R, "l2_bytes": l2,
            "launches_timed": k * n, "device_error": err}


def kv_bytes(wl) -> int:
    """Bytes of the resident K+V cache of a workload's decode state."""
    cfg = wl.cfg
    if cfg.page_size:
        rows = cfg.n_layers * wl.n_pages * cfg.n_kv_heads * cfg.page_size
    else:
        rows = cfg.n_layers * cfg.batch * cfg.n_kv_heads * (int(wl.len0.max()) + cfg.steps)
    return rows * BYTES_PER_ROW


def data_of(cfg) -> str:
    model = ("Zipf(1.1) key-norm boost" if cfg.key_model == "zipf" else
             "planted heavy hitters" + (", drifting at boundaries" if cfg.drift else ""))
    trig = ("trigger tokens in seeded per-sequence token streams" if cfg.trigger == "tokens"
            else "seeded boundary masks")
    return f"synthetic (seeded counter-based generator; {model}; slow steps from {trig})"


def workload_config(wl, slow_steps: int):
    cfg = wl.cfg
    fast_ws = (cfg.n_layers * cfg.batch * cfg.n_kv_heads *
               (cfg.n_sink + cfg.n_select + cfg.n_window) * BYTES_PER_ROW)
    return {"workload": cfg.name, "layers": cfg.n_layers, "batch": cfg.batch,
            "q_heads": cfg.n_q_heads, "kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim,
            "context": int(wl.len0.max()) if cfg.ctx_lo == cfg.ctx else f"{cfg.ctx_lo}-{cfg.ctx}",
            "paged": bool(cfg.page_size), "decode_steps_per_step": cfg.steps,
            "slow_steps_per_step": slow_steps,
            "trigger": "tokens" if cfg.trigger == "tokens" else "boundary mask",
            "budget": f"{cfg.n_sink} sinks + {cfg.n_window} window + {cfg.n_select} selected",
            "l2": (f"no flush: the {kv_bytes(wl) / 1e6:.0f} MB KV cache is larger than L2 and every "
                   f"slow step streams it from HBM; the fast steps' working set (packed rows + "
                   f"window, up to {fast_ws / 1e6:.1f} MB per launch) is re-read by consecutive "
                   f"fast steps, and stays L2-resident between them when it fits (the in-run, "
                   f"warm figure); roofline.cold times the fast step over replica states whose "
                   f"working sets together exceed 2x L2")}


def main():
    args = parse()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from synth.configs import WORKLOADS
    from synth.workload import HostWorkload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    wl = HostWorkload(WORKLOADS[args.workload])
    res = measure(wl, args, world, dev, stream, args.steps, args.warmup, extras=not args.no_extras,
                  clock_index=local, cold_fast=not args.no_extras)
    torch.cuda.empty_cache()
    others = {}
    if not args.no_extras and args.also:
        for name in [n for n in args.also.split(",") if n and n != args.workload]:
            w2 = HostWorkload(WORKLOADS[name])
            big = w2.cfg.n_layers * w2.cfg.batch * w2.cfg.ctx > 32 * 10 ** 6
            multi = w2.cfg.n_layers > 1
            r2 = measure(w2, args, world, dev, stream, 2 if big else max(3, args.steps // 4),
                         1 if big else 2, extras=False, dense_only_runs=1 if big else 2,
                         pipeline_runs=(1 if big else 2) if multi else 0, cold_fast=not big,
                         concurrent_runs=1 if big else max(3, args.steps // 4))
            others[name] = {"tokens_per_s": r2["value"], "ms_per_run": r2["ms_per_run"],
                            "config": workload_config(w2, r2["slow_steps"]),
                            "kernels": r2["kernels"],
                            "device_error": r2["device_error"]}
            if "dense_only" in r2:
                others[name]["dense_only"] = r2["dense_only"]
                others[name]["sfi_vs_dense_speedup"] = r2["value"] / r2["dense_only"]["tokens_per_s"]
            if "layer_pipeline" in r2:
                others[name]["layer_pipeline"] = r2["layer_pipeline"]
            if "fast_cold" in r2:
                others[name]["fast_step_cold"] = r2["fast_cold"]
            if "one_stream" in r2:
                others[name]["mixed_steps_on_one_stream"] = r2["one_stream"]
            torch.cuda.empty_cache()

    peak, peak_kind = measured_peaks()
    ks = res["kernels"]
    dom_name, dom = max(ks.items(), key=lambda x: -1 if x[1] is None else x[1]["total_us_per_run"])
    traffic = traffic_record(dom_name, args.workload)
    warm = {"achieved": dom["achieved_gbs"], "frac": dom["achieved_gbs"] / peak,
            "avg_launch_us": dom["avg_us"], "bytes_per_launch": dom["bytes_per_launch"],
            "how": "in the timed runs (CUDA events around every slow step's dense kernel and "
                   "every stretch of consecutive fast steps)"}
    cold = None
    if dom_name == "sfi_sparse_decode_attn" and res.get("fast_cold"):
        fc = res["fast_cold"]
        cold = {"achieved": fc["achieved_gbs"], "frac": fc["frac_of_peak"],
                "avg_launch_us": fc["avg_us"], "bytes_per_launch": fc["bytes_per_launch"],
                "how": f"fast steps over {fc['replicas']} replica states taken in turn "
                       f"({fc['working_set_bytes_all_replicas'] / 1e6:.0f} MB of working sets, "
                       f"L2 {fc['l2_bytes'] / 1e6:.0f} MB)"}
    head = cold or warm
    roofline = {"bound": "hbm", "achieved": head["achieved"], "peak": peak, "unit": "GB/s",
                "frac": head["achieved"] / peak, "kernel": dom_name,
                "peak_kind": f"{peak_kind} (hbm_gbs, STREAM-style copy); frac is judged on it",
                "frac_of_nominal": head["achieved"] / NOMINAL_HBM_GBS,
                "nominal_gbs": NOMINAL_HBM_GBS,
                "bytes_per_launch": head["bytes_per_launch"], "avg_launch_us": head["avg_launch_us"],
                "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                "cold": cold, "warm": warm,
                "headline": "cold" if cold else "in-run"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_extras:
        cpu = cpu_baseline(wl)
    if rank == 0:
        line = {
            "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_run"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": data_of(wl.cfg),
            "config": dict(workload_config(wl, res["slow_steps"]),
                           parallelism="replicas" if world > 1 else "single"),
            "roofline": roofline,
            "kernels": ks,
            "dense_isolated": res.get("dense_isolated"),
            "cpu_baseline": cpu,
            "e2e": res.get("e2e"),
            "gpu_launches": res["launches_per_run"] * args.steps,
            "clocks": res.get("clocks"),
            "modes": res.get("modes"),
            "refinements": res.get("refinements"),
            "other_workloads": others,
            "device_error": res["device_error"],
        }
        print(json.dumps(line))


if __name__ == "__main__":
    main()
