#!/usr/bin/env python
"""Decode-step benchmark on GB300: decode tokens/s and achieved HBM GB/s.

Default workload: the 8B-shaped decode step, batch 1, FP16 KV at context 2048
(32 layers, D 4096, 32/8 heads, d 128, F 14336, V 128256; W4 group-32 weights
N(0, 0.02), FP16 LM head, KV N(0, 1), 16-token blocks). Every timed step runs
on its own session holding exactly 2048 prior tokens, so each step is that
workload. The inputs (5.4 GB of weights, 268 MB of KV per session) are far
larger than the 126 MB L2, so no L2 flush is needed between steps.

python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import pool_order  # noqa: E402
from synth.workloads import (DECODE_8B, LLAMA8B, LONG_FP16, LONG_INT4, LONG_INT8, KV_FP16, KV_INT4, KV_INT8,  # noqa
                             PREFILL_8B,
                             Workload, agent_batch, shrink)

METRIC = "decode tokens/s per GB300 and achieved HBM GB/s (% of peak) per decode step"
UNIT = "tokens/s"


def workload_by_name(name: str, seed: int) -> Workload:
    table = {w.name: w for w in (DECODE_8B, LONG_FP16, LONG_INT8, LONG_INT4)}
    if name.startswith("8b-decode-b16-agent"):
        return agent_batch(seed)
    return table[name]


def kv_token_bytes(shape, dt) -> int:
    per_head = {KV_FP16: 2 * shape.head_dim, KV_INT8: shape.head_dim + 2,
                KV_INT4: shape.head_dim // 2 + (shape.head_dim // 32) * 4}[dt]
    return 2 * shape.n_layers * shape.n_kv_heads * per_head


def weight_bytes(shape) -> dict:
    """Algorithmic bytes of each projection (packed codes + fp16 scale/min) and of the fp16 LM head."""
    D, F, R, Hd = shape.hidden, shape.ffn, shape.qkv_rows, shape.n_heads * shape.head_dim
    w4 = lambda n, k: n * (-(-k // 32)) * (16 + 4)
    return {"qkv": w4(R, D), "o_proj": w4(D, Hd), "gate_up": w4(2 * F, D), "down": w4(D, F),
            "lm_head": shape.vocab * D * 2, "norms": (2 * shape.n_layers + 1) * D * 2}


def step_bytes(wl: Workload) -> int:
    """Bytes the step must move: every weight once, the live KV once, the appended KV once."""
    s = wl.shape
    wb = weight_bytes(s)
    w = s.n_layers * (wb["qkv"] + wb["o_proj"] + wb["gate_up"] + wb["down"]) + wb["lm_head"] + wb["norms"]
    kv = kv_token_bytes(s, wl.kv_dtype)
    return w + sum(p * kv for p in wl.prior) + wl.batch * kv


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return None
        sm = [float(r[1]) for r in self.rows if len(r) > 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 8 and r[2].replace(".", "").isdigit()]
        reasons = set()
        for r in self.rows:
            if len(r) > 8:
                for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                   r[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_job(world, elapsed_s: float, units: float):
    """Whole-job throughput: units summed over ranks / slowest rank's time (replicas, weak scaling)."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ============================================================================ oracle (CPU) leg

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


class OracleStep:
    """The oracle running whole decode steps of a workload (every layer, the full LM head), on a chosen
    number of host threads. Every step sees exactly the workload's prior context: the stores are cut back
    to it before each step."""

    def __init__(self, wl: Workload, seed: int):
        import oracle
        import synth
        from tests.helpers import model_cfg, oracle_weights
        self.wl, self.seed = wl, seed
        s = wl.shape
        t0 = time.perf_counter()
        self.w = oracle_weights(s, seed)
        self.cfg = model_cfg(s, wl.kv_dtype)
        self.kvs = []
        L, H, d = s.n_layers, s.n_kv_heads, s.head_dim
        for i, p in enumerate(wl.prior):
            kv = oracle.KV(self.cfg, p + 1)
            for t0_ in range(0, p, 4096):
                n = min(4096, p - t0_)
                k = np.empty((L, n, H, d), np.float16)
                v = np.empty((L, n, H, d), np.float16)
                for l in range(L):
                    k[l] = synth.prior_kv_f16(seed, i, l, "K", n, H, d, tok0=t0_)
                    v[l] = synth.prior_kv_f16(seed, i, l, "V", n, H, d, tok0=t0_)
                kv.append(k, v)
            self.kvs.append(kv)
        self.rope = oracle.rope_table(max(wl.prior) + 2, s.head_dim, s.rope_base)
        self.setup_s = time.perf_counter() - t0

    def step(self, step: int, threads: int = 0) -> float:
        """Seconds of one whole step on `threads` threads (0: every core)."""
        import oracle
        from synth import driver
        x = driver.step_inputs(self.wl, self.seed, step)
        for kv, p in zip(self.kvs, self.wl.prior):
            kv.truncate(p)
        oracle.set_threads(threads)
        try:
            t0 = time.perf_counter()
            oracle.forward(self.cfg, self.w, self.kvs, [1] * self.wl.batch, x, *self.rope)
            return time.perf_counter() - t0
        finally:
            oracle.set_threads(0)


def cpu_cores():
    try:
        import oracle
        return oracle.set_threads(0)
    except Exception:
        try:
            return len(os.sched_getaffinity(0))
        except Exception:
            return os.cpu_count() or 1


def cpu_baseline_leg(wl: Workload, seed: int, timed: int = 3) -> dict:
    """The oracle as it stands on this host: whole steps of the workload on every core (one untimed, then
    `timed` steps; the median is the value), and one whole step on a single thread; the same for the tiny
    one-layer configuration."""
    from synth.workloads import TINY_DECODE
    st = OracleStep(wl, seed)
    st.step(0)
    ts = [st.step(1 + i) for i in range(timed)]
    s_med = statistics.median(ts)
    one = st.step(1 + timed, threads=1)
    tiny = OracleStep(TINY_DECODE, seed)
    tiny.step(0)
    tiny_all = statistics.median([tiny.step(1 + i) for i in range(5)])
    tiny_one = statistics.median([tiny.step(1 + i, threads=1) for i in range(5)])
    cores = cpu_cores()
    return {"value": wl.batch / s_med, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"{timed} whole decode steps of {wl.name} ({wl.shape.n_layers} layers, full "
                       f"{'/'.join(map(str, wl.prior))}-token KV, full {wl.shape.vocab}-row LM head), "
                       f"median; not scaled"),
            "s_per_step": s_med, "s_per_step_all": ts, "cpu_model": cpu_model(),
            "one_thread": {"s_per_step": one, "value": wl.batch / one, "unit": UNIT},
            "tiny": {"workload": TINY_DECODE.name, "us_per_step": tiny_all * 1e6, "cores": cores,
                     "us_per_step_one_thread": tiny_one * 1e6},
            "setup_s": st.setup_s}


def run_reference(args, world, rank):
    """The reference arm: the oracle (the pages print no code to install), whole steps of the workload."""
    if rank != 0:
        return
    wl = workload_by_name(args.workload, args.seed)
    st = OracleStep(wl, args.seed)
    for i in range(args.warmup):
        st.step(i)
    ts = [st.step(args.warmup + i) for i in range(args.steps)]
    total = sum(ts)
    value = wl.batch * args.steps / total
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) KV and inputs)",
            "config": {"workload": wl.name, "batch": wl.batch, "context": list(wl.prior), "kv_dtype": wl.kv_dtype},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} whole decode steps of {wl.name} (every layer, full KV and "
                                       f"LM head), not scaled", "cpu_model": cpu_model(),
                             "ms_per_step_median": 1e3 * statistics.median(ts)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "setup_s": st.setup_s}
    print(json.dumps(line), flush=True)


# ============================================================================ GPU leg

def traffic_from_profile(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            prof = json.load(f)
        srcs = prof["sources"] if "sources" in prof else [prof["source"]]
        hs = hashlib.sha256()
        for name in srcs:
            hs.update(open(os.path.join(ROOT, "quantized_decode_step_gb300", "csrc", name), "rb").read())
        h = hs.hexdigest()[:16]
        e = prof["kernels"][kernel_key]
        return e["dram_bytes_per_launch"] if e.get("source_sha") == h else None
    except Exception:
        return None


def pct(ms):
    """Median, p10 and p90 of replay times (ms)."""
    a = np.asarray(ms, np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90)),
            "n": int(a.size)}


def replay_times(ctx, stream, sids, lens, x, out, n):
    """Device time of n graph-replayed decode steps, each bracketed by its own CUDA event pair on the
    context's stream; the sessions are cut back to their prior lengths after every step, so each replay
    is the same workload. Steps are enqueued back to back."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record(stream)
        ctx.decode_step(sids, x, out)
        b.record(stream)
        for sid, p in zip(sids, lens):
            ctx.session_truncate(sid, p)
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def open_with_priors(ctx, stream, wl: Workload, seed: int):
    """Open one session per prior context of the workload and append its seeded prior K/V."""
    import torch
    from synth import driver
    sids = []
    with torch.cuda.stream(stream):
        for i, p in enumerate(wl.prior):
            sid = ctx.session_open()
            driver.append_prior(ctx, sid, wl.shape, seed, i, p)
            sids.append(sid)
    stream.synchronize()
    return sids


def clone_weights(src, dst, shape, seed, stream):
    """Load dst with src's weights: every W4 projection read back in W4G32 bytes and loaded packed (no
    second draw and quantisation), the norm gains and the LM head drawn again from the same seed."""
    import torch
    import quantized_decode_step_gb300 as mag
    import synth
    from synth import driver
    with torch.cuda.stream(stream):
        for l in range(shape.n_layers):
            for name, tid in driver.PROJ:
                n, k = driver.proj_shape(shape, name)
                nb = n * (-(-k // 32)) * 20
                buf = torch.empty(nb, dtype=torch.uint8, device="cuda")
                src.debug_read_weights(tid, l, buf, nb)
                dst.load_weights(tid, l, buf, mag.FMT_W4G32, nb)
                stream.synchronize()
            for tag, tid in ((f"L{l}.g1", mag.NORM_ATTN), (f"L{l}.g2", mag.NORM_FFN)):
                g = torch.from_numpy(synth.norm_gain_f16(seed, tag, shape.hidden)).cuda()
                dst.load_weights(tid, l, g, mag.FMT_F16, g.numel() * 2)
        g = torch.from_numpy(synth.norm_gain_f16(seed, "gf", shape.hidden)).cuda()
        dst.load_weights(mag.NORM_FINAL, 0, g, mag.FMT_F16, g.numel() * 2)
        if shape.vocab:
            lm = torch.from_numpy(synth.lm_head_f16(seed, shape.vocab, shape.hidden)).cuda()
            dst.load_weights(mag.LM_HEAD, 0, lm, mag.FMT_F16, lm.numel() * 2)
    stream.synchronize()


def decode_config(ctx, stream, wl: Workload, seed: int, hbm: float, n_replays: int, sids=None) -> dict:
    """One decode configuration on a loaded context: median / p10 / p90 of graph replays, tokens/s and the
    fraction of the measured HBM bandwidth the step's algorithmic bytes reach at the median."""
    import torch
    import synth
    if sids is None:
        sids = open_with_priors(ctx, stream, wl, seed)
    B, shape = wl.batch, wl.shape
    with torch.cuda.stream(stream):
        x = torch.from_numpy(synth.hidden_f16(seed, B, shape.hidden, tag="x.step0")).cuda()
        out = torch.empty((B, shape.vocab or shape.hidden), dtype=torch.float16, device="cuda")
    lens = list(wl.prior)
    replay_times(ctx, stream, sids, lens, x, out, 5)
    ms = replay_times(ctx, stream, sids, lens, x, out, n_replays)
    st = pct(ms)
    sb = step_bytes(wl)
    row = {"workload": wl.name, "batch": B, "kv_dtype": wl.kv_dtype, "replays": st,
           "ms_per_step": st["median"], "tokens_per_s": B / (st["median"] / 1e3), "step_bytes": sb,
           "hbm_gbs": sb / (st["median"] / 1e3) / 1e9, "hbm_frac": sb / (st["median"] / 1e3) / 1e9 / hbm,
           "launches_per_step": ctx.last_step_launches()}
    if wl.shape.vocab == 0:
        row["us_per_step"] = st["median"] * 1e3
    if B > 1 or len(set(wl.prior)) > 1:
        row["context"] = list(wl.prior)
    else:
        row["context"] = wl.prior[0]
    return row


def run_gpu(args, world, rank, local):
    import torch
    import quantized_decode_step_gb300 as mag
    from synth import driver, hidden_f16
    from synth.workloads import TINY_DECODE

    torch.cuda.set_device(local)
    mag.build()
    wl = workload_by_name(args.workload, args.seed)
    if args.layers:
        from dataclasses import replace as _replace
        wl = _replace(wl, name=wl.name + f"-{args.layers}layers", shape=shrink(wl.shape, n_layers=args.layers))
    shape = wl.shape
    hbm, tc, peak_src = measured_peaks()
    e2e_steps = max(3, min(args.steps, 10))
    prof_steps = 3
    B = wl.batch
    # the headline workload's sessions are reused: after every step they are cut back to their prior length
    long_fp16 = None
    if not args.no_configs and wl.name == DECODE_8B.name and not args.layers:
        long_fp16 = LONG_FP16  # same weights, KV precision and pool order: shares the context
    max_ctx = max(wl.prior) + 1 if long_fp16 is None else max(max(wl.prior), max(long_fp16.prior)) + 1
    blocks = sum(-(-(p + 1) // 16) for p in wl.prior)
    if long_fp16 is not None:
        blocks += sum(-(-(p + 1) // 16) for p in long_fp16.prior)
    stream = torch.cuda.Stream()
    order = pool_order(args.seed, blocks) if wl.scattered_pool else None
    cfg = mag.make_config(shape, kv_dtype=wl.kv_dtype, pool_blocks=blocks, max_sessions=B + 1, max_batch=B,
                          max_context=max_ctx, pool_order=order, flags=mag.FLAG_NO_GRAPH if args.eager else 0)
    t_setup = time.time()
    ctx = mag.Context(cfg, stream.cuda_stream)
    with torch.cuda.stream(stream):
        driver.load_weights(ctx, shape, args.seed)
    sids = open_with_priors(ctx, stream, wl, args.seed)
    lens = list(wl.prior)
    with torch.cuda.stream(stream):
        x = torch.from_numpy(hidden_f16(args.seed, B, shape.hidden, tag="x.step0")).cuda()
        width = shape.vocab or shape.hidden
        out = torch.empty((B, width), dtype=torch.float16, device="cuda")
    stream.synchronize()
    t_setup = time.time() - t_setup

    def one_step():
        ctx.decode_step(sids, x, out)
        for sid, p in zip(sids, lens):
            ctx.session_truncate(sid, p)

    # ---- timed region: K steps of the workload
    for _ in range(args.warmup):
        one_step()
    stream.synchronize()
    launches_per_step = ctx.last_step_launches()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            one_step()
        ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        # the distribution over 100 graph replays, each bracketed by its own events
        dist_ms = replay_times(ctx, stream, sids, lens, x, out, 100)
    elapsed_s = ev0.elapsed_time(ev1) / 1e3
    job_s, job_units = reduce_job(world, elapsed_s, B * args.steps)
    value = job_units / job_s
    ms_per_step = 1e3 * elapsed_s / args.steps

    # ---- end to end: host buffers through the C ABI, copies inside the timed region
    x_host = hidden_f16(args.seed, B, shape.hidden, tag="x.step0")
    out_host = np.empty((B, width), np.float16)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        ctx.decode_step_host(sids, x_host, out_host)
        for sid, p in zip(sids, lens):
            ctx.session_truncate(sid, p)
    e2e_s = time.perf_counter() - t0
    e2e_job_s, e2e_units = reduce_job(world, e2e_s, B * e2e_steps)

    # ---- per-kernel device times: the same step launched kernel by kernel with an event pair per launch
    per_kind = {}
    for _ in range(prof_steps):
        for kind, ms in ctx.profile_step(sids, x, out):
            per_kind.setdefault(kind, []).append(ms)
        for sid, p in zip(sids, lens):
            ctx.session_truncate(sid, p)
    stream.synchronize()

    configs = {}
    if rank == 0 and long_fp16 is not None:
        configs = run_configs(args, ctx, stream, hbm, tc)
    prefill = None
    if rank == 0 and not args.no_prefill:
        prefill = run_prefill(args, tc, src=ctx if not args.layers else None)
    ctx.close()
    del ctx
    torch.cuda.empty_cache()
    if rank != 0:
        return
    sb = step_bytes(wl)
    wb = weight_bytes(shape)
    kernel_bytes = {"gate_up": wb["gate_up"], "qkv": wb["qkv"], "o_proj": wb["o_proj"], "down": wb["down"],
                    "lm_head": wb["lm_head"]}
    kern_rows = {}
    for kind, v in per_kind.items():
        per_launch = statistics.mean(v)
        row = {"launches_per_step": len(v) // prof_steps, "ms_per_launch": per_launch,
               "ms_per_step": sum(v) / prof_steps}
        if kind in kernel_bytes:
            row["gbs"] = kernel_bytes[kind] / (per_launch / 1e3) / 1e9
        kern_rows[kind] = row
    dom = "gate_up"
    dom_ms = kern_rows[dom]["ms_per_launch"]
    achieved = kernel_bytes[dom] / (dom_ms / 1e3) / 1e9
    clocks = clk.summary()
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(wl, args.seed)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "data": "synthetic: seeded N(0,0.02) weights quantised to W4 g32, fp16 LM head, N(0,1) KV and inputs",
        "config": {"workload": wl.name, "batch": B, "context": list(wl.prior), "kv_dtype": wl.kv_dtype,
                   "layers": shape.n_layers, "hidden": shape.hidden, "heads": [shape.n_heads, shape.n_kv_heads],
                   "head_dim": shape.head_dim, "ffn": shape.ffn, "vocab": shape.vocab,
                   "l2": "inputs larger than L2 (5.4 GB weights + KV per step), no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "step_bytes": sb, "hbm_gbs_step": sb / (ms_per_step / 1e3) / 1e9,
        "hbm_frac_step": sb / (ms_per_step / 1e3) / 1e9 / hbm,
        "replays": pct(dist_ms),
        "roofline": {"bound": "hbm", "kernel": "W4 gate-up GEMV (RMSNorm + SwiGLU fused), 28672x4096",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": peak_src, "algorithmic_bytes_per_launch": kernel_bytes[dom],
                     "timing": "kernel by kernel (no graph, no programmatic launch), an event pair around each "
                               "launch on the context's stream; mean over the step's 32 launches x 3 steps",
                     "traffic": traffic_from_profile(dom)},
        "kernels": kern_rows,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_units / e2e_job_s, "unit": UNIT, "h2d_bytes_per_step": B * shape.hidden * 2,
                "d2h_bytes_per_step": B * width * 2},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "setup_s": t_setup,
    }
    if configs:
        line["configs"] = configs
    if prefill is not None:
        line["prefill"] = prefill
    print(json.dumps(line), flush=True)


def run_configs(args, ctx_main, stream, hbm, tc) -> dict:
    """Every other decode configuration, each with its own replay distribution: the long FP16 context on
    the headline context; the agent batch (scattered pool), INT8 and INT4 long contexts on contexts loaded
    with the headline context's weights; the tiny one-layer model (latency)."""
    import torch
    import quantized_decode_step_gb300 as mag
    from synth import driver
    from synth.workloads import TINY_DECODE
    res = {}
    t0 = time.time()
    res["long_fp16"] = decode_config(ctx_main, stream, LONG_FP16, args.seed, hbm, 100)
    for key, wl in (("agent_b16", agent_batch(args.seed)), ("long_int8", LONG_INT8), ("long_int4", LONG_INT4)):
        blocks = sum(-(-(p + 1) // 16) for p in wl.prior)
        order = pool_order(args.seed, blocks) if wl.scattered_pool else None
        cfg = mag.make_config(wl.shape, kv_dtype=wl.kv_dtype, pool_blocks=blocks, max_sessions=wl.batch,
                              max_batch=wl.batch, max_context=max(wl.prior) + 1, pool_order=order)
        ctx = mag.Context(cfg, stream.cuda_stream)
        clone_weights(ctx_main, ctx, wl.shape, args.seed, stream)
        res[key] = decode_config(ctx, stream, wl, args.seed, hbm, 100)
        ctx.close()
        del ctx
        torch.cuda.empty_cache()
    with torch.cuda.stream(stream):
        ctx, sids = driver.setup(TINY_DECODE, args.seed, stream=stream.cuda_stream)
    res["tiny"] = decode_config(ctx, stream, TINY_DECODE, args.seed, hbm, 200, sids=sids)
    res["tiny"]["note"] = "L2-resident (0.52 MB): latency, not a bandwidth figure"
    ctx.close()
    res["setup_and_run_s"] = time.time() - t0
    return res


def prefill_flops(shape, prior: int, T: int) -> float:
    """Algorithmic FLOPs of one chunk: 2 T N K over the projections, QK^T and PV over the causal key
    ranges, and the last token's LM head."""
    D, F, d = shape.hidden, shape.ffn, shape.head_dim
    per_layer = shape.qkv_rows * D + D * shape.n_heads * d + 2 * F * D + D * F
    keys = T * (prior + 1) + T * (T - 1) // 2
    attn = 4 * shape.n_heads * d * keys
    return shape.n_layers * (2.0 * T * per_layer + attn) + 2.0 * shape.vocab * D


def run_prefill(args, tc_peak, src=None):
    """The chunked-prefill configuration: 512-token chunks on a session holding the 800-token prior cache
    (cut back to it after every chunk), timed per chunk with CUDA events; then the verify and batched
    prefill legs. Weights come from `src` (the headline context) when given, else from the seed."""
    import torch
    import quantized_decode_step_gb300 as mag
    from synth import driver, hidden_f16

    wl = PREFILL_8B
    if args.layers:
        from dataclasses import replace as _replace
        wl = _replace(wl, name=wl.name + f"-{args.layers}layers", shape=shrink(wl.shape, n_layers=args.layers))
    shape, T, p = wl.shape, wl.chunk, wl.prior[0]
    warm, runs = 3, 20
    n_draft = 4  # the verify leg: drafts checked in one call on a session after its chunk
    n_sess = 5
    blocks = n_sess * -(-(p + T + n_draft) // 16)
    stream = torch.cuda.Stream()
    # max_batch = n_draft: the verify leg runs on the decode kernels, one row per draft
    cfg = mag.make_config(shape, kv_dtype=wl.kv_dtype, pool_blocks=blocks, max_sessions=n_sess,
                          max_batch=n_draft, max_chunk=T, max_context=p + T + n_draft)
    t_setup = time.time()
    ctx = mag.Context(cfg, stream.cuda_stream)
    if src is not None:
        clone_weights(src, ctx, shape, args.seed, stream)
    else:
        with torch.cuda.stream(stream):
            driver.load_weights(ctx, shape, args.seed)
    prior = Workload(wl.name + "-prior", shape, wl.kv_dtype, n_sess, (p,) * n_sess)
    with torch.cuda.stream(stream):
        sids = []
        L, H, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
        k = np.empty((L, p, H, d), np.float16)
        v = np.empty((L, p, H, d), np.float16)
        import synth
        for l in range(L):
            k[l] = synth.prior_kv_f16(args.seed, 0, l, "K", p, H, d)
            v[l] = synth.prior_kv_f16(args.seed, 0, l, "V", p, H, d)
        kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
        for _ in range(prior.batch):
            sid = ctx.session_open()
            ctx.kv_append(sid, p, kt, vt)
            sids.append(sid)
        x = torch.from_numpy(hidden_f16(args.seed, T, shape.hidden, tag="chunk0")).cuda()
        out = torch.empty(shape.vocab or shape.hidden, dtype=torch.float16, device="cuda")
    stream.synchronize()
    del kt, vt
    t_setup = time.time() - t_setup
    sid0 = sids[0]
    for _ in range(warm):
        ctx.prefill_chunk(sid0, T, x, out)
        ctx.session_truncate(sid0, p)
    stream.synchronize()
    launches = ctx.last_step_launches()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
    for a, b in evs:
        a.record(stream)
        ctx.prefill_chunk(sid0, T, x, out)
        b.record(stream)
        ctx.session_truncate(sid0, p)
    stream.synchronize()
    ch = pct([a.elapsed_time(b) for a, b in evs])
    s_chunk = ch["median"] / 1e3
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # verify leg: n_draft draft tokens in one call on a session holding p + T tokens, truncated back after
    # each call so every call sees the same cache
    sid_v = sids[0]
    ctx.prefill_chunk(sid_v, T, x, out)
    base_len = ctx.session_length(sid_v)
    with torch.cuda.stream(stream):
        xv = torch.from_numpy(hidden_f16(args.seed, n_draft, shape.hidden, tag="drafts")).cuda()
        ov = torch.empty((n_draft, shape.vocab or shape.hidden), dtype=torch.float16, device="cuda")
    for _ in range(3):
        ctx.verify_tokens(sid_v, n_draft, xv, ov)
        ctx.session_truncate(sid_v, base_len)
    v_launches = ctx.last_step_launches()
    v_runs = 20
    ev0.record(stream)
    for _ in range(v_runs):
        ctx.verify_tokens(sid_v, n_draft, xv, ov)
        ctx.session_truncate(sid_v, base_len)
    ev1.record(stream)
    ev1.synchronize()
    s_verify = ev0.elapsed_time(ev1) / 1e3 / v_runs
    # batch leg: four sessions of the prior cache take 128 tokens each, in one mag_prefill_batch call and
    # as four mag_prefill_chunk calls (the same 512 rows); sessions are truncated back after every call
    n_b, t_b = 4, T // 4
    bsids = sids[1:1 + n_b]
    with torch.cuda.stream(stream):
        xb = torch.from_numpy(hidden_f16(args.seed, n_b * t_b, shape.hidden, tag="batch")).cuda()
        ob = torch.empty((n_b, shape.vocab or shape.hidden), dtype=torch.float16, device="cuda")

    def one_batch():
        ctx.prefill_batch(bsids, [t_b] * n_b, xb, ob)
        for sid in bsids:
            ctx.session_truncate(sid, p)

    def four_chunks():
        for i, sid in enumerate(bsids):
            ctx.prefill_chunk(sid, t_b, xb[i * t_b:(i + 1) * t_b], ob[i])
        for sid in bsids:
            ctx.session_truncate(sid, p)

    legs = {}
    for name, fn in (("one_call", one_batch), ("separate_calls", four_chunks)):
        fn()
        stream.synchronize()
        ev0.record(stream)
        for _ in range(5):
            fn()
        ev1.record(stream)
        ev1.synchronize()
        legs[name] = ev0.elapsed_time(ev1) / 5
    fl = prefill_flops(shape, p, T)
    st = ctx.memory_stats()
    ctx.close()
    achieved = fl / s_chunk / 1e12
    return {"workload": wl.name, "chunk": T, "prior": p, "ms_per_chunk": s_chunk * 1e3, "chunks": ch,
            "tokens_per_s": T / s_chunk, "algorithmic_tflop_per_chunk": fl / 1e12,
            "roofline": {"bound": "tensor", "scope": "whole chunk (median of the timed chunks)",
                         "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
                         "note": "fp16 kind::f16 at the measured bf16 rate; algorithmic flops only"},
            "launches_per_chunk": launches, "prefill_weight_bytes": st["prefill_weight_bytes"],
            "verify": {"drafts": n_draft, "context": base_len, "ms_per_call": s_verify * 1e3,
                       "tokens_per_s": n_draft / s_verify, "launches_per_call": v_launches},
            "batch": {"sessions": n_b, "tokens_each": t_b, "prior": p, "ms_one_call": legs["one_call"],
                      "ms_separate_calls": legs["separate_calls"]},
            "setup_s": t_setup}


def run_plans(args):
    """Measurement aid for the adaptive plans: decode step time (8B, one session) at short, medium and long
    contexts under every attention launch shape a plan can take (split count x 4-warp or wide blocks),
    each forced in turn; FP16 at 40 .. 19,431 keys, INT8 at 38,863 and INT4 at 77,726. Prints one JSON
    line {"plans": {kv: {shape: {context: ms per step}}}, "presets": ...} and exits."""
    import torch
    import quantized_decode_step_gb300 as mag
    from synth import driver
    mag.build()
    steps = max(args.steps, 8)
    runs = ((KV_FP16, (40, 100, 300, 700, 2048, 8192, 19431)), (KV_INT8, (38863,)), (KV_INT4, (77726,)))
    res = {}
    for dt, lens in runs:
        wl = Workload(f"8b-plans-kv{dt}", LLAMA8B, dt, len(lens), lens)
        ctx, sids = driver.setup(wl, args.seed, extra_tokens=steps + args.warmup + 8)
        x = torch.zeros((1, LLAMA8B.hidden), dtype=torch.float16, device="cuda")
        out = torch.empty((1, LLAMA8B.vocab), dtype=torch.float16, device="cuda")
        table = {}
        for S in (1, 2, 4, 8, 16, 32, 48, 64):
            for wide in (0, 1):
                if (dt != KV_FP16 and S < 8) or (wide and S >= 16):
                    continue  # long contexts: few splits are far off; wide clusters of 16 queue
                ctx.set_adaptive(True, force_plan=1, plan_splits=(S, S, S), plan_wide=(wide,) * 3)
                row = {}
                for sid, n in zip(sids, lens):
                    for _ in range(args.warmup):
                        ctx.decode_step([sid], x, out)
                    torch.cuda.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for _ in range(steps):
                        ctx.decode_step([sid], x, out)
                    e1.record()
                    e1.synchronize()
                    row[n] = round(e0.elapsed_time(e1) / steps, 4)
                    ctx.session_truncate(sid, n)
                table[f"S{S}{'w' if wide else ''}"] = row
                print(f"kv{dt} S{S} wide{wide}", row, file=sys.stderr, flush=True)
        res[f"kv{dt}"] = table
        ctx.close()
        torch.cuda.empty_cache()
    a = mag.adapt_defaults()
    print(json.dumps({"plans": res, "presets": {"splits": list(a.plan_splits), "wide": list(a.plan_wide)},
                      "unit": "ms per decode step", "workload": "8b decode, 1 session; contexts per KV type"}))


def run_timeline(args):
    """Measurement aid: the phases of one decode step of the workload (8B, batch 1, FP16 KV at 2048 by
    default) from the step timeline (mag_debug_timeline: the step's launches made one by one with
    programmatic dependent launch, their blocks stamping the GPU's global timer). Per launch kind, the mean
    over the middle layers of: streaming = the median block's activations staged -> the first block of
    the next launch entering (an SM freed); tail = first to last block of the next launch entering;
    boundary = the last block of the next launch entering -> its median block staged (the wait on this
    launch's completion and the next staging). Attention: entry -> after its wait, -> keys done, -> last
    block's end. Also the step's timeline length against the graph-replayed step. Prints one JSON line."""
    import torch
    import quantized_decode_step_gb300 as mag
    from quantized_decode_step_gb300 import timeline as tl
    from synth import driver, hidden_f16
    mag.build()
    wl = workload_by_name(args.workload, args.seed)
    shape = wl.shape
    ctx, sids = driver.setup(wl, args.seed, extra_tokens=args.warmup + args.steps + 8)
    lens = [ctx.session_length(s) for s in sids]
    x = torch.from_numpy(hidden_f16(args.seed, wl.batch, shape.hidden, tag="x.step0")).cuda()
    out = torch.empty((wl.batch, shape.vocab or shape.hidden), dtype=torch.float16, device="cuda")
    for _ in range(args.warmup):
        ctx.decode_step(sids, x, out)
        for sid, p in zip(sids, lens):
            ctx.session_truncate(sid, p)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        ctx.decode_step(sids, x, out)
        for sid, p in zip(sids, lens):
            ctx.session_truncate(sid, p)
    e1.record()
    e1.synchronize()
    graph_ms = e0.elapsed_time(e1) / args.steps
    recs = torch.zeros((1 << 18, 4), dtype=torch.int64, device="cuda")
    for _ in range(3):  # the last of three
        n = ctx.timeline(sids, x, out, recs)
        for sid, p in zip(sids, lens):
            ctx.session_truncate(sid, p)
    Ls = tl.launches(recs[:min(n, recs.shape[0])].cpu().numpy())
    names = {(shape.qkv_rows // 16, shape.hidden // 64): "qkv",
             (shape.hidden // 16, shape.n_heads * shape.head_dim // 64): "o",
             (2 * shape.ffn // 16, shape.hidden // 64): "gate_up", (shape.hidden // 16, shape.ffn // 64): "down"}
    kinds = []
    for L in Ls:
        cls, a, b, _ = L["kind"]
        kinds.append("attention" if cls == tl.ATTN else names.get((a, b), f"gemv{a}x{b}"))
    us = lambda v: v / 1000.0
    per = {}
    L_ = shape.n_layers
    for i in range(len(Ls) - 1):
        if i < 5 or i > len(Ls) - 7:
            continue  # the middle layers
        e, en = Ls[i]["ev"], Ls[i + 1]["ev"]
        d = per.setdefault(kinds[i], {})
        if Ls[i]["kind"][0] == tl.ATTN:
            d.setdefault("wait_us", []).append(us(e[1][len(e[1]) // 2] - e[0][0]))
            d.setdefault("keys_us", []).append(us(e[2][len(e[2]) // 2] - e[1][len(e[1]) // 2]))
            d.setdefault("merge_us", []).append(us(e[3][-1] - e[2][len(e[2]) // 2]))
            d.setdefault("to_next_ready_us", []).append(us(en[2 if Ls[i + 1]["kind"][0] == tl.GEMV else 1][len(en[0]) // 2] - e[3][-1]))
        else:
            ready = e[2][len(e[2]) // 2]
            nready = en[2 if Ls[i + 1]["kind"][0] == tl.GEMV else 1]
            d.setdefault("streaming_us", []).append(us(en[0][0] - ready))
            d.setdefault("tail_us", []).append(us(en[0][-1] - en[0][0]))
            d.setdefault("boundary_us", []).append(us(nready[len(nready) // 2] - en[0][-1]))
    summary = {k: {m: round(float(np.mean(v)), 2) for m, v in d.items()} for k, d in per.items()}
    qkv = [Ls[i]["ev"][0][0] for i in range(len(Ls)) if kinds[i] == "qkv"]
    first = min(L["ev"][0][0] for L in Ls)
    last = max(max(v[-1] for v in L["ev"].values()) for L in Ls)
    print(json.dumps({"timeline": summary, "layer_us": round(float(np.mean(np.diff(qkv))) / 1000, 2),
                      "layers": L_, "launches": len(Ls), "records": int(n), "span_ms": round((last - first) / 1e6, 4),
                      "graph_step_ms": round(graph_ms, 4), "workload": wl.name,
                      "note": "span_ms: first to last stamp of the timeline step (launched one by one); the LM "
                              "head's streaming is not in span_ms (no stamp after its staging)"}))


def run_elastic(args):
    """Measurement aid for the elastic KV pool: the 8B decode step (one FP16 session, context 2048) with a
    fixed and with an elastic pool, and the elastic pool's own costs: an append that maps a new group
    (one 2 MiB page per layer), and the close that gives groups back. Host wall times around synchronised
    calls. Prints one JSON line and exits."""
    import torch
    import quantized_decode_step_gb300 as mag
    from synth import driver
    mag.build()
    shape, ctx_len, steps = LLAMA8B, 2048, max(args.steps, 8)
    L, H, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
    res = {}
    for name, flags in (("fixed", 0), ("elastic", mag.FLAG_ELASTIC_POOL)):
        cfg = mag.make_config(shape, kv_dtype=KV_FP16, pool_blocks=4 * 8192 // 16, max_sessions=4, max_batch=1,
                              max_context=8192, flags=flags)
        stream = torch.cuda.current_stream()
        ctx = mag.Context(cfg, stream.cuda_stream)
        driver.load_weights(ctx, shape, args.seed)
        sid = ctx.session_open()
        driver.append_prior(ctx, sid, shape, args.seed, 0, ctx_len)
        x = torch.zeros((1, shape.hidden), dtype=torch.float16, device="cuda")
        out = torch.empty((1, shape.vocab), dtype=torch.float16, device="cuda")
        for _ in range(args.warmup):
            ctx.decode_step([sid], x, out)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            ctx.decode_step([sid], x, out)
        e1.record()
        e1.synchronize()
        r = {"ms_per_step": e0.elapsed_time(e1) / steps}
        # appends of 2048 tokens into a second session: every 512 tokens need one more 32-block group
        k = torch.zeros((L, 512, H, d), dtype=torch.float16, device="cuda")
        sid2 = ctx.session_open()
        times = []
        for _ in range(4):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            ctx.kv_append(sid2, 512, k, k)
            torch.cuda.synchronize()
            times.append((time.perf_counter() - t0) * 1e3)
        r["append_512_ms"] = [round(t, 3) for t in times]
        st = ctx.memory_stats()
        r["mapped_mb_before_close"] = st["kv_pool_mapped_bytes"] / 2**20
        t0 = time.perf_counter()
        ctx.session_close(sid2)
        torch.cuda.synchronize()
        ctx.session_close(ctx.session_open())  # the trim that unmaps what the stream has passed
        r["close_and_release_ms"] = round((time.perf_counter() - t0) * 1e3, 3)
        r["mapped_mb_after_close"] = ctx.memory_stats()["kv_pool_mapped_bytes"] / 2**20
        r["group_blocks"] = st["pool_group_blocks"]
        res[name] = r
        ctx.close()
        del k
        torch.cuda.empty_cache()
    print(json.dumps({"elastic_pool": res, "workload": "8b decode, 1 FP16 session, context 2048; appends of "
                      "512 tokens (one 32-block group each) into a second session", "steps": steps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default=DECODE_8B.name)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the chunked-prefill leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other decode configurations (agent batch, long contexts, tiny)")
    ap.add_argument("--eager", action="store_true",
                    help="profiling aid: launch the step's kernels one by one instead of replaying a CUDA graph")
    ap.add_argument("--plans", action="store_true",
                    help="measurement aid: decode step time per attention split count and context, then exit")
    ap.add_argument("--elastic", action="store_true",
                    help="measurement aid: decode step and map / release costs of the elastic KV pool, then exit")
    ap.add_argument("--timeline", action="store_true",
                    help="measurement aid: the phases of one decode step from the device timeline, then exit")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: the same per-layer shapes with fewer layers (not a bench configuration)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    if args.plans:
        run_plans(args)
        return
    if args.elastic:
        run_elastic(args)
        return
    if args.timeline:
        run_timeline(args)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
