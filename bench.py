"""Benchmark of the grouped differential attention hot path on GB300.

One JSON line on rank 0.  A step is one causal prefill of the long-context
3:1 workload (B=1, L=32768, 24 signal + 8 noise heads, d=64, dv=128, 1% of
key positions boosted x4, bf16 I/O; the largest prefill workload) through
gda_attn_fwd; `value` is its throughput in TFLOP/s (causal-pair flop count
below) with the inputs already in HBM.  Side measurements in the same line:
the 3:1 B=4 L=2048 and 4:1 d=128 dv=256 prefills, the 64-sequence split-KV
decode in GB/s of KV cache read (and its fp8 / paged variants), chunked
prefill, the backward passes.  Inputs are synthetic (seeded normal tensors
at the workloads' shapes).

Flop count per causal (query, key) pair: 2 d (h_s + h_n) for the logits of
every signal head and, once per noise head, of the shared noise map, plus
2 * 2 dv h_s for applying both maps to V.  Pairs per sequence: L (L + 1) / 2.
Decode bytes per cached position: 2 (h_s d + h_n d + h_s dv).

`--impl reference` times the float64 CPU oracle instead (the reference arm:
there is no reference implementation to run), each step evaluating a bounded
sample of query rows of the same workload.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "GDA causal prefill TFLOP/s (bf16) and decode HBM GB/s, % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM counters of one ncu capture per kernel, valid while the kernel's
# sources hash to the recorded value
PROFILES = {
    "prefill": (os.path.join(ROOT, "profiles", "prefill_group_counters.json"),
                ["grouped_differential_attention_gb300/csrc/gda_prefill_group.cu",
                 "grouped_differential_attention_gb300/csrc/gda_prefill_common.cuh",
                 "grouped_differential_attention_gb300/csrc/gda_device.cuh"]),
    "decode": (os.path.join(ROOT, "profiles", "decode_split_counters.json"),
               ["grouped_differential_attention_gb300/csrc/gda_decode.cu",
                "grouped_differential_attention_gb300/csrc/gda_device.cuh"]),
}
N_INPUT_SETS = 4          # rotating input copies: 4 x 84 MB > 129 MB of L2


# ------------------------------------------------------------------ helpers --

def prefill_flops(B, L, hs, hn, d, dv, causal=True):
    pairs = B * (L * (L + 1) // 2 if causal else L * L)
    return pairs * (2 * d * (hs + hn) + 4 * dv * hs)


def prefill_min_flops(B, L, hs, hn, d, dv):
    return B * (L * (L + 1) // 2) * (2 * d * (hs + hn) + 2 * dv * hs)


def row_flops(B, rows, hs, hn, d, dv):
    """Causal-pair flops of the listed query rows (all batches and heads)."""
    return sum(B * (i + 1) * (2 * d * (hs + hn) + 4 * dv * hs) for i in rows)


def backward_flops(B, L, hs, hn, d, dv):
    """Algorithmic flops of the backward over the causal pairs: the two logit
    maps (2d per signal and per noise head), dA = dO . v and dV (4dv per
    signal head), dq_sig and dk_sig (4d per signal head), dq_noise and
    dk_noise after summing the group's score gradients (4d per noise head)."""
    pairs = B * L * (L + 1) // 2
    return pairs * (2 * d * (hs + hn) + 4 * dv * hs + 4 * d * hs + 4 * d * hn)


# float32 FMA throughput of the CUDA cores: 152 SMs x 128 lanes x 2 flops x 2.07 GHz
FP32_SIMT_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def decode_bytes(lens, hs, hn, d, dv):
    return int(sum(int(n) for n in lens)) * 2 * (hs * d + hn * d + hs * dv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured (MEASURED_PEAKS.json)"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback (no MEASURED_PEAKS.json)"


def kernel_hash(kind="prefill"):
    h = hashlib.sha256()
    for rel in PROFILES[kind][1]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind="prefill", workload=None):
    """DRAM bytes per launch from the committed ncu summary, if it matches the
    kernel's sources and (when given) the workload."""
    try:
        with open(PROFILES[kind][0]) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, None
    if rec.get("kernel_hash") != kernel_hash(kind):
        return None, None
    if workload is not None and rec.get("workload") != workload:
        return None, None
    return rec.get("dram_bytes_per_launch"), rec.get("workload")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        target = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            target = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            target = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "25"]
        if target:
            cmd += ["-i", target]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (host-side timing reduction only)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# -------------------------------------------------------------- oracle arms --

def oracle_rows_throughput(w, rows_per_sample: int, target_s: float, seed: int = 0):
    """Time the float64 oracle on samples of query rows of workload w (TFLOP/s)."""
    import numpy as np
    import oracle
    from grouped_differential_attention_gb300 import workloads as W
    inp = W.make_prefill_inputs(w, seed=seed)
    rng = np.random.default_rng(1234)
    done_flops, spent, nrows = 0, 0.0, 0
    while spent < target_s:
        rows = sorted(rng.choice(w.L, size=min(rows_per_sample, w.L), replace=False).tolist())
        t0 = time.perf_counter()
        oracle.prefill_rows(*inp, w.lambda_init, rows, causal=w.causal, eps=w.eps)
        spent += time.perf_counter() - t0
        done_flops += row_flops(w.B, rows, w.h_s, w.h_n, w.d, w.dv)
        nrows += len(rows)
    return done_flops / spent / 1e12, nrows, spent, oracle.max_threads()


def run_reference(args, world, rank):
    """The reference arm: the float64 CPU oracle, as it stands, on host cores."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from grouped_differential_attention_gb300 import workloads as W
    w = W.PREFILL_WORKLOADS[args.workload]
    inp = W.make_prefill_inputs(w)
    rng = np.random.default_rng(99)
    rows_per_step = 1

    def step():
        rows = sorted(rng.choice(w.L, size=rows_per_step, replace=False).tolist())
        oracle.prefill_rows(*inp, w.lambda_init, rows, causal=w.causal, eps=w.eps)
        return row_flops(w.B, rows, w.h_s, w.h_n, w.d, w.dv)

    for _ in range(args.warmup):
        step()
    flops = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        flops += step()
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"{rows_per_step} query row(s) per step (all {w.B} sequences x {w.h_s} heads), "
              f"rows drawn uniformly from the {w.L}-row causal workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) tensors at the workload's shapes)",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "h_s": w.h_s, "h_n": w.h_n, "d": w.d,
                   "dv": w.dv, "causal": w.causal, "parallelism": "cpu oracle, OpenMP"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm --

def run_gda(args, world, rank, local):
    import grouped_differential_attention_gb300 as gda
    from grouped_differential_attention_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = W.PREFILL_WORKLOADS[args.workload]
    if w.dtype != "bf16":
        raise SystemExit("bench.py times the bf16 tensor-core path")
    peaks, peak_src = load_peaks()

    # ---- inputs: N_INPUT_SETS rotating copies resident in HBM (weak scaling: seed = rank)
    sets = []
    for s in range(N_INPUT_SETS):
        host = W.make_prefill_inputs(w, seed=rank * 100 + s) if s == 0 else None
        if s == 0:
            base = [t.to(dev) for t in host]
            sets.append(base)
        else:
            sets.append([t.clone() for t in base])
    out = torch.empty((w.B, w.L, w.h_s, w.dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        q1, k1, q2, k2, v, lam = sets[i % N_INPUT_SETS]
        gda.gda_attn_fwd(q1, k1, q2, k2, v, lam, w.lambda_init, causal=w.causal, eps=w.eps,
                         out=out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    gda.gda_device_error(clear=True)

    # ---- timed region: K prefill steps, device time from CUDA events on the launch stream
    sampler = ClockSampler(dev.index)
    time.sleep(0.05)
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    prefill_ms = ev0.elapsed_time(ev1)

    # ---- decode: 64 sequences over bf16 caches of 4096..8192 positions (> L2)
    dw = W.GDA3_DECODE_B64
    dinp = [t.to(dev) for t in W.make_decode_inputs(dw, seed=rank)]
    lens_host = dinp[5].cpu()
    dout = torch.empty((dw.B, dw.h_s, dw.dv), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gda.gda_attn_decode_workspace_size(dw.B, dw.Lcap, dw.h_s, dw.h_n, dw.dv),
                     dtype=torch.uint8, device=dev)

    def dstep():
        gda.gda_attn_decode(*dinp, dw.lambda_init, eps=dw.eps, out=dout, workspace=ws)

    dec_steps = max(20, args.steps // 20)
    for _ in range(max(3, args.warmup // 4)):
        dstep()
    barrier(world)
    torch.cuda.synchronize(dev)
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev2.record(stream)
    for _ in range(dec_steps):
        dstep()
    ev3.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    decode_ms = ev2.elapsed_time(ev3)

    # ---- the same decode over fp8 (e4m3) caches with per-head scales
    d8 = [t.to(dev) for t in W.make_decode_inputs_fp8(dw, seed=rank)]
    d8_bytes = decode_bytes(d8[8].cpu(), dw.h_s, dw.h_n, dw.d, dw.dv) // 2

    def d8step():
        gda.gda_attn_decode_fp8(*d8, dw.lambda_init, eps=dw.eps, out=dout, workspace=ws)

    for _ in range(max(3, args.warmup // 4)):
        d8step()
    torch.cuda.synchronize(dev)
    ev6, ev7 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev6.record(stream)
    for _ in range(dec_steps):
        d8step()
    ev7.record(stream)
    torch.cuda.synchronize(dev)
    d8_ms_step = ev6.elapsed_time(ev7) / dec_steps
    del d8

    # ---- the same decode over paged caches (64-position pages, random page order)
    page_size = 64
    cpu_dec = W.make_decode_inputs(dw, seed=rank)
    k1p, k2p, vp, table = W.page_caches(cpu_dec[2], cpu_dec[3], cpu_dec[4], page_size, seed=rank)
    dpg = [t.to(dev) for t in (cpu_dec[0], cpu_dec[1], k1p, k2p, vp, table, cpu_dec[5], cpu_dec[6])]
    del cpu_dec, k1p, k2p, vp

    def dpstep():
        gda.gda_attn_decode_paged(*dpg, dw.lambda_init, eps=dw.eps, out=dout, workspace=ws)

    for _ in range(max(3, args.warmup // 4)):
        dpstep()
    torch.cuda.synchronize(dev)
    ev8, ev9 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev8.record(stream)
    for _ in range(dec_steps):
        dpstep()
    ev9.record(stream)
    torch.cuda.synchronize(dev)
    dp_ms_step = ev8.elapsed_time(ev9) / dec_steps
    del dpg

    # ---- the same decode over paged fp8 caches
    cpu_d8 = W.make_decode_inputs_fp8(dw, seed=rank)
    k1p8, k2p8, vp8, table8 = W.page_caches(cpu_d8[2], cpu_d8[3], cpu_d8[4], page_size, seed=rank)
    dpg8 = [t.to(dev) for t in (cpu_d8[0], cpu_d8[1], k1p8, k2p8, vp8, cpu_d8[5], cpu_d8[6], cpu_d8[7], table8,
                                cpu_d8[8], cpu_d8[9])]
    del cpu_d8, k1p8, k2p8, vp8

    def dp8step():
        gda.gda_attn_decode_paged_fp8(*dpg8, dw.lambda_init, eps=dw.eps, out=dout, workspace=ws)

    for _ in range(max(3, args.warmup // 4)):
        dp8step()
    torch.cuda.synchronize(dev)
    ev8.record(stream)
    for _ in range(dec_steps):
        dp8step()
    ev9.record(stream)
    torch.cuda.synchronize(dev)
    dp8_ms_step = ev8.elapsed_time(ev9) / dec_steps
    del dpg8

    # ---- the headline workload held to the per-signal-head single-pass kernel (for comparison)
    for i in range(3):
        step_sp = sets[i % N_INPUT_SETS]
        gda.gda_attn_fwd(*step_sp, w.lambda_init, causal=w.causal, eps=w.eps, out=out, flags=gda.GDA_FLAG_SINGLE_PASS)
    torch.cuda.synchronize(dev)
    sp_steps = 10
    eva, evb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    eva.record(stream)
    for i in range(sp_steps):
        gda.gda_attn_fwd(*sets[i % N_INPUT_SETS], w.lambda_init, causal=w.causal, eps=w.eps, out=out,
                         flags=gda.GDA_FLAG_SINGLE_PASS)
    evb.record(stream)
    torch.cuda.synchronize(dev)
    sp_ms = eva.elapsed_time(evb) / sp_steps

    # ---- the 3:1 B=4 L=2048 workload through gda_attn_fwd (rotating input sets, > L2)
    w2 = W.GDA3_PREFILL_L2048
    sets2 = []
    for s_ in range(N_INPUT_SETS):
        if s_ == 0:
            base2 = [t.to(dev) for t in W.make_prefill_inputs(w2, seed=rank * 100 + 7)]
            sets2.append(base2)
        else:
            sets2.append([t.clone() for t in base2])
    out2 = torch.empty((w2.B, w2.L, w2.h_s, w2.dv), dtype=torch.bfloat16, device=dev)

    def step2(i, flags=0):
        q1, k1, q2, k2, v, lam = sets2[i % N_INPUT_SETS]
        gda.gda_attn_fwd(q1, k1, q2, k2, v, lam, w2.lambda_init, causal=w2.causal, eps=w2.eps, out=out2,
                         flags=flags)

    ms2 = {}
    for tag, fl in (("default", 0), ("single_pass", gda.GDA_FLAG_SINGLE_PASS)):
        for i in range(10):
            step2(i, fl)
        torch.cuda.synchronize(dev)
        n2 = 200
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(n2):
            step2(i, fl)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        ms2[tag] = ev0.elapsed_time(ev1) / n2
    fl2 = prefill_flops(w2.B, w2.L, w2.h_s, w2.h_n, w2.d, w2.dv, w2.causal)
    fl2_min = prefill_min_flops(w2.B, w2.L, w2.h_s, w2.h_n, w2.d, w2.dv)
    tf2 = fl2 / (ms2["default"] * 1e-3) / 1e12

    # ---- chunked prefill: 512 new rows continuing a 7680-row cached prefix
    w = w2
    ck_L, ck_Lk = 512, 8192
    g = torch.Generator().manual_seed(rank + 21)
    ck = [torch.randn(w.B, ck_L, w.h_s, w.d, generator=g).to(torch.bfloat16),
          torch.randn(w.B, ck_Lk, w.h_s, w.d, generator=g).to(torch.bfloat16),
          torch.randn(w.B, ck_L, w.h_n, w.d, generator=g).to(torch.bfloat16),
          torch.randn(w.B, ck_Lk, w.h_n, w.d, generator=g).to(torch.bfloat16),
          torch.randn(w.B, ck_Lk, w.h_s, w.dv, generator=g).to(torch.bfloat16)]
    ck = [t.to(dev) for t in ck] + [sets2[0][5]]
    ck_out = torch.empty(w.B, ck_L, w.h_s, w.dv, dtype=torch.bfloat16, device=dev)
    ck_flops = row_flops(w.B, range(ck_Lk - ck_L, ck_Lk), w.h_s, w.h_n, w.d, w.dv)
    for _ in range(5):
        gda.gda_attn_fwd_chunk(*ck, w.lambda_init, eps=w.eps, out=ck_out)
    torch.cuda.synchronize(dev)
    ck_steps = 50
    eva, evb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    eva.record(stream)
    for _ in range(ck_steps):
        gda.gda_attn_fwd_chunk(*ck, w.lambda_init, eps=w.eps, out=ck_out)
    evb.record(stream)
    torch.cuda.synchronize(dev)
    ck_ms = eva.elapsed_time(evb) / ck_steps
    del ck

    # ---- per-launch distribution of the headline kernel: 50 launches, each timed alone
    # (10 warm-up launches first), rotating input sets
    w = W.PREFILL_WORKLOADS[args.workload]
    for i in range(10):
        step(i)
    torch.cuda.synchronize(dev)
    lat_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for i, (a, b) in enumerate(lat_ev):
        a.record(stream)
        step(i)
        b.record(stream)
    torch.cuda.synchronize(dev)
    lat_us = sorted(a.elapsed_time(b) * 1e3 for a, b in lat_ev)

    # ---- the float32 CUDA-core prefill at its own workload (B=1, L=128, 2+2 heads): latency only
    wf = W.DIFF_F32_L128
    f32_in = [t.to(dev) for t in W.make_prefill_inputs(wf)]
    f32_out = torch.empty((wf.B, wf.L, wf.h_s, wf.dv), dtype=torch.float32, device=dev)
    for _ in range(10):
        gda.gda_attn_fwd_f32(*f32_in, wf.lambda_init, causal=wf.causal, eps=wf.eps, out=f32_out)
    torch.cuda.synchronize(dev)
    f32_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for a, b in f32_ev:
        a.record(stream)
        gda.gda_attn_fwd_f32(*f32_in, wf.lambda_init, causal=wf.causal, eps=wf.eps, out=f32_out)
        b.record(stream)
    torch.cuda.synchronize(dev)
    f32_us = sorted(a.elapsed_time(b) * 1e3 for a, b in f32_ev)
    del f32_in, f32_out

    # ---- two-pass prefill (difference map before the value product) on the 3:1 L=2048 inputs
    w = w2
    tp_ws = torch.empty(gda.gda_attn_fwd_2pass_workspace_size(w.B, w.L, w.h_s, w.h_n), dtype=torch.uint8,
                        device=dev)
    tp_out = torch.empty_like(out2)

    def tpstep(i):
        q1, k1, q2, k2, v, lam = sets2[i % N_INPUT_SETS]
        gda.gda_attn_fwd_2pass(q1, k1, q2, k2, v, lam, w.lambda_init, causal=w.causal, eps=w.eps, out=tp_out,
                               workspace=tp_ws)

    for i in range(5):
        tpstep(i)
    torch.cuda.synchronize(dev)
    tp_steps = 50
    eve, evf = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    eve.record(stream)
    for i in range(tp_steps):
        tpstep(i)
    evf.record(stream)
    torch.cuda.synchronize(dev)
    tp_ms = eve.elapsed_time(evf) / tp_steps
    tp_tflops = prefill_flops(w.B, w.L, w.h_s, w.h_n, w.d, w.dv, w.causal) / (tp_ms * 1e-3) / 1e12
    del tp_ws, tp_out

    # ---- the 4:1 d=128 dv=256 prefill through gda_attn_fwd_2pass (caller workspace) and through
    # gda_attn_fwd (single pass, no workspace); one input set of 302 MB (larger than L2)
    w4 = W.GDA4_PREFILL_L8192
    in4 = [t.to(dev) for t in W.make_prefill_inputs(w4, seed=rank + 41)]
    out4 = torch.empty((w4.B, w4.L, w4.h_s, w4.dv), dtype=torch.bfloat16, device=dev)
    ws4 = torch.empty(gda.gda_attn_fwd_2pass_workspace_size(w4.B, w4.L, w4.h_s, w4.h_n), dtype=torch.uint8,
                      device=dev)
    fl4 = prefill_flops(w4.B, w4.L, w4.h_s, w4.h_n, w4.d, w4.dv, w4.causal)
    ms4 = {}
    for tag in ("two_pass", "single_pass"):
        def step4():
            if tag == "two_pass":
                gda.gda_attn_fwd_2pass(*in4, w4.lambda_init, causal=w4.causal, eps=w4.eps, out=out4,
                                       workspace=ws4)
            else:
                gda.gda_attn_fwd(*in4, w4.lambda_init, causal=w4.causal, eps=w4.eps, out=out4)
        for _ in range(3):
            step4()
        torch.cuda.synchronize(dev)
        n4 = 20
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(n4):
            step4()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        ms4[tag] = ev0.elapsed_time(ev1) / n4
    del in4, out4, ws4

    # ---- one attention training step: forward, then the tensor-core backward of its inputs
    w = w2
    tr_in = [t.to(dev) for t in W.make_backward_inputs(w, seed=rank + 61)]
    tr_out = torch.empty((w.B, w.L, w.h_s, w.dv), dtype=torch.bfloat16, device=dev)
    tr_ws = torch.empty(gda.gda_attn_bwd_bf16_workspace_size(w.B, w.L, w.h_s, w.h_n, w.dv), dtype=torch.uint8,
                        device=dev)
    tr_grads = gda.gda_attn_bwd_bf16(*tr_in[:6], w.lambda_init, tr_in[6], causal=w.causal, eps=w.eps,
                                     workspace=tr_ws)

    def trstep():
        gda.gda_attn_fwd(*tr_in[:6], w.lambda_init, causal=w.causal, eps=w.eps, out=tr_out)
        gda.gda_attn_bwd_bf16(*tr_in[:6], w.lambda_init, tr_in[6], causal=w.causal, eps=w.eps, workspace=tr_ws,
                              grads=tr_grads)

    for _ in range(3):
        trstep()
    torch.cuda.synchronize(dev)
    tr_steps = 30
    evi, evj = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evi.record(stream)
    for _ in range(tr_steps):
        trstep()
    evj.record(stream)
    torch.cuda.synchronize(dev)
    tr_ms = evi.elapsed_time(evj) / tr_steps
    del tr_in, tr_out, tr_ws, tr_grads

    # ---- float32 backward (gradients of all six inputs) at the prefill workload's sizes
    bw_in = [t.to(dev) for t in W.make_backward_inputs(w, dtype="f32", seed=rank + 31)]
    bw_ws = torch.empty(gda.gda_attn_bwd_workspace_size(w.B, w.L, w.h_s, w.d, w.dv), dtype=torch.uint8,
                        device=dev)
    bw_grads = None

    def bwstep():
        return gda.gda_attn_bwd(*bw_in[:6], w.lambda_init, bw_in[6], causal=w.causal, eps=w.eps,
                                workspace=bw_ws, grads=bw_grads)

    bw_grads = bwstep()
    for _ in range(3):
        bwstep()
    torch.cuda.synchronize(dev)
    bw_steps = 10
    evc, evd = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evc.record(stream)
    for _ in range(bw_steps):
        bwstep()
    evd.record(stream)
    torch.cuda.synchronize(dev)
    bw_ms = evc.elapsed_time(evd) / bw_steps
    bw_flops = backward_flops(w.B, w.L, w.h_s, w.h_n, w.d, w.dv)
    bw_tflops = bw_flops / (bw_ms * 1e-3) / 1e12
    del bw_in, bw_ws, bw_grads

    # ---- tensor-core bf16 backward at the prefill workload's sizes
    bb_in = [t.to(dev) for t in W.make_backward_inputs(w, seed=rank + 51)]
    bb_ws = torch.empty(gda.gda_attn_bwd_bf16_workspace_size(w.B, w.L, w.h_s, w.h_n, w.dv), dtype=torch.uint8,
                        device=dev)
    bb_grads = gda.gda_attn_bwd_bf16(*bb_in[:6], w.lambda_init, bb_in[6], causal=w.causal, eps=w.eps,
                                     workspace=bb_ws)

    def bbstep():
        gda.gda_attn_bwd_bf16(*bb_in[:6], w.lambda_init, bb_in[6], causal=w.causal, eps=w.eps, workspace=bb_ws,
                              grads=bb_grads)

    for _ in range(3):
        bbstep()
    torch.cuda.synchronize(dev)
    bb_steps = 30
    evg, evh = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evg.record(stream)
    for _ in range(bb_steps):
        bbstep()
    evh.record(stream)
    torch.cuda.synchronize(dev)
    bb_ms = evg.elapsed_time(evh) / bb_steps
    bb_tflops = backward_flops(w.B, w.L, w.h_s, w.h_n, w.d, w.dv) / (bb_ms * 1e-3) / 1e12
    del bb_in, bb_ws, bb_grads

    # ---- lambda re-parameterisation for one layer's heads (launch-latency bound)
    g = torch.Generator().manual_seed(rank + 11)
    lvec = [(0.1 * torch.randn(w.h_s, w.d, generator=g)).to(dev) for _ in range(4)]
    lout = torch.empty(w.h_s, dtype=torch.float32, device=dev)
    lam_steps = 200
    for _ in range(5):
        gda.gda_lambda_reparam(*lvec, w.lambda_init, out=lout)
    torch.cuda.synchronize(dev)
    ev4, ev5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev4.record(stream)
    for _ in range(lam_steps):
        gda.gda_lambda_reparam(*lvec, w.lambda_init, out=lout)
    ev5.record(stream)
    torch.cuda.synchronize(dev)
    lam_us = ev4.elapsed_time(ev5) / lam_steps * 1e3
    clocks = sampler.stop()
    dev_err = gda.gda_device_error(clear=True)
    w = W.PREFILL_WORKLOADS[args.workload]
    del sets2, out2

    # ---- end to end through the public API with pinned host buffers: every step copies its
    # inputs host -> device, runs gda_attn_fwd and copies its output device -> host.  Copies
    # and compute run on three streams with two device buffer sets, so step i's upload and
    # step i-1's download overlap step i-1's / i's compute (an input pipeline); each step's
    # bytes still cross the host link inside the timed region.
    host_in = [t.cpu().pin_memory() for t in sets[0]]
    dev_bufs = [sets[1], sets[2]]
    outs = [out, torch.empty_like(out)]
    host_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_outs[0].numel() * host_outs[0].element_size()
    e2e_steps = max(10, min(args.steps, 200))
    s_up, s_up2, s_run, s_down = (torch.cuda.Stream(dev) for _ in range(4))
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_up2 = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    for e in ev_run + ev_down:
        e.record(stream)

    def e2e_step(i):
        k = i % 2
        # the compute that last read this buffer set is done; the upload is split over two
        # streams (two copy engines): K1 and V on one, the other tensors on the other
        s_up.wait_event(ev_run[k])
        s_up2.wait_event(ev_run[k])
        for j, (hsrc, ddst) in enumerate(zip(host_in, dev_bufs[k])):
            with torch.cuda.stream(s_up2 if j in (1, 4) else s_up):
                ddst.copy_(hsrc, non_blocking=True)
        ev_up[k].record(s_up)
        ev_up2[k].record(s_up2)
        s_run.wait_event(ev_up[k])
        s_run.wait_event(ev_up2[k])
        s_run.wait_event(ev_down[k])               # the output buffer has been read back
        with torch.cuda.stream(s_run):
            q1, k1, q2, k2, v, lam = dev_bufs[k]
            gda.gda_attn_fwd(q1, k1, q2, k2, v, lam, w.lambda_init, causal=w.causal, eps=w.eps, out=outs[k])
        ev_run[k].record(s_run)
        s_down.wait_event(ev_run[k])
        with torch.cuda.stream(s_down):
            host_outs[k].copy_(outs[k], non_blocking=True)
        ev_down[k].record(s_down)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    ev4, ev5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev4.record(s_up)
    for i in range(e2e_steps):
        e2e_step(i)
    s_down.wait_event(ev_up[(e2e_steps - 1) % 2])
    s_down.wait_event(ev_up2[(e2e_steps - 1) % 2])
    s_down.wait_event(ev_run[(e2e_steps - 1) % 2])
    ev5.record(s_down)                             # after the last download: the whole job
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = ev4.elapsed_time(ev5)

    # ---- reduce over ranks (max time), aggregate throughput over all ranks
    prefill_ms = max_over_ranks(prefill_ms, world)
    decode_ms = max_over_ranks(decode_ms, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    if rank != 0:
        return

    flops = prefill_flops(w.B, w.L, w.h_s, w.h_n, w.d, w.dv, w.causal)
    ms_per_step = prefill_ms / args.steps
    value = world * flops * args.steps / (prefill_ms * 1e-3) / 1e12
    per_launch_s = ms_per_step * 1e-3
    achieved = flops / per_launch_s / 1e12
    traffic, traffic_wl = profiled_traffic("prefill", w.name)
    dec_traffic, dec_traffic_wl = profiled_traffic("decode", dw.name)
    dec_bytes = decode_bytes(lens_host, dw.h_s, dw.h_n, dw.d, dw.dv)
    dec_ms_step = decode_ms / dec_steps
    dec_gbs = dec_bytes / (dec_ms_step * 1e-3) / 1e9
    e2e_value = world * flops * e2e_steps / (e2e_ms * 1e-3) / 1e12

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) tensors at the workload's shapes)",
        "config": {
            "workload": w.name, "B": w.B, "L": w.L, "h_s": w.h_s, "h_n": w.h_n, "d": w.d,
            "dv": w.dv, "causal": w.causal, "lambda_init": w.lambda_init,
            "flop_count": "causal pairs x (2d(h_s+h_n) + 4 dv h_s)",
            "flops_per_step": flops,
            "min_flops_per_step": prefill_min_flops(w.B, w.L, w.h_s, w.h_n, w.d, w.dv),
            "l2": f"{N_INPUT_SETS} rotating input sets ({N_INPUT_SETS} x "
                  f"{sum(t.numel() * t.element_size() for t in sets[0]) / 1e6:.0f} MB) > 129 MB L2",
            "parallelism": f"{world} independent replica(s), no collective on the data path",
        },
        "roofline": {
            "kernel": (f"gda_prefill_group_kernel<3, {int((w.L + 127) // 128 <= 28)}>"
                       if (w.d == 64 and w.dv == 128 and w.h_s == 3 * w.h_n) else "gda_prefill_tc_kernel"),
            "bound": "tensor",
            "achieved": achieved,
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"],
            "traffic": traffic,
            "traffic_workload": traffic_wl,
            "peak_source": f"{peak_src}: dense bf16 burst (cuBLAS)",
        },
        "decode": {
            "workload": dw.name,
            "value": dec_gbs,
            "unit": "GB/s",
            "ms_per_step": dec_ms_step,
            "steps": dec_steps,
            "bytes_per_step": dec_bytes,
            "gpu_launches": 2 * dec_steps,
            "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                         "traffic": dec_traffic, "traffic_workload": dec_traffic_wl,
                         "peak_source": f"{peak_src}: HBM copy"},
        },
        "decode_fp8": {"workload": dw.name + " with fp8 e4m3 caches (per-head scales)",
                       "value": d8_bytes / (d8_ms_step * 1e-3) / 1e9, "unit": "GB/s",
                       "ms_per_step": d8_ms_step, "steps": dec_steps, "bytes_per_step": d8_bytes,
                       "speedup_vs_bf16_cache": dec_ms_step / d8_ms_step,
                       "roofline": {"bound": "hbm", "achieved": d8_bytes / (d8_ms_step * 1e-3) / 1e9,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": d8_bytes / (d8_ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"]}},
        "decode_paged": {"workload": dw.name + f" with {page_size}-position pages in random pool order",
                         "value": dec_bytes / (dp_ms_step * 1e-3) / 1e9, "unit": "GB/s",
                         "ms_per_step": dp_ms_step, "steps": dec_steps, "bytes_per_step": dec_bytes,
                         "roofline": {"bound": "hbm", "achieved": dec_bytes / (dp_ms_step * 1e-3) / 1e9,
                                      "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": dec_bytes / (dp_ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"]}},
        "launch_stats": {"kernel": "gda_attn_fwd (grouped kernel at d = 64, dv = 128)", "launches": len(lat_us), "warmup": 10,
                         "us_min": lat_us[0], "us_median": lat_us[len(lat_us) // 2],
                         "us_p90": lat_us[int(0.9 * (len(lat_us) - 1))],
                         "tflops_at_median": flops / (lat_us[len(lat_us) // 2] * 1e-6) / 1e12,
                         "tflops_min_count_at_median": prefill_min_flops(w.B, w.L, w.h_s, w.h_n, w.d, w.dv)
                         / (lat_us[len(lat_us) // 2] * 1e-6) / 1e12,
                         "min_count": "causal pairs x (2d(h_s+h_n) + 2 dv h_s): one product of the difference "
                                      "map with V"},
        "prefill_f32": {"workload": wf.name, "us_median": f32_us[len(f32_us) // 2], "us_min": f32_us[0],
                        "us_p90": f32_us[int(0.9 * (len(f32_us) - 1))], "launches": len(f32_us),
                        "bound": "latency: 64 CTAs of 4 rows walk up to 4 key tiles each (precision path; no "
                                 "roofline claim)"},
        "decode_paged_fp8": {"workload": dw.name + f" with fp8 e4m3 caches in {page_size}-position pages, random "
                                                   "pool order",
                             "value": d8_bytes / (dp8_ms_step * 1e-3) / 1e9, "unit": "GB/s",
                             "ms_per_step": dp8_ms_step, "steps": dec_steps, "bytes_per_step": d8_bytes,
                             "roofline": {"bound": "hbm", "achieved": d8_bytes / (dp8_ms_step * 1e-3) / 1e9,
                                          "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                          "frac": d8_bytes / (dp8_ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"]}},
        "prefill_chunk": {"workload": f"B={w2.B}, {ck_L} new rows after a {ck_Lk - ck_L}-row cached prefix, "
                                      f"{w2.h_s}+{w2.h_n} heads, d={w2.d}, dv={w2.dv}",
                          "value": ck_flops / (ck_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ck_ms,
                          "steps": ck_steps,
                          "roofline": {"bound": "tensor", "achieved": ck_flops / (ck_ms * 1e-3) / 1e12,
                                       "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                       "frac": ck_flops / (ck_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]}},
        "prefill_2pass": {"workload": w2.name + ": pass 1 row log-sum-exp of every signal and noise map, "
                                            "pass 2 one P V product per head with P = A1 - lambda A2",
                          "value": tp_tflops, "unit": "TFLOP/s", "ms_per_step": tp_ms, "steps": tp_steps,
                          "gpu_launches": 2 * tp_steps,
                          "speed_vs_gda_attn_fwd": tp_tflops / tf2,
                          "flops_counted": "the single-pass kernel's algorithmic count, so value ratios are "
                                           "time ratios",
                          "roofline": {"bound": "tensor", "achieved": tp_tflops, "peak": peaks["bf16_tflops"],
                                       "unit": "TFLOP/s", "frac": tp_tflops / peaks["bf16_tflops"]}},
        "prefill_4to1": {"workload": w4.name + " through gda_attn_fwd_2pass (two-pass kernels, caller workspace)",
                         "value": fl4 / (ms4["two_pass"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                         "ms_per_step": ms4["two_pass"], "steps": 20, "gpu_launches": 2 * 20,
                         "gda_attn_fwd_tflops": fl4 / (ms4["single_pass"] * 1e-3) / 1e12,
                         "gda_attn_fwd_ms": ms4["single_pass"],
                         "gda_attn_fwd_kernel": "single pass, dv split over a CTA pair (no workspace)",
                         "roofline": {"bound": "tensor", "achieved": fl4 / (ms4["two_pass"] * 1e-3) / 1e12,
                                      "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                      "frac": fl4 / (ms4["two_pass"] * 1e-3) / 1e12 / peaks["bf16_tflops"]}},
        "headline_single_pass": {"workload": w.name + " through gda_attn_fwd with GDA_FLAG_SINGLE_PASS (noise map "
                                              "recomputed per signal head, P1 and P2 rounded separately)",
                                 "ms_per_step": sp_ms, "steps": sp_steps,
                                 "value": flops / (sp_ms * 1e-3) / 1e12, "unit": "TFLOP/s"},
        "prefill_3to1_L2048": {"workload": w2.name + " through gda_attn_fwd",
                               "value": tf2, "unit": "TFLOP/s", "ms_per_step": ms2["default"], "steps": 200,
                               "tflops_min_count": fl2_min / (ms2["default"] * 1e-3) / 1e12,
                               "single_pass_kernel_ms": ms2["single_pass"],
                               "single_pass_kernel_tflops": fl2 / (ms2["single_pass"] * 1e-3) / 1e12,
                               "l2": f"{N_INPUT_SETS} rotating input sets",
                               "roofline": {"bound": "tensor", "achieved": tf2, "peak": peaks["bf16_tflops"],
                                            "unit": "TFLOP/s", "frac": tf2 / peaks["bf16_tflops"]}},
        "backward_bf16": {"workload": f"tensor-core gradients of q_sig, k_sig, q_noise, k_noise, v, lambda from bf16 "
                                      f"inputs at B={w2.B}, L={w2.L}, {w2.h_s}+{w2.h_n} heads, d={w2.d}, dv={w2.dv}, causal",
                          "value": bb_tflops, "unit": "TFLOP/s", "ms_per_step": bb_ms, "steps": bb_steps,
                          "gpu_launches": 5 * bb_steps,
                          "speedup_vs_f32": bw_ms / bb_ms,
                          "roofline": {"bound": "tensor", "achieved": bb_tflops, "peak": peaks["bf16_tflops"],
                                       "unit": "TFLOP/s", "frac": bb_tflops / peaks["bf16_tflops"]}},
        "train_step": {"workload": f"gda_attn_fwd then gda_attn_bwd_bf16 at B={w2.B}, L={w2.L}, {w2.h_s}+{w2.h_n} heads, "
                                   f"d={w2.d}, dv={w2.dv}, causal",
                       "value": w2.B * w2.L / (tr_ms * 1e-3), "unit": "tokens/s", "ms_per_step": tr_ms,
                       "steps": tr_steps, "gpu_launches": 6 * tr_steps,
                       "tflops": (prefill_flops(w2.B, w2.L, w2.h_s, w2.h_n, w2.d, w2.dv, w2.causal)
                                  + backward_flops(w2.B, w2.L, w2.h_s, w2.h_n, w2.d, w2.dv)) / (tr_ms * 1e-3) / 1e12},
        "backward_f32": {"workload": f"float32 gradients of q_sig, k_sig, q_noise, k_noise, v, lambda at "
                                     f"B={w2.B}, L={w2.L}, {w2.h_s}+{w2.h_n} heads, d={w2.d}, dv={w2.dv}, causal",
                         "value": bw_tflops, "unit": "TFLOP/s", "ms_per_step": bw_ms, "steps": bw_steps,
                         "gpu_launches": 3 * bw_steps,
                         "roofline": {"bound": "alu", "achieved": bw_tflops, "peak": FP32_SIMT_TFLOPS,
                                      "unit": "TFLOP/s", "frac": bw_tflops / FP32_SIMT_TFLOPS,
                                      "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 flops x 2.07 GHz"}},
        "lambda_reparam": {"workload": f"h_s={w2.h_s} heads, d={w2.d}", "us_per_call": lam_us,
                           "calls": lam_steps, "gpu_launches": lam_steps,
                           "bound": "host launch rate: back-to-back calls through the Python binding "
                                    "(16 B x h_s x d read per call)"},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                "host_link_gbs": (h2d + d2h) * e2e_steps / (e2e_ms * 1e-3) / 1e9,
                "pipeline": "upload (two streams), compute and download on separate streams, two device buffer sets"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "device_error_word": dev_err,
    }
    if world == 1:
        cpu_value, nrows, spent, cores = oracle_rows_throughput(w, rows_per_sample=8,
                                                                target_s=args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": cpu_value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{nrows} query rows (all {w.B} sequences x {w.h_s} heads) of the same "
                      f"workload, {spent:.1f} s of float64 oracle time"}
        # the same oracle on one core, a shorter sample
        import oracle
        oracle.set_threads(1)
        one_value, one_rows, one_spent, _ = oracle_rows_throughput(w, rows_per_sample=2,
                                                                   target_s=max(0.5, args.cpu_seconds / 5))
        oracle.set_threads(cores)
        line["cpu_baseline"]["one_core"] = {"value": one_value, "unit": "TFLOP/s", "cores": 1,
                                            "sample": f"{one_rows} query rows, {one_spent:.1f} s"}
    print(json.dumps(line), flush=True)


def main():
    from grouped_differential_attention_gb300 import workloads as W
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["gda", "reference"], default="gda")
    ap.add_argument("--workload", default=W.GDA3_PREFILL_L32768.name,
                    choices=sorted(n for n, x in W.PREFILL_WORKLOADS.items() if x.dtype == "bf16"))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.gpus != world and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gda(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
