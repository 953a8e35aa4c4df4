"""Benchmark of the latent causal attention path on GB300.

One step = one pass of the whole path over the prefill workload
(B=2, T=4096, H=32, d=128, rank=512, bf16): the down-projection
latent = hidden @ w_down of hidden (2,4096,4096), then the causal latent
attention on that latent (query absorption, flash loop over the latent,
value up-projection).  The metric is algorithmic TFLOP/s of the step:
  projection 2*M*model_dim*rank + attention 4*rank*pairs*H + 4*B*T*H*rank*d.
A secondary line measures the bandwidth-bound decode workload (B=64, one
query at t=4095, H=128) in GB/s of algorithmic bytes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own copy of the workload (weak scaling, no
collective on the data path); rank 0 prints one JSON line with the max time
over ranks.  ``--impl reference`` times the float64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "latent-attention TFLOP/s and HBM GB/s on 1 GB300; fraction of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Published per-GPU figures, reported as a second denominator beside the
# measured ones: HBM3e bandwidth about 8 TB/s per GB300; dense BF16 tensor
# throughput 2.25 PFLOP/s per GPU (NVIDIA lists FP16/BF16 tensor throughput of
# 36 PFLOPS per 8 Blackwell Ultra GPUs of an HGX B300 with 2:4 sparsity; dense
# is half of the sparse figure).
SPEC_PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0,
              "source": "NVIDIA Blackwell Ultra (GB300 / HGX B300) specifications: HBM3e 8 TB/s "
                        "per GPU; FP16/BF16 tensor 36 PFLOPS per 8 GPUs with 2:4 sparsity = "
                        "2.25 PFLOP/s dense per GPU"}


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's);
    one all_reduce(MAX) of a scalar, outside the timed regions."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, steps: int, world: int, max_ms: float,
                   scale: float = 1e12) -> float:
    """Whole-job rate: every rank processes its own copy of the workload (weak
    scaling), so the job does world * units per step, over the slowest rank's time."""
    return world * units_per_rank_step * steps / (max_ms * 1e-3) / scale


def load_peaks(device_name=None):
    """The roofline denominators: the measured HBM copy and bf16 GEMM rates of
    this GPU pool when their record is present, complete and taken on the
    same kind of GPU as ``device_name`` (when given), else the fallback
    figures (one earlier GB300 measurement)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        if all(isinstance(p.get(k), (int, float)) and p[k] > 0
               for k in ("hbm_gbs", "bf16_tflops")):
            rec = p.get("gpu_name")
            if device_name is not None and rec and rec != device_name:
                return dict(FALLBACK_PEAKS), f"fallback (the record is for {rec})"
            return p, "measured"
    except (OSError, ValueError, AttributeError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.summarise(self.lines)

    @classmethod
    def summarise(cls, lines):
        """Median SM clock under sampling, the maximum clock and the throttle
        reasons seen active, from nvidia-smi CSV lines in FIELDS order."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def flash_traffic():
    """DRAM bytes per launch of the prefill flash kernel from the committed ncu
    capture, or None when the kernel source changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "flash_prefill_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for name in ("flash_tc.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "latent_causal_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != rec.get("source_sha256_16"):
        return None
    return int(rec["traffic_bytes_per_launch"])


# ------------------------------------------------------------------ oracle timing
_ORACLE_CACHE = {}


def time_oracle(budget_s: float = 15.0, seed_rows: int = 0, literal: bool = True):
    """The float64 oracle (its absorbed form, pinned equal to the literal
    definition) over sampled (b, i) rows of the prefill workload, all heads;
    returns (TFLOP/s of algorithmic work, details)."""
    import numpy as np
    import oracle
    from latent_causal_attention_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS["prefill_bf16"]
    if "prep" not in _ORACLE_CACHE:
        x = make_inputs(w, with_projection=False)
        _ORACLE_CACHE["o"] = oracle.get()
        _ORACLE_CACHE["prep"] = _ORACLE_CACHE["o"].prepare(x["q"], x["kv_latent"], x["w_up_k"],
                                                           x["w_up_v"])
    o, prep = _ORACLE_CACHE["o"], _ORACLE_CACHE["prep"]
    rng = np.random.default_rng(seed_rows)
    cores = os.cpu_count() or 1
    done_rows, flops, t_total = 0, 0.0, 0.0
    while t_total < budget_s:
        rows = [(int(rng.integers(w.B)), int(rng.integers(w.Tq))) for _ in range(cores)]
        t0 = time.perf_counter()
        o.attention_rows(None, None, None, None, w.scale, rows, prepared=prep, form="absorbed")
        t_total += time.perf_counter() - t0
        for (_, i) in rows:
            flops += 4.0 * w.rank * (i + 1) * w.H + 4.0 * w.H * w.rank * w.d
        done_rows += len(rows)
    value = flops / t_total / 1e12
    # the literal form (k and v rebuilt from the latent for every key) on a few
    # rows, for context: the same algorithmic FLOP count over its wall time
    lit_rows, lit_flops, lit_t = 0, 0.0, 0.0
    while literal and lit_t < min(5.0, budget_s / 3):
        row = [(int(rng.integers(w.B)), int(rng.integers(w.Tq)))]
        t0 = time.perf_counter()
        o.attention_rows(None, None, None, None, w.scale, row, prepared=prep, form="literal")
        lit_t += time.perf_counter() - t0
        lit_flops += 4.0 * w.rank * (row[0][1] + 1) * w.H + 4.0 * w.H * w.rank * w.d
        lit_rows += 1
    lit = None if not literal else {
        "value": round(lit_flops / lit_t / 1e12, 6), "unit": "TFLOP/s",
        "sample": f"float64 C oracle, literal form (k, v rebuilt per key), {lit_rows} random "
                  f"(b, i) rows over all i x {w.H} heads in {lit_t:.1f} s"}
    return value, {"kind": "oracle", "cores": cores, "literal_form": lit,
                   "sample": f"float64 C oracle (absorbed form, OpenMP over rows x heads), "
                             f"{done_rows} random (b, i) rows x {w.H} heads of the prefill "
                             f"attention B2 T4096 H32 d128 R512 in {t_total:.1f} s; algorithmic "
                             f"FLOPs of those rows / wall time"}


def _omp_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP loops for the calling thread
    (libgomp's omp_set_num_threads; the oracle library has loaded libgomp)."""
    import ctypes
    try:
        ctypes.CDLL("libgomp.so.1").omp_set_num_threads(int(n))
    except (OSError, AttributeError):
        pass


def _literal_flops(w) -> float:
    """FLOPs of the literal form: k and v rebuilt (R*d multiply-adds each) for
    every causal (query, key) pair and head, plus the q.k and p.v dot products."""
    return (4.0 * w.rank * w.d + 4.0 * w.d) * w.pairs() * w.H


def oracle_table(budget_s: float = 4.0):
    """The float64 oracle on every workload, on this host's cores: the literal
    form (k, v rebuilt per key), the absorbed form (C, pinned equal to it) and
    the explicit numpy brute force (k, v materialised).  Each runs in full
    where that takes a few seconds, else on a random sample of rows (or of
    heads / sequences for the explicit form) timed for about ``budget_s``
    seconds, with the full run's time extrapolated from the sample's rate.
    Rates are algorithmic FLOPs (the metric's count) per second.  Single-core
    times (OpenMP limited to one thread) for the three smaller workloads."""
    import numpy as np
    import oracle
    from oracle import explicit
    from latent_causal_attention_gb300.inputs import WORKLOADS, make_inputs

    o = oracle.get()
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(77)

    def row_flops(w, i):          # algorithmic FLOPs of row (b, i), all heads
        t = w.Tkv - w.Tq + i
        keys = (t + 1) if w.causal else w.Tkv
        return 4.0 * w.rank * keys * w.H + 4.0 * w.H * w.rank * w.d

    def rows_run(w, prep, form, budget):
        """Random (b, i) rows over all i, timed until ``budget`` seconds have
        passed; each call takes one row per core of ONE random head (a slice
        of the prepared inputs), so that a call stays short even where a row
        of every head would take minutes in the literal form."""
        q, lat, wk, wv, (B, Tq, Tkv, H, d, R) = prep
        heads = {}
        n, fl, t = 0, 0.0, 0.0
        while t < budget:
            h = int(rng.integers(H))
            if h not in heads:
                heads[h] = (np.ascontiguousarray(q[:, :, h:h + 1]), lat,
                            np.ascontiguousarray(wk[:, h:h + 1]),
                            np.ascontiguousarray(wv[:, h:h + 1]), (B, Tq, Tkv, 1, d, R))
            rows = [(int(rng.integers(w.B)), int(rng.integers(w.Tq))) for _ in range(cores)]
            t0 = time.perf_counter()
            o.attention_rows(None, None, None, None, w.scale, rows, prepared=heads[h], form=form)
            t += time.perf_counter() - t0
            fl += sum(row_flops(w, i) for _, i in rows) / w.H
            n += len(rows)
        return n, fl, t

    def entry(w, fl_total, seconds, mode, sample):
        return {"mode": mode, "seconds_full": round(seconds, 4),
                "GFLOP_per_s": round(fl_total / seconds / 1e9, 3), "sample": sample}

    table = {}
    full_lit = {"tiny_f32", "proj_f32"}
    full_abs = {"tiny_f32", "proj_f32", "mid_bf16", "decode_bf16"}
    full_exp = {"tiny_f32", "proj_f32", "mid_bf16"}
    for name in ("tiny_f32", "proj_f32", "mid_bf16", "prefill_bf16", "decode_bf16"):
        w = WORKLOADS[name]
        x = make_inputs(w)
        fl = float(w.attention_flops())
        rec = {"algorithmic_GFLOP": round(fl / 1e9, 6),
               "literal_GFLOP": round(_literal_flops(w) / 1e9, 6)}
        args = (x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"])
        if name == "proj_f32":          # the workload starts with the projection
            t0 = time.perf_counter()
            wk2, wv2 = x["w_up_k"].reshape(w.rank, -1), x["w_up_v"].reshape(w.rank, -1)
            o.project(x["hidden"], x["w_down"], wk2, wv2)
            rec["projection"] = {"mode": "full", "seconds": round(time.perf_counter() - t0, 5),
                                 "GFLOP": round(w.projection_flops(with_kv=True) / 1e9, 6)}
        for form, full_set in (("literal", full_lit), ("absorbed", full_abs)):
            fn = o.attention if form == "literal" else o.attention_absorbed
            if name in full_set:
                t0 = time.perf_counter()
                fn(*args, w.scale, w.causal)
                dt = time.perf_counter() - t0
                rec[form] = entry(w, fl, dt, "full", "every output row")
            else:
                prep = o.prepare(*args)
                n, f_s, t_s = rows_run(w, prep, form, budget_s)
                rec[form] = entry(w, fl, fl / (f_s / t_s), "sampled",
                                  f"{n} random (b, i, head) rows in {t_s:.1f} s; full time "
                                  f"extrapolated from their rate")
        # explicit numpy brute force: whole workload, or a subset of heads /
        # sequences with the time scaled to the whole
        if name in full_exp:
            t0 = time.perf_counter()
            explicit.attention(*args, w.scale, w.causal)
            dt = time.perf_counter() - t0
            rec["explicit"] = entry(w, fl, dt, "full", "every output row")
        elif name == "prefill_bf16":
            hs = [0, 9, 21, 31]
            t0 = time.perf_counter()
            for h in hs:
                explicit.attention(x["q"][:, :, h:h + 1], x["kv_latent"], x["w_up_k"][:, h:h + 1],
                                   x["w_up_v"][:, h:h + 1], w.scale, w.causal)
            dt = (time.perf_counter() - t0) * w.H / len(hs)
            rec["explicit"] = entry(w, fl, dt, "sampled",
                                    f"heads {hs} of {w.H}; full time scaled by heads")
        else:
            bs = [0, 21, 42, 63]
            t0 = time.perf_counter()
            for b in bs:
                explicit.attention(x["q"][b:b + 1], x["kv_latent"][b:b + 1], x["w_up_k"],
                                   x["w_up_v"], w.scale, w.causal)
            dt = (time.perf_counter() - t0) * w.B / len(bs)
            rec["explicit"] = entry(w, fl, dt, "sampled",
                                    f"sequences {bs} of {w.B}; full time scaled by sequences")
        table[name] = rec
    # one core: the C oracle's literal and absorbed forms on the small workloads
    single = {}
    _omp_threads(1)
    try:
        for name in ("tiny_f32", "proj_f32", "mid_bf16"):
            w = WORKLOADS[name]
            x = make_inputs(w)
            args = (x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"])
            fl = float(w.attention_flops())
            rec = {}
            for form in ("literal", "absorbed"):
                if name == "mid_bf16":
                    prep = o.prepare(*args)
                    n, f_s, t_s = rows_run(w, prep, form, budget_s / 2)
                    rec[form] = entry(w, fl, fl / (f_s / t_s), "sampled",
                                      f"{n} random (b, i, head) rows, one thread, {t_s:.1f} s; "
                                      f"full time extrapolated")
                else:
                    fn = o.attention if form == "literal" else o.attention_absorbed
                    t0 = time.perf_counter()
                    fn(*args, w.scale, w.causal)
                    rec[form] = entry(w, fl, time.perf_counter() - t0, "full", "one thread")
            single[name] = rec
    finally:
        _omp_threads(cores)
    return {"kind": "oracle", "cores": cores, "workloads": table, "single_core": single,
            "note": "float64 C oracle (OpenMP over rows x heads) and numpy float64 brute force "
                    "(its BLAS threads), on this host's cores; a baseline, not the target"}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    steps = []
    detail = None
    for _ in range(args.warmup):
        time_oracle(budget_s=0.5, seed_rows=123, literal=False)
    for k in range(args.steps):
        v, detail = time_oracle(budget_s=max(1.0, 60.0 / max(args.steps, 1)), seed_rows=k,
                                literal=False)
        steps.append(v)
    value = statistics.mean(steps)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "prefill_bf16: projection (2,4096,4096)@(4096,512) + causal "
                                   "latent attention B2 T4096 H32 d128 rank512 (oracle: sampled "
                                   "rows)", "l2": "n/a (CPU)"},
            "cpu_baseline": {**detail, "value": round(value, 6), "unit": "TFLOP/s"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def run_ours(args, rank: int, world: int):
    import torch
    import torch.distributed as dist

    import latent_causal_attention_gb300 as mla
    from latent_causal_attention_gb300.build import build
    from latent_causal_attention_gb300.inputs import WORKLOADS, make_inputs

    build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks(torch.cuda.get_device_name(dev))

    w = WORKLOADS["prefill_bf16"]
    x = make_inputs(w)
    d = {k: v.to(dev) for k, v in x.items()}
    del d["kv_latent"]                        # the attention consumes the projection's latent
    lat = torch.empty(w.B, w.Tkv, w.rank, device=dev, dtype=torch.bfloat16)
    out = torch.empty(w.B, w.Tq, w.H, w.d, device=dev, dtype=torch.float32)
    ws = torch.empty(max(1, mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank,
                                               torch.bfloat16)), device=dev, dtype=torch.uint8)
    flush = torch.empty(256 * 1024 * 1024, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def step():
        mla.project(d["hidden"], d["w_down"], latent=lat)
        mla.attention(d["q"], lat, d["w_up_k"], d["w_up_v"], w.scale, True, out=out, workspace=ws)

    flops_proj = w.projection_flops()
    flops_attn = w.attention_flops()
    flops_step = flops_proj + flops_attn
    # The prefill attention runs as one fused kernel (no workspace): its
    # algorithmic FLOPs are the whole attention's (absorption, q'.latent,
    # p.latent, value up-projection).  Otherwise the flash kernel does only
    # q'.latent and p.latent.
    fused = mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank, torch.bfloat16) == 0
    flops_flash = flops_attn if fused else 4 * w.rank * w.pairs() * w.H

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(int(vis.split(",")[local]) if vis else local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    launches0 = mla.launch_count()
    for k in range(args.steps):
        flush.zero_()                          # L2 flush between timed steps (outside the events)
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    launches = mla.launch_count() - launches0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    # The same loop again with the library's per-kernel events (caller events
    # recorded around each kernel on the launching stream): the kernels'
    # own durations for the roofline.  Events between kernels end the overlap
    # of a kernel's set-up with its predecessor's tail, so the step time above
    # is taken without them.
    ev = [mla.StageEvents() for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        ev[k].install()
        step()
    torch.cuda.synchronize()
    mla.StageEvents.uninstall()
    clocks = sampler.stop()
    flash_ms = [e.elapsed_ms(1) for e in ev]
    stage_ids = [(4, "projection"), (1, "attention_fused")] if fused else \
        [(4, "projection"), (0, "absorb"), (1, "flash"), (3, "v_up")]
    stages = {name: statistics.mean(e.elapsed_ms(i) for e in ev) for i, name in stage_ids}
    step_ms_median = statistics.median(step_ms)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(flops_step, args.steps, world, total_ms)

    # --- end to end: pinned host inputs -> device -> path -> host result.
    # Every step copies its inputs from pinned host memory and its result back.
    # The copies run on their own streams into / out of double-buffered device
    # tensors, so step k's compute overlaps the input copy of step k+1 and the
    # result copy of step k-1 (host<->device copies in both directions and the
    # kernels run concurrently); the timed region spans the first input copy to
    # the last result copy.
    host = {k: v.pin_memory() for k, v in x.items() if k != "kv_latent"}
    host_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    e2e_steps = max(3, args.steps)
    dbuf = [d, {k_: torch.empty_like(v_) for k_, v_ in d.items()}]
    obuf = [out, torch.empty_like(out)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def ev():
        return torch.cuda.Event()

    def e2e_run(n):
        in_ready = [ev(), ev()]
        in_free = [None, None]          # compute done with input buffer i
        computed = [ev(), ev()]
        out_free = [None, None]         # result copy of output buffer i done
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for k_ in range(n):
            i = k_ & 1
            with torch.cuda.stream(s_in):
                if in_free[i] is not None:
                    s_in.wait_event(in_free[i])
                for name, hv in host.items():
                    dbuf[i][name].copy_(hv, non_blocking=True)
                in_ready[i].record(s_in)
            stream.wait_event(in_ready[i])
            if out_free[i] is not None:
                stream.wait_event(out_free[i])
            mla.project(dbuf[i]["hidden"], dbuf[i]["w_down"], latent=lat)
            mla.attention(dbuf[i]["q"], lat, dbuf[i]["w_up_k"], dbuf[i]["w_up_v"], w.scale, True,
                          out=obuf[i], workspace=ws)
            computed[i].record(stream)
            in_free[i] = ev()
            in_free[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[i])
                host_out[i].copy_(obuf[i], non_blocking=True)
                out_free[i] = ev()
                out_free[i].record(s_out)
        t1.record(s_out)                # the last result copy is the last operation
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    e2e_run(2)
    e2e_ms = e2e_run(e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = job_throughput(flops_step, e2e_steps, world, e2e_ms)

    # --- decode workload (bandwidth-bound): GB/s of algorithmic bytes
    dec = None
    if not args.no_decode:
        wd = WORKLOADS["decode_bf16"]
        dms, dflash = time_attention_only(wd, dev, flush, stream, max(10, args.steps),
                                          max(3, args.warmup))
        nbytes = wd.attention_bytes(out_bytes=4)
        dec = {"workload": "decode_bf16: B64, one query at t=4095 over 4096 latent rows, H128 d128 "
                           "rank512, bf16 in, fp32 out",
               "GB_per_s": round(nbytes / (dms * 1e-3) / 1e9, 1),
               "ms": round(dms, 4), "algorithmic_bytes": nbytes,
               "frac_hbm": round(nbytes / (dms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
               "frac_hbm_spec": round(nbytes / (dms * 1e-3) / 1e9 / SPEC_PEAKS["hbm_gbs"], 4),
               "TFLOP_per_s": round(wd.attention_flops() / (dms * 1e-3) / 1e12, 2),
               "flash_ms": round(dflash, 4),
               "flash_frac_hbm": round(268435456 * 1.0 / (dflash * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                       4)}

    # --- the mid-size prefill workload (rank 256: one CTA per row block, no
    # CTA pair): TFLOP/s of the whole attention, one fused kernel
    mid = None
    if not args.no_mid:
        wm = WORKLOADS["mid_bf16"]
        mms, mflash = time_attention_only(wm, dev, flush, stream, max(10, args.steps),
                                          max(3, args.warmup))
        mid = {"workload": "mid_bf16: causal latent attention B4 T1024 H16 d64 rank256, bf16 in, "
                           "fp32 out",
               "ms": round(mms, 4), "kernel_ms": round(mflash, 4),
               "TFLOP_per_s": round(wm.attention_flops() / (mms * 1e-3) / 1e12, 2),
               "frac_peak": round(wm.attention_flops() / (mms * 1e-3) / 1e12
                                  / peaks["bf16_tflops"], 4),
               "frac_peak_spec": round(wm.attention_flops() / (mms * 1e-3) / 1e12
                                       / SPEC_PEAKS["bf16_tflops"], 4)}

    # --- comparator: the same prefill step with k and v materialised (projection
    # with w_up_k / w_up_v outputs, then attention over explicit k, v)
    expl = None
    if not args.no_explicit:
        kb = torch.empty(w.B, w.Tkv, w.H * w.d, device=dev, dtype=torch.bfloat16)
        vb = torch.empty_like(kb)
        shp = (w.B, w.Tkv, w.H, w.d)

        def xstep():
            lat_, k_, v_ = mla.project(d["hidden"], d["w_down"], d["w_up_k"], d["w_up_v"],
                                       latent=lat)
            mla.explicit_attention(d["q"], k_.reshape(shp), v_.reshape(shp), w.scale, True,
                                   out=out)

        for _ in range(max(3, args.warmup)):
            xstep()
        n = max(5, min(args.steps, 20))
        xs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        xe = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        torch.cuda.synchronize()
        for k_i in range(n):
            flush.zero_()
            xs[k_i].record(stream)
            xstep()
            xe[k_i].record(stream)
        torch.cuda.synchronize()
        xms = statistics.mean(a.elapsed_time(b) for a, b in zip(xs, xe))
        xev = [mla.StageEvents() for _ in range(n)]          # per-kernel times: a second loop
        for k_i in range(n):
            flush.zero_()
            xev[k_i].install()
            xstep()
        torch.cuda.synchronize()
        mla.StageEvents.uninstall()
        xattn = statistics.mean(e.elapsed_ms(1) for e in xev)
        xflops_attn = 4 * w.d * w.pairs() * w.H            # q.k and p.v over d
        expl = {"workload": "prefill_bf16, k and v materialised (bf16) by the projection, then "
                            "attention over explicit k, v",
                "ms_per_step": round(xms, 4),
                "attention_ms": round(xattn, 4),
                "projection_with_kv_ms": round(xms - xattn, 4),
                "TFLOP_per_s_absorbed_count": round(flops_step / (xms * 1e-3) / 1e12, 2),
                "attention_TFLOP_per_s_explicit_count": round(xflops_attn / (xattn * 1e-3) / 1e12,
                                                              2),
                "attention_frac_explicit_count": round(
                    xflops_attn / (xattn * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}

    small = time_small(dev) if not args.no_small else None

    if rank != 0:
        return
    flash_avg = statistics.mean(flash_ms)
    achieved = flops_flash / (flash_avg * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    cpu_val, cpu_detail, otable = (None, None, None)
    if not args.no_cpu_baseline:
        cpu_val, cpu_detail = time_oracle(budget_s=15.0)
        otable = oracle_table(budget_s=4.0)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0, std) inputs of the workload's shapes)",
        "config": {"workload": "prefill_bf16: projection hidden (2,4096,4096) @ w_down (4096,512) "
                               "-> bf16 latent, then causal latent attention B2 T4096 H32 d128 "
                               "rank512, fp32 out",
                   "l2": "flushed between timed steps (256 MiB write, outside the events)",
                   "flops_per_step": flops_step},
        "ms_per_step_median": round(step_ms_median, 4),
        "stages_ms": {k: round(v, 4) for k, v in stages.items()},
        # the same step counted as if k and v were materialised (q.k and p.v over
        # d, plus k = latent w_up_k and v = latent w_up_v once per key): context
        # for the absorbed form's R/d = 4 times larger score work
        "explicit_equivalent": {
            "flops_per_step": flops_proj + 4 * w.d * w.pairs() * w.H
            + 4 * w.B * w.Tkv * w.rank * w.H * w.d,
            "TFLOP_per_s": round((flops_proj + 4 * w.d * w.pairs() * w.H
                                  + 4 * w.B * w.Tkv * w.rank * w.H * w.d)
                                 * args.steps * world / (total_ms * 1e-3) / 1e12, 3)},
        "frac_of_peak_step": round(value / world / peak, 4),
        "roofline": {"bound": "tensor",
                     "kernel": ("flash_persistent_pair_kernel<256, 128> (resident CTA pairs, "
                                "the whole fused attention)") if fused else "flash_packed_kernel",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} bf16 dense (burst)",
                     "peak_spec": SPEC_PEAKS["bf16_tflops"],
                     "frac_spec": round(achieved / SPEC_PEAKS["bf16_tflops"], 4),
                     "peak_spec_source": SPEC_PEAKS["source"],
                     "flops_per_launch": flops_flash, "traffic": flash_traffic(),
                     "traffic_unit": "bytes per launch (ncu dram read + write)"},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "input copy of step k+1 and result copy of step k-1 run on their own "
                           "streams during step k (double-buffered device tensors)"},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "decode": dec,
        "mid": mid,
        "explicit_kv_comparator": expl,
        "small_fp32_latency": small,
    }
    if cpu_val is not None:
        line["cpu_baseline"] = {**cpu_detail, "value": round(cpu_val, 6), "unit": "TFLOP/s"}
        line["oracle_table"] = otable
    print(json.dumps(line), flush=True)


def time_attention_only(w, dev, flush, stream, n: int, warmup: int):
    """Mean CUDA-event time (ms) of one attention call on workload w with its
    inputs resident and the L2 flushed before every call (outside the events),
    and, from a second loop with the library's per-kernel events, the mean
    time of its main attention kernel."""
    import torch

    import latent_causal_attention_gb300 as mla
    from latent_causal_attention_gb300.inputs import make_inputs

    x = {k: v.to(dev) for k, v in make_inputs(w).items()}
    out = torch.empty(w.B, w.Tq, w.H, w.d, device=dev, dtype=torch.float32)
    ws = torch.empty(max(1, mla.workspace_size(w.B, w.Tq, w.Tkv, w.H, w.d, w.rank,
                                               torch.bfloat16)), device=dev, dtype=torch.uint8)

    def call():
        mla.attention(x["q"], x["kv_latent"], x["w_up_k"], x["w_up_v"], w.scale, True,
                      out=out, workspace=ws)

    for _ in range(warmup):
        call()
    s_ = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    e_ = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize()
    for k in range(n):
        flush.zero_()
        s_[k].record(stream)
        call()
        e_[k].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in zip(s_, e_))
    evs = [mla.StageEvents() for _ in range(n)]
    for k in range(n):
        flush.zero_()
        evs[k].install()
        call()
    torch.cuda.synchronize()
    mla.StageEvents.uninstall()
    kernel_ms = statistics.mean(e.elapsed_ms(1) for e in evs)
    return ms, kernel_ms


def time_small(dev, n: int = 200, warmup: int = 20):
    """Latency of the two fp32 workloads, in microseconds per call:
    tiny_f32 (causal attention B2 T32 H4 d16 rank 24) and proj_f32 (projection
    (4,96,256) -> rank 48 -> k, v, then attention H4 d32 on that latent).
    ``device_us``: n back-to-back calls between two CUDA events, inputs
    resident; ``call_us``: median of per-call event pairs; ``e2e_us``: median
    wall time of one call through the public API with the inputs copied in
    from pinned host memory and the result copied back, synchronised."""
    import torch

    import latent_causal_attention_gb300 as mla
    from latent_causal_attention_gb300.inputs import WORKLOADS, make_inputs

    res = {}
    stream = torch.cuda.current_stream(dev)
    for name in ("tiny_f32", "proj_f32"):
        w = WORKLOADS[name]
        x = make_inputs(w)
        if name == "proj_f32":
            x["w_up_k"] = x["w_up_k"].reshape(w.rank, w.H, w.d)
            x["w_up_v"] = x["w_up_v"].reshape(w.rank, w.H, w.d)
        d = {k: v.to(dev) for k, v in x.items()}
        out = torch.empty(w.B, w.Tq, w.H, w.d, device=dev, dtype=torch.float32)
        lat = torch.empty(w.B, w.Tkv, w.rank, device=dev, dtype=torch.float32)

        def call(dd):
            if name == "proj_f32":
                mla.project(dd["hidden"], dd["w_down"], dd["w_up_k"].reshape(w.rank, -1),
                            dd["w_up_v"].reshape(w.rank, -1), latent=lat)
                mla.attention(dd["q"], lat, dd["w_up_k"], dd["w_up_v"], w.scale, True, out=out)
            else:
                mla.attention(dd["q"], dd["kv_latent"], dd["w_up_k"], dd["w_up_v"], w.scale,
                              True, out=out)

        for _ in range(warmup):
            call(d)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call(d)
        e1.record(stream)
        torch.cuda.synchronize()
        device_us = e0.elapsed_time(e1) * 1e3 / n
        per = []
        for _ in range(n // 4):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(d)
            b.record(stream)
            b.synchronize()
            per.append(a.elapsed_time(b) * 1e3)
        host = {k: v.pin_memory() for k, v in x.items() if not (name == "proj_f32" and
                                                                  k == "kv_latent")}
        host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        e2e = []
        for it in range(n // 4 + warmup):
            t0 = time.perf_counter()
            for k, v in host.items():
                d[k].copy_(v, non_blocking=True)
            call(d)
            host_out.copy_(out, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
            if it >= warmup:
                e2e.append((time.perf_counter() - t0) * 1e6)
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        res[name] = {"device_us": round(device_us, 2), "call_us": round(statistics.median(per), 2),
                     "e2e_us": round(statistics.median(e2e), 2), "h2d_bytes": h2d,
                     "d2h_bytes": host_out.numel() * 4,
                     "flops": w.attention_flops() + w.projection_flops(with_kv=True)}
    return res


def run_attention_only(args, name: str):
    """Only one workload's attention (decode_bf16, mid_bf16 or prefill_bf16): warm-up, then
    timed calls with the L2 flushed between them; one JSON line.  A small
    driver for profiling that workload's kernels."""
    import torch

    from latent_causal_attention_gb300.build import build
    from latent_causal_attention_gb300.inputs import WORKLOADS

    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks(torch.cuda.get_device_name(dev))
    w = WORKLOADS[name]
    flush = torch.empty(256 * 1024 * 1024, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)
    ms, kernel_ms = time_attention_only(w, dev, flush, stream, args.steps, args.warmup)
    nbytes = w.attention_bytes(out_bytes=4)
    tflops = w.attention_flops() / (ms * 1e-3) / 1e12
    print(json.dumps({"mode": "attention-only", "workload": name, "ms": round(ms, 4),
                      "kernel_ms": round(kernel_ms, 4),
                      "GB_per_s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                      "frac_hbm": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                      "TFLOP_per_s": round(tflops, 2),
                      "frac_peak": round(tflops / peaks["bf16_tflops"], 4),
                      "steps": args.steps, "warmup": args.warmup}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-explicit", action="store_true")
    ap.add_argument("--no-mid", action="store_true")
    ap.add_argument("--no-small", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode attention (a driver for profiling its kernels)")
    ap.add_argument("--mid-only", action="store_true",
                    help="time only the mid-size attention (a driver for profiling its kernel)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prefill attention (a driver for profiling its kernel)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.decode_only or args.mid_only or args.prefill_only:
        run_attention_only(args, "decode_bf16" if args.decode_only else
                           "mid_bf16" if args.mid_only else "prefill_bf16")
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
