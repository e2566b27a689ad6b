"""Attention-forward benchmark: one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--pass fwd|bwd|linear] [--splits K]

A step is one exact attention forward over the workload's synthetic inputs,
already resident in HBM: the V pre-pass and the fused attention kernel (tile
loads, scores, masks, online softmax, correction, PV, epilogue), plus the
split-KV combine when the key range is split.  Between timed steps the L2 cache
is flushed by writing a 256 MiB buffer; each step's kernel is timed with CUDA
events on the stream it is launched on, and the steps' times are summed.
nvidia-smi samples the clocks from the start of the warm-up, which runs the
same (untimed) step until the GPU has been under this load for 0.5 s
("untimed_steps"), through the timed steps: the timed region alone is a few
milliseconds, far shorter than the sampling interval.

Default workload: B=2, H=16, N=4096, d=128, causal, bf16, seed 2.  Metric:
attention forward TFLOP/s with causal FLOPs counted at half (4*B*H*N^2*d/2).

Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of the
workload (independent heads/batches need no exchange; no collective touches
the data path), timed between barriers; `value` is the FLOPs of all ranks
divided by the slowest rank's time (weak scaling).

--impl reference times the fp64 CPU oracle (plain loops, the definition of the
result) on the host cores, on a bounded sample of query rows of the same
workload, in the same metric.

--pass bwd times the backward instead (fattn_bwd: dQ, dK, dV from dO and the
forward's O and LSE, which are computed once before the timed region), with
FLOPs counted as 2.5x the forward's (five GEMMs of the forward's size).

--pass linear times causal linear attention (fattn_linear_fwd: chunk state,
prefix scan, output kernels) on the linear workloads (--workload lin_...),
in TFLOP/s of the page's recurrence (4*E*M + 4*E per row), its roofline the
fp32 CUDA-core FMA peak.

roofline.achieved is the dominant kernel's rate on its own device time: the
library records two CUDA events around it on its stream
(fattn_set_kernel_events) -- the attention kernel of the forward, the dK/dV
kernel of the backward, the output kernel of linear attention -- while
`value` covers the whole step.  For the forward the kernel's events are taken
on a second set of as many steps after the timed ones, since an event
between the V pre-pass and the attention kernel would keep the kernel from
starting early (programmatic dependent launch on grids smaller than the GPU).  The forward's roofline has two legs, tensor
(algorithmic FLOPs at the measured bf16 burst peak) and HBM (algorithmic bytes
at the measured copy bandwidth); `bound` names the one whose time at peak is
longer, and roofline.frac / kernel_frac_of_peak / step_frac_of_peak are that
roof's fractions for the kernel alone and for the whole step.  The tensor rate
against the clock-derived peak (SMs x 8192 FLOP/clk x the sampled SM clock)
and the tensor-pipe activity of the committed ncu summary are reported beside
it.  roofline.traffic is that kernel's DRAM bytes
per launch from its committed ncu summary (profiles/), reported only while
the summary's kernel_source_hash matches the kernel's current code.

The forward splits each query block's key range (split-KV, with a combine
kernel) when the library's plan says so -- on shapes with fewer blocks of 256
query rows than SMs; --splits K forces K splits (1: none), and the split count
used is reported in config.kv_splits.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_softmax_attention_fattn_gb300.inputs import (  # noqa: E402
    HEADLINE, LINEAR_WORKLOADS, WORKLOADS, algorithmic_bytes, causal_flops, make_inputs)

KERNEL_NAME = "fattn_fwd_kernel"
METRIC = "attention fwd TFLOP/s (causal-adjusted) and % of GB300 bf16 dense peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
# Dense bf16 tensor-core rate of one SM per clock (a 128x128x16 MMA every 64
# cycles): the clock-derived peak is SMs x this x the sampled SM clock.
TENSOR_FLOP_PER_CLK_SM = 8192.0
CSRC = os.path.join(ROOT, "exact_softmax_attention_fattn_gb300", "csrc")


KERNEL_SOURCES = ("fattn_kernel.cuh", "ptx.cuh")
BWD_SOURCES = ("fattn_bwd.cuh", "ptx.cuh")
BWD256_SOURCES = ("fattn_bwd256.cuh", "fattn_bwd.cuh", "ptx.cuh")
D256_SOURCES = ("fattn_d256.cuh", "ptx.cuh")
LINEAR_SOURCES = ("linear_tc.cuh", "ptx.cuh")


def code_only(text: str) -> str:
    """C++ source without its comments, trailing blanks and empty lines: what
    decides the compiled kernel (string literals here hold no comment marks)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash(sources: tuple[str, ...] = KERNEL_SOURCES) -> str:
    """Hash of a kernel's own source code (not the host launcher), comments
    excluded, so that a capture stays valid across comment edits only."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(name.encode() + code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> tuple[float, str, float | None]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        hbm = float(pk["hbm_gbs"]) if pk.get("hbm_gbs") else FALLBACK_HBM_GBS
        return float(pk["bf16_tflops"]), "measured", hbm
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback", FALLBACK_HBM_GBS


def profile_field(profile: str, field: str, sources: tuple[str, ...] = KERNEL_SOURCES) -> str | None:
    """A field of a committed ncu summary (profiles/<profile>.txt), only while
    the summary's kernel_source_hash matches the current kernel source."""
    try:
        fields = {}
        with open(os.path.join(ROOT, "profiles", profile + ".txt")) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("kernel_source_hash", "").split()[:1] != [kernel_source_hash(sources)]:
            return None
        return fields.get(field)
    except OSError:
        return None


def forward_roofline(flops: float, nbytes: float, kernel_ms: float, step_ms: float, peak_tf: float,
                     peak_kind: str, hbm_gbs: float, sm_mhz: float | None, sms: int) -> dict:
    """Both roofs of one forward: tensor (algorithmic FLOPs at the measured
    bf16 peak) and HBM (algorithmic bytes at the measured copy bandwidth).
    `bound` is the roof with the longer time at peak; `achieved`, `peak` and
    `frac` are that roof's, on the dominant kernel's own CUDA-event time.
    The other roof, the whole step's fractions and the tensor fraction of the
    clock-derived peak (SMs x 8192 FLOP/clk x the sampled SM clock) follow."""
    t_tensor = flops / (peak_tf * 1e12)
    t_hbm = nbytes / (hbm_gbs * 1e9)
    tensor = {"achieved": flops / (kernel_ms * 1e-3) / 1e12, "peak": peak_tf, "unit": "TFLOP/s",
              "peak_kind": f"bf16 dense burst, {peak_kind}"}
    tensor["frac"] = tensor["achieved"] / peak_tf
    tensor["step_frac"] = flops / (step_ms * 1e-3) / 1e12 / peak_tf
    hbm = {"achieved": nbytes / (kernel_ms * 1e-3) / 1e9, "peak": hbm_gbs, "unit": "GB/s",
           "peak_kind": f"copy bandwidth, {peak_kind}", "algorithmic_bytes": nbytes}
    hbm["frac"] = hbm["achieved"] / hbm_gbs
    hbm["step_frac"] = nbytes / (step_ms * 1e-3) / 1e9 / hbm_gbs
    bound, other = ("tensor", "hbm") if t_tensor >= t_hbm else ("hbm", "tensor")
    legs = {"tensor": tensor, "hbm": hbm}
    out = {"bound": bound}
    out.update({k: legs[bound][k] for k in ("achieved", "peak", "unit", "frac", "peak_kind")})
    out["kernel_frac_of_peak"] = legs[bound]["frac"]
    out["step_frac_of_peak"] = legs[bound]["step_frac"]
    out[other] = legs[other]
    out["time_at_peak_us"] = {"tensor": t_tensor * 1e6, "hbm": t_hbm * 1e6}
    if sm_mhz:
        clock_peak = sms * TENSOR_FLOP_PER_CLK_SM * sm_mhz * 1e6 / 1e12
        out["tensor_frac_of_clock_peak"] = tensor["achieved"] / clock_peak
        out["clock_peak_tflops"] = clock_peak
    return out


def ncu_traffic(workload: str, profile: str | None = None, sources: tuple[str, ...] = KERNEL_SOURCES,
                field: str = "dram_bytes_per_launch") -> float | None:
    """DRAM bytes per launch of the dominant kernel from its committed ncu
    summary (profiles/<profile>.txt, default the attention kernel's for this
    workload), if the summary was taken on the current kernel source (its
    kernel_source_hash line matches); else None."""
    path = os.path.join(ROOT, "profiles", f"{profile or KERNEL_NAME + '_' + workload}.txt")
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("kernel_source_hash", "").split()[:1] != [kernel_source_hash(sources)]:
            return None
        return float(fields[field].split()[0])
    except (OSError, KeyError, ValueError, IndexError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": float(max(power)) if power else None}


def kernel_event_pairs(n: int, stream):
    """n (start, stop) CUDA event pairs for fattn_set_kernel_events, recorded
    once so that their CUDA events exist."""
    import torch

    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in pairs:
        a.record(stream)
        b.record(stream)
    return pairs


def warm_up(step, flush, warmup: int, sampler, dev, load_seconds: float = 0.5) -> int:
    """The untimed warm-up: `warmup` steps (each after an L2 flush), extended
    with more untimed steps of the same work until the clock sampler (started
    before it) has watched the GPU under this load for `load_seconds`, so the
    clock samples describe the clocks the timed steps run at.  Returns the
    number of untimed steps run."""
    import torch

    if sampler:
        sampler.start()
    t_end = time.perf_counter() + (load_seconds if sampler else 0.0)
    n = 0
    while n < warmup or time.perf_counter() < t_end:
        flush.fill_(1)
        step()
        n += 1
        if n % 16 == 0:
            torch.cuda.synchronize(dev)  # keep the queue short so the load tracks the wall clock
    torch.cuda.synchronize(dev)
    return n


# ---------------------------------------------------------------- oracle leg
def oracle_sample(workload: str, seconds: float, x=None):
    """Time the fp64 oracle on a bounded sample of query rows; returns
    (TFLOP/s, rows, seconds, threads, description)."""
    import oracle

    w = WORKLOADS[workload]
    if x is None:
        x = make_inputs(w)
    threads = oracle.default_threads()
    rng = np.random.default_rng(1234)
    total_rows = w.B * w.H * w.N

    def visible(rows):
        i = rows % w.N
        b = rows // (w.H * w.N)
        kl = np.full(rows.shape, w.N) if x.key_len is None else np.clip(x.key_len[b], 0, w.N)
        return np.minimum(kl, i + 1) if w.causal else kl

    def run(n):
        rows = np.sort(rng.choice(total_rows, size=min(n, total_rows), replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.forward(x.q, x.k, x.v, w.softmax_scale, w.causal, key_len=x.key_len, rows=rows, threads=threads)
        return rows, time.perf_counter() - t0

    rows, dt = run(threads * 2)
    n = int(max(threads, min(total_rows, len(rows) * seconds / max(dt, 1e-6))))
    rows, dt = run(n)
    flops = 4.0 * w.d * float(np.sum(visible(rows)))
    desc = (f"{len(rows)} random query rows of {total_rows} ({workload}), full fp64 score rows, "
            f"{threads} threads")
    return flops / dt / 1e12, len(rows), dt, threads, desc


def reference_arm(args, rank: int, world: int):
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    x = make_inputs(w)
    per_step = max(1.0, min(20.0, 100.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(args.workload, per_step / 4, x)
    vals, secs, rows_tot = [], 0.0, 0
    threads, desc = 1, ""
    for _ in range(args.steps):
        v, rows, dt, threads, desc = oracle_sample(args.workload, per_step, x)
        vals.append(v)
        secs += dt
        rows_tot += rows
    value = float(np.mean(vals))
    flops_step = causal_flops(w, x.key_len)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        # measured: the oracle's seconds per timed step (one bounded sample of rows)
        "ms_per_step": secs / max(1, args.steps) * 1e3,
        # not measured: the whole workload's time at the sampled rate
        "projected_ms_full_workload": flops_step / (value * 1e12) * 1e3 if value > 0 else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64/Box-Muller, bf16-rounded)",
        "config": {"workload": args.workload, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "sample": "bounded random query rows per step (oracle on host cores)",
                   "rows_per_step": rows_tot / max(1, args.steps)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ranks
def aggregate_ranks(ms_total: float, flops_per_step: float, steps: int, world: int, device=None):
    """Whole-job throughput over ranks: the slowest rank's time (MAX) and the
    FLOPs of all ranks (SUM).  Returns (ms_per_step, TFLOP/s)."""
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([ms_total], dtype=torch.float64, device=device)
        f = torch.tensor([flops_per_step], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(f, op=dist.ReduceOp.SUM)
        ms_total, flops_per_step = float(t.item()), float(f.item())
    ms_per_step = ms_total / steps
    return ms_per_step, flops_per_step / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------- CUDA leg
def our_arm(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    from exact_softmax_attention_fattn_gb300 import binding

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    binding.load_library()
    w = WORKLOADS[args.workload]
    x = make_inputs(w)

    def dev_bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = dev_bf16(x.q), dev_bf16(x.k), dev_bf16(x.v)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    kl = None if x.key_len is None else torch.from_numpy(x.key_len).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = causal_flops(w, x.key_len)

    def step():
        binding.forward_into(q, k, v, o, lse, causal=w.causal, scale=w.softmax_scale, key_len=kl, n_splits=args.splits)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n_splits = binding.splitkv_plan(w.B, w.H, w.N, w.causal, sms, args.splits or 0)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    untimed = warm_up(step, flush, args.warmup, sampler, dev)
    st, detail = binding.last_error(stream)
    if st != binding.FATTN_OK:
        raise RuntimeError(f"kernel reported {binding.status_string(st)} {detail}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kev = kernel_event_pairs(args.steps, stream)  # around the attention kernel, recorded by the library
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    # the attention kernel's own time, on as many further steps: the events
    # the library records around it sit between the V pre-pass and the
    # kernel, so they are kept out of the steps timed above (on small grids
    # the kernel is launched to overlap the pre-pass's end)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        binding.set_kernel_events(*kev[i])
        step()
    binding.set_kernel_events(None, None)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    st, detail = binding.last_error(stream)
    if st != binding.FATTN_OK:
        raise RuntimeError(f"kernel reported {binding.status_string(st)} {detail}")
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    attn_ms = [a.elapsed_time(b) for a, b in kev]
    ms_per_step, value = aggregate_ranks(float(sum(kernel_ms)), flops, args.steps, world, dev)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        klh = None if x.key_len is None else torch.from_numpy(x.key_len)
        # fattn_fwd_host through the public forward() (the library's own split-KV choice per chunk)
        # warm-up in the timed loop's own pattern: each call's pinned O and LSE
        # are allocated while the previous call's are still held, so two sets
        # of pinned blocks must be in the host allocator's cache before timing
        for _ in range(3):
            oh, lh = binding.forward(qh, kh, vh, causal=w.causal, scale=w.softmax_scale, key_len=klh)
        n_e2e = max(3, min(args.steps, 10))
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            oh, lh = binding.forward(qh, kh, vh, causal=w.causal, scale=w.softmax_scale, key_len=klh)
        torch.cuda.synchronize(dev)
        e2e_s = (time.perf_counter() - t0) / n_e2e
        h2d = 3 * q.numel() * 2 + (0 if klh is None else klh.numel() * 4)
        d2h = oh.numel() * 2 + lh.numel() * 4
        e2e = {"value": flops / e2e_s / 1e12 * world, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3}

    if rank != 0:
        return
    peak, peak_kind, hbm_gbs = measured_peaks()
    # the dominant kernel (the attention kernel) on its own CUDA-event time
    attn_mean_ms = float(np.mean(attn_ms))
    # head dims above 128 run the 256-column kernel, profiled under its own name
    prof_name, prof_src = ((f"fattn_fwd_d256_kernel_{args.workload}", D256_SOURCES) if w.d > 128 else
                           (KERNEL_NAME + "_" + args.workload, KERNEL_SOURCES))
    traffic = ncu_traffic(args.workload, prof_name, prof_src)
    roof = forward_roofline(flops, algorithmic_bytes(w, x.key_len), attn_mean_ms, ms_per_step, peak, peak_kind,
                            hbm_gbs, (clocks or {}).get("sm_mhz"), sms)
    roof.update({"traffic": traffic if n_splits == 1 else None,
                 "kernel": "attention kernel alone (V pre-pass and split-KV combine excluded)",
                 "kernel_ms_mean": attn_mean_ms})
    tpa = profile_field(prof_name, "tensor_pipe_active_pct_of_active", prof_src)
    if tpa:
        roof["ncu_tensor_pipe_active_pct"] = float(tpa.split()[0])
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v_cpu, rows, dt, threads, desc = oracle_sample(args.workload, args.cpu_seconds, x)
        cpu = {"value": v_cpu, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
               "seconds": round(dt, 2)}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "untimed_steps": untimed, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64/Box-Muller, bf16-rounded)",
        "config": {"workload": args.workload, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "key_padding": x.key_len is not None, "flops_per_step": flops,
                   "kv_splits": n_splits, "kv_split_choice": "library" if args.splits is None else "forced",
                   "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas x{world}"},
        "roofline": roof,
        # the whole call (every kernel of the step) against the same roof as roofline.frac
        "kernel_frac_of_peak": roof["kernel_frac_of_peak"],
        "step_frac_of_peak": roof["step_frac_of_peak"],
        "clocks": clocks,
        "e2e": e2e,
        # V pre-pass + attention kernel per step, + the split-KV combine when split
        "gpu_launches": (2 + (n_splits > 1)) * args.steps,
        "kernel": KERNEL_NAME + (" + fattn_splitkv_combine_kernel" if n_splits > 1 else ""),
        "kernel_ms": {"min": min(kernel_ms), "median": float(np.median(kernel_ms)), "max": max(kernel_ms)},
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def linear_parts(B: int, H: int, N: int, sms: int) -> int:
    """Parts per head of the tensor-core linear attention (feature sizes up
    to 64), as the library cuts them: about one CTA per SM over all heads."""
    n_tiles = -(-N // 128)
    n_parts = max(1, min(n_tiles, sms // max(1, B * H)))
    tpp = -(-n_tiles // n_parts)
    return -(-n_tiles // tpp)


def linear_arm(args, rank: int, world: int, local_rank: int):
    """--pass linear: causal linear attention (fattn_linear_fwd, fp32) on one
    of LINEAR_WORKLOADS, timed like the forward; FLOPs are the page's
    recurrence (linear_flops).  At feature sizes up to 64 it runs on the
    tensor cores (a part-totals launch when a head is cut into parts, then the
    output launch); the roofline is the output kernel's, with the HBM leg
    (Q, K, V read and the output written once, in fp32) and the tensor leg."""
    import torch
    import torch.distributed as dist

    import oracle
    from exact_softmax_attention_fattn_gb300 import binding
    from exact_softmax_attention_fattn_gb300.inputs import LINEAR_WORKLOADS, linear_flops, make_linear_inputs

    name = args.workload if args.workload in LINEAR_WORKLOADS else "lin_b2h16n4096e64"
    w = LINEAR_WORKLOADS[name]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    binding.load_library()
    x = make_linear_inputs(w)
    q, k, v = (torch.from_numpy(a).to(dev) for a in (x.q, x.k, x.v))
    kl = None if x.key_len is None else torch.from_numpy(x.key_len).to(dev)
    out = torch.empty((w.B, w.H, w.N, w.M), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = linear_flops(w)

    def step():
        binding.linear_forward(q, k, v, key_len=kl, out=out)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    untimed = warm_up(step, flush, args.warmup, sampler, dev)
    st, detail = binding.last_error(stream)
    if st != binding.FATTN_OK:
        raise RuntimeError(f"kernel reported {binding.status_string(st)} {detail}")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kev = kernel_event_pairs(args.steps, stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        binding.set_kernel_events(*kev[i])
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    binding.set_kernel_events(None, None)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    st, detail = binding.last_error(stream)
    if st != binding.FATTN_OK:
        raise RuntimeError(f"kernel reported {binding.status_string(st)} {detail}")
    step_ms = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    out_ms = [a.elapsed_time(b) for a, b in kev]
    ms_per_step, value = aggregate_ranks(float(sum(step_ms)), flops, args.steps, world, dev)

    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        qd, kd, vd = (torch.empty_like(t) for t in (q, k, v))

        def e2e_step():
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            binding.linear_forward(qd, kd, vd, key_len=kl, out=out)
            oh.copy_(out, non_blocking=True)
            torch.cuda.synchronize(dev)

        for _ in range(2):
            e2e_step()
        n_e2e = max(3, min(args.steps, 10))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        e2e_s = (time.perf_counter() - t0) / n_e2e
        e2e = {"value": flops / e2e_s / 1e12 * world, "unit": UNIT,
               "h2d_bytes_per_step": sum(t.numel() * 4 for t in (q, k, v)), "d2h_bytes_per_step": out.numel() * 4,
               "ms_per_step": e2e_s * 1e3}
    if rank != 0:
        return
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out_mean = float(np.mean(out_ms))
    n_parts = linear_parts(w.B, w.H, w.N, sms)
    nbytes = float(w.B * w.H * w.N) * (2 * w.E + 2 * w.M) * 4
    peak_tf, peak_kind, hbm_gbs = measured_peaks()
    roof = forward_roofline(flops, nbytes, out_mean, ms_per_step, peak_tf, peak_kind, hbm_gbs,
                            (clocks or {}).get("sm_mhz"), sms)
    roof.update({"traffic": ncu_traffic(name, f"fattn_linear_kernels_{name}", LINEAR_SOURCES,
                                        "output_dram_bytes_per_launch"),
                 "kernel": "fattn_linear_tc_kernel (output launch) alone", "kernel_ms_mean": out_mean,
                 "flops_counted": "the recurrence's 4*E*M + 4*E per row (the tensor cores run three bf16 "
                                  "terms of each chunked product)"})
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        t0 = time.perf_counter()
        oracle.linear(x.q[:1, :1], x.k[:1, :1], x.v[:1, :1], key_len=None if x.key_len is None else x.key_len[:1])
        dt = time.perf_counter() - t0
        cpu = {"value": flops / (w.B * w.H) / dt / 1e12, "unit": UNIT, "cores": oracle.default_threads(),
               "kind": "oracle", "sample": f"head 0 of {w.B * w.H} ({name}), full fp64 recurrence",
               "seconds": round(dt, 3)}
    line = {
        "metric": "causal linear attention TFLOP/s (the recurrence's 4*E*M + 4*E FLOPs per row)",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "untimed_steps": untimed, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded SplitMix64/Box-Muller, float32)",
        "config": {"workload": name, "pass": "linear", "B": w.B, "H": w.H, "N": w.N, "E": w.E, "M": w.M,
                   "key_padding": x.key_len is not None, "flops_per_step": flops,
                   "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "kernel_frac_of_peak": roof["kernel_frac_of_peak"],
        "step_frac_of_peak": roof["step_frac_of_peak"],
        "clocks": clocks,
        "e2e": e2e,
        # part totals (when a head is cut into parts) + output
        "gpu_launches": (1 + (n_parts > 1)) * args.steps,
        "kernel": "fattn_linear_tc_kernel<STATE> + fattn_linear_tc_kernel<OUTPUT>",
        "config_parts_per_head": n_parts,
        "kernel_ms": {"min": min(step_ms), "median": float(np.median(step_ms)), "max": max(step_ms)},
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def bwd_arm(args, rank: int, world: int, local_rank: int):
    """The backward pass, timed like the forward (one JSON line on rank 0)."""
    import torch

    import oracle
    from exact_softmax_attention_fattn_gb300 import binding

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    binding.load_library()
    w = WORKLOADS[args.workload]
    x = make_inputs(w)
    g_bits = make_inputs(w.replace(seed=w.seed + 1000)).v  # dL/dO ~ N(0, 1)

    def dev_bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v, go = dev_bf16(x.q), dev_bf16(x.k), dev_bf16(x.v), dev_bf16(g_bits)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    kl = None if x.key_len is None else torch.from_numpy(x.key_len).to(dev)
    binding.forward_into(q, k, v, o, lse, causal=w.causal, scale=w.softmax_scale, key_len=kl)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = 2.5 * causal_flops(w, x.key_len)

    def step():
        binding.backward_into(q, k, v, o, lse, go, dq, dk, dv, causal=w.causal, scale=w.softmax_scale, key_len=kl)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    untimed = warm_up(step, flush, args.warmup, sampler, dev)
    st, detail = binding.last_error(stream)
    if st != binding.FATTN_OK:
        raise RuntimeError(f"kernel reported {binding.status_string(st)} {detail}")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kev = kernel_event_pairs(args.steps, stream)  # around the dK/dV kernel, recorded by the library
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        binding.set_kernel_events(*kev[i])
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    binding.set_kernel_events(None, None)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    st, detail = binding.last_error(stream)
    if st != binding.FATTN_OK:
        raise RuntimeError(f"kernel reported {binding.status_string(st)} {detail}")
    kernel_ms = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    dkdv_ms = [a.elapsed_time(b) for a, b in kev]
    ms_per_step, value = aggregate_ranks(float(sum(kernel_ms)), flops, args.steps, world, dev)

    # end to end: the six inputs copied in from pinned host buffers, three gradients copied out
    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in (q, k, v, o, go)] + [lse.cpu().pin_memory()]
        host_out = [torch.empty(q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
        dev_in = [torch.empty_like(t, device=dev) for t in host_in]

        def e2e_step():
            for hd, dd in zip(host_in, dev_in):
                dd.copy_(hd, non_blocking=True)
            binding.backward_into(dev_in[0], dev_in[1], dev_in[2], dev_in[3], dev_in[5], dev_in[4], dq, dk, dv,
                                  causal=w.causal, scale=w.softmax_scale, key_len=kl)
            for hd, dd in zip(host_out, (dq, dk, dv)):
                hd.copy_(dd, non_blocking=True)

        for _ in range(2):  # untimed: first copies into these buffers, scratch pool growth
            e2e_step()
        n_e2e = max(3, min(args.steps, 10))
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize(dev)
        e2e_s = (time.perf_counter() - t0) / n_e2e
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        e2e = {"value": flops / e2e_s / 1e12 * world, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3}
    if rank != 0:
        return
    peak, peak_kind, _ = measured_peaks()
    # the dominant kernel on its own CUDA-event time: up to head dim 128 the
    # dK/dV kernel (S, dP, dV, dK = 4 of the forward's 2 GEMMs), above it the
    # dK pass of the three-pass backward (S, dP, dK = 3)
    big = w.d > 128
    # the single-kernel backward (FATTN_BWD_FUSED=1, head dims 72..128): all 5 GEMMs
    fused = os.environ.get("FATTN_BWD_FUSED", "").startswith("1") and 64 < w.d <= 128
    dkdv_mean_ms = float(np.mean(dkdv_ms))
    achieved = (flops / 2.5 * (1.5 if big else 2.5 if fused else 2.0)) / (dkdv_mean_ms * 1e-3) / 1e12
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        # the fp64 oracle backward on one head (about 2.5x the head's forward FLOPs)
        t0 = time.perf_counter()
        oracle.backward(x.q, x.k, x.v, g_bits, w.softmax_scale, w.causal, key_len=x.key_len, heads=[0])
        dt = time.perf_counter() - t0
        head_flops = flops / (w.B * w.H)
        cpu = {"value": head_flops / dt / 1e12, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
               "sample": f"head 0 of {w.B * w.H} ({args.workload}), full fp64 backward", "seconds": round(dt, 2)}
    line = {
        "metric": "attention bwd TFLOP/s (causal-adjusted, 2.5x forward FLOPs) and % of GB300 bf16 dense peak",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "untimed_steps": untimed,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded SplitMix64/Box-Muller, bf16-rounded)",
        "config": {"workload": args.workload, "pass": "bwd", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "key_padding": x.key_len is not None, "flops_per_step": flops,
                   "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "peak_kind": f"bf16 dense burst, {peak_kind}",
                     "traffic": None if fused else ncu_traffic(args.workload, f"fattn_bwd_kernels_{args.workload}",
                                                               BWD256_SOURCES if big else BWD_SOURCES,
                                                               "dkdv_dram_bytes_per_launch"),
                     "kernel": ("dK pass alone (its 3 GEMMs: 1.5x the forward's FLOPs)" if big else
                                "fused backward kernel alone (its 5 GEMMs: 2.5x the forward's FLOPs)" if fused else
                                "dK/dV kernel alone (its 4 GEMMs: 2x the forward's FLOPs)"),
                     "kernel_ms_mean": dkdv_mean_ms},
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "clocks": clocks,
        "e2e": e2e,
        # prep + dK/dV + dQ kernels (prep + three passes; prep + fused + dQ conversion, and a memset) per step
        "gpu_launches": (4 if big else 3) * args.steps,
        "kernel": ("fattn_bwd_prep_kernel + fattn_bwd256_kernel (dV, dK, dQ passes)" if big else
                   "fattn_bwd_prep_kernel + fattn_bwd_fused_kernel + fattn_bwd_dq_finalize_kernel" if fused else
                   "fattn_bwd_prep_kernel + fattn_bwd_dkdv_kernel + fattn_bwd_dq_kernel"),
        "kernel_ms": {"min": min(kernel_ms), "median": float(np.median(kernel_ms)), "max": max(kernel_ms)},
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS) + sorted(LINEAR_WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "linear"], default="fwd",
                    help="time the forward (default), the backward, or causal linear attention")
    ap.add_argument("--splits", type=int, default=None,
                    help="forward: force this many key splits per query block (split-KV; 1 = none); "
                         "default: the library's choice")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        {"bwd": bwd_arm, "linear": linear_arm}.get(args.pass_, our_arm)(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
