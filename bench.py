#!/usr/bin/env python
"""Benchmark of the hot path on the long-context workload.

One step = attnq_prepare (mean-key centring, random-sign Hadamard, per-head
scales, E4M3 cast) + attnq_fwd (causal FP8 attention, reverse KV order,
S = 256) over one batch: B=2, Hq=32, Hkv=8, N=32768, d=128, bf16 inputs,
bf16 output.  The inputs (805 MB per step) exceed the 129 MB L2, so no flush
is needed between steps.

Prints one JSON line (rank 0).  `value` is algorithmic attention TFLOP/s
(4*d per unmasked (i, j) pair, summed over all ranks) over the device-timed
step; `e2e` repeats the measurement through the C ABI's host-buffer pipeline
(attnq_attention_host): every step copies its bf16 inputs in from pinned host
memory and its output back inside the timed region, the copies of
neighbouring steps overlapping each step's kernels (its own SM-clock sample
in `e2e.clocks`).  Under torchrun every rank runs its own independent replica
(weak scaling, no collective on the data path).

Each kernel's roofline object gives its mean per-launch time over the timed
steps (CUDA events on its stream) with the median and the best beside it;
`device` names the GPU (CUDA device properties).

The attention roofline divides by this GPU's dense FP8 GEMM rate, measured
in the same run after the timed region (cuBLASLt E4M3 GEMM at 8192^3 through
torch._scaled_mm, best of 10: the burst figure, as the timed region is well
under a second); the datasheet fraction is reported beside it.

Variants of the same workload (not the default line): --qk int8 (INT8 Q/K
codes, Q.K^T on the bf16 tensor path; the roofline peak then combines the
bf16 and FP8 rates), --stat-len P (mean key and slice scales from the first
P tokens), --scales tile (per-128-token Q/K scales); --report harm times the
four-condition harm report on one Qwen-0.5B-shaped layer instead.

The other workloads, one JSON line each: --config 1 (sink probe), 2 (P-cast
isolation sweep: MSE and underflow fraction of all 78 runs, --report-md
writes the table), 3 and 4 (every layer of the Qwen-0.5B- and 1.5B-shaped
workloads in all four conditions); each times the GPU (configs 1, 3 and 4,
whose kernels last microseconds, as one CUDA graph replay per step, with the
direct-call time beside it) and, in its cpu_baseline leg, the oracle on the
whole workload, with parity figures.

--impl reference times the CPU oracle (the plain C++ implementation used by
the tests) on a bounded sample of the same workload.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal FP8 attention fwd TFLOP/s, % of GB300 FP8 peak; rel-Frobenius err vs FP64"
WL = dict(B=2, Hq=32, Hkv=8, N=32768, d=128, kv_tile=128, S=256.0, kv_order="reverse")
L2_BYTES = 129 * 1024 * 1024


def attn_flops(B, Hq, N, d, rows=None):
    """Algorithmic flops: 4*d per unmasked causal (i, j) pair."""
    if rows is None:
        pairs = N * (N + 1) // 2
    else:
        pairs = int(np.sum(np.asarray(rows, dtype=np.int64) + 1))
    return 4.0 * d * pairs * B * Hq


def prepare_bytes(B, Hq, Hkv, N, d, in_bytes=2, qk_code_bytes=1):
    """Algorithmic bytes of one prepare: read Q, K, V once, write their codes once
    (E4M3: 1 byte; INT8 Q/K codes held in bf16: 2 bytes)."""
    elems = (B * Hq + 2 * B * Hkv) * N * d
    qk = (B * Hq + B * Hkv) * N * d
    return elems * in_bytes + (elems - qk) + qk * qk_code_bytes


# Dense tensor peaks from the datasheet, TFLOP/s: FP8 for the E4M3 step; for
# INT8-QK half the flops run on the bf16 path, so 1 / (0.5 / 2250 + 0.5 / 4500).
DATASHEET_MMA_TFLOPS = {"e4m3": 4500.0, "int8": 3000.0}


def device_info(dev) -> dict:
    """The GPU the line was measured on, from the CUDA device properties."""
    import torch
    pr = torch.cuda.get_device_properties(dev)
    l2 = getattr(pr, "L2_cache_size", None)
    return {"name": pr.name, "sm_count": pr.multi_processor_count, "cc": f"{pr.major}.{pr.minor}",
            "l2_mb": None if l2 is None else round(l2 / 2**20, 1), "hbm_gib": round(pr.total_memory / 2**30, 1)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


def measure_fp8_peak(device, n: int = 8192, reps: int = 10):
    """Dense FP8 (E4M3 x E4M3, fp32 accumulate) GEMM rate of this GPU, measured
    the way the bf16 peaks are: a library GEMM (cuBLASLt through
    torch._scaled_mm) at n^3, 2 n^3 flops a call, best of `reps` timed calls
    (the burst figure), CUDA events on the current stream.  Both accumulation
    modes are tried and the faster one kept.  Returns None where the call is
    not available (the roofline then falls back to twice the bf16 burst peak
    and says so)."""
    import torch
    try:
        g = torch.Generator(device=device)
        g.manual_seed(11)
        a = torch.randn((n, n), device=device, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=device, generator=g).to(torch.float8_e4m3fn)
        one = torch.ones((), device=device, dtype=torch.float32)
        best, best_mode = float("inf"), None
        for fast in (False, True):
            def mm():
                return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16,
                                        use_fast_accum=fast)
            for _ in range(3):
                mm()
            torch.cuda.synchronize()
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                mm()
                e1.record()
                e1.synchronize()
                ms = e0.elapsed_time(e1)
                if ms < best:
                    best, best_mode = ms, fast
        del a, b
        torch.cuda.synchronize()
        return {"tflops": 2.0 * n ** 3 / (best * 1e-3) / 1e12, "n": n, "reps": reps,
                "use_fast_accum": best_mode,
                "method": f"torch._scaled_mm e4m3 x e4m3 -> bf16 (cuBLASLt), {n}^3, best of {reps}"}
    except Exception as exc:  # noqa: BLE001 - any failure means "not measured"
        return {"tflops": None, "error": f"{type(exc).__name__}: {exc}"[:200]}


def code_lines(text: str) -> str:
    """Source without // comments and blank lines (what the compiler sees of it)."""
    out = []
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            out.append(code)
    return "\n".join(out)


def kernel_source_hash(files):
    """Hash of the kernels' code, blind to comments, so a counter capture stays
    valid across comment edits and is dropped when the code changes."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "precision_attention_numerics_gb300", "csrc", f)) as fh:
            h.update(code_lines(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel and parts[2] == src_hash:
                return float(parts[1])
    return None


def launches_per_step(flags: int) -> int:
    """Kernels one prepare + forward step launches: the prepare's
    initialisation (counters and work list) and its persistent kernel, then
    the attention kernel."""
    return 3


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"attnq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(x: float, dist, device) -> float:
    """Largest x over all ranks (the slowest replica sets the job's time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(flops_per_step: float, steps: int, world: int, elapsed_max: float) -> float:
    """Whole-job TFLOP/s: every replica does the same work; the job ends with the slowest."""
    return flops_per_step * steps * world / elapsed_max / 1e12


def replica_seed(rank: int) -> int:
    """Each replica draws its own batch (weak scaling: independent problems)."""
    return 5000 + rank


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# oracle (CPU) sample: the CPU baseline and the reference arm
# ---------------------------------------------------------------------------

def oracle_sample(q, k, v, signs, rows, heads_group=0, b=0, stat_len=0, extra_flags=0):
    """Oracle prepare of one (batch, KV group) and quantised emulation of the
    given query rows of its query heads.  Returns (seconds, flops, threads)."""
    import oracle
    G = WL["Hq"] // WL["Hkv"]
    qs = q[b:b + 1, heads_group * G:(heads_group + 1) * G]
    ks = k[b:b + 1, heads_group:heads_group + 1]
    vs = v[b:b + 1, heads_group:heads_group + 1]
    N, d = WL["N"], WL["d"]
    t0 = time.perf_counter()
    fl = oracle.ROTATE | oracle.CENTER_K | extra_flags
    prep = oracle.prepare(qs, ks, vs, flags=fl, signs=signs, stat_len=stat_len)
    t1 = time.perf_counter()
    oracle.attn_quant(prep, (1, G, 1, N, d), fl, WL["S"], 1, True, WL["kv_tile"],
                      rows=rows)
    t2 = time.perf_counter()
    oracle_sample.split = (t1 - t0, t2 - t1)
    return t2 - t0, attn_flops(1, G, N, d, rows=rows), oracle.threads()


def extrapolated_oracle_step(t_prep_group: float, t_emu: float, flops_sample: float) -> float:
    """Oracle time for a whole step, extrapolated from the sample: the prepare
    of one (batch, KV group) times the number of groups, plus the emulation
    time scaled by causal pair count (whole step's flops over the sample's)."""
    groups = WL["B"] * WL["Hkv"]
    full = attn_flops(WL["B"], WL["Hq"], WL["N"], WL["d"])
    return t_prep_group * groups + t_emu * full / flops_sample


def sample_rows(n_rows):
    N = WL["N"]
    return np.unique(np.linspace(N // 2, N - 1, n_rows).astype(np.int64))


def make_inputs(seed):
    import synth
    return synth.long_context_inputs(seed, WL["B"], WL["Hq"], WL["Hkv"], WL["N"], WL["d"])


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import synth
    q, k, v = make_inputs(5000)
    signs = synth.hadamard_signs(17, WL["d"])
    rows = sample_rows(args.ref_rows)
    times, flops, thr = [], 0.0, 1
    for s in range(args.warmup + args.steps):
        dt, fl, thr = oracle_sample(q, k, v, signs, rows)
        if s >= args.warmup:
            times.append(dt)
            flops = fl
    mean = sum(times) / len(times)
    value = flops / mean / 1e12
    sample = (f"oracle prepare of one (batch, KV group) slice set (4 query heads, 1 KV head) + quantised "
              f"emulation of {len(rows)} query rows in [N/2, N) of those 4 heads per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 emulation of e4m3", "data": "synthetic",
            "config": {"workload": "long_context", **WL, "step": "oracle sample (see cpu_baseline.sample)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the four-condition harm report (a widening row, not the timed hot path)
# ---------------------------------------------------------------------------

FP64_PEAK_TFLOPS = 1.25  # nominal dense FP64 of a GB300 (no measured figure exists)


def run_harm(args):
    """One Qwen-0.5B-shaped layer through attnq_harm_report: the FP64 reference
    attention, then prepare + forward + per-head error for the four
    conditions.  Reports the time per layer, the reference kernel's FP64 rate
    against the nominal FP64 peak, and the oracle doing the same on one
    (batch, KV group)."""
    import torch

    import oracle
    import precision_attention_numerics_gb300 as aq
    import synth
    wl = synth.WORKLOADS["qwen05b"]
    B, Hq, Hkv, N, d, T = wl["B"], wl["Hq"], wl["Hkv"], wl["N"], wl["d"], wl["kv_tile"]
    q, k, v = synth.qwen_like_inputs(3000, B, Hq, Hkv, N, d, key_norm=wl["key_norm"],
                                     key_channels=wl["key_channels"])
    signs = synth.hadamard_signs(3001, d)
    dev = torch.device("cuda")
    Q, K, V = (torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(dev) for a in (q, k, v))
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16, 0, torch.from_numpy(signs).to(dev))
    ws = torch.empty(aq.attnq_harm_workspace(desc), dtype=torch.uint8, device=dev)
    err = torch.empty((4, B * Hq), dtype=torch.float64, device=dev)
    O_ref = torch.empty((B, Hq, N, d), dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    ms_ref = timed(lambda: aq.attnq_ref_attention(desc, Q, K, V, True, O_ref))
    ms_rep = timed(lambda: aq.attnq_harm_report(desc, Q, K, V, 256.0, aq.ATTNQ_KV_REVERSE, T, ws, err))
    assert aq.attnq_device_status() == 0
    e = err.cpu().numpy()
    harm = (e[1] - e[0]).reshape(B, Hq).mean(axis=0)
    ref_tflops = attn_flops(B, Hq, N, d) / (ms_ref * 1e-3) / 1e12
    # oracle: the same four conditions on batch 0, KV group 0 (its G query heads)
    G = Hq // Hkv
    qs, ks, vs = q[:1, :G], k[:1, :1], v[:1, :1]
    t0 = time.perf_counter()
    exact = oracle.attn_exact(qs, ks, vs)
    for flags in (0, 1, 2, 3):
        prep = oracle.prepare(qs, ks, vs, flags=flags, signs=signs)
        emu, _ = oracle.attn_quant(prep, (1, G, 1, N, d), flags, 256.0, 1, True, T)
        oracle.err(emu, exact)
    dt = time.perf_counter() - t0
    line = {"metric": "four-condition harm report, ms per Qwen-0.5B-shaped layer", "value": ms_rep, "unit": "ms",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
            "vs_baseline": None, "dtype": "f64 reference + e4m3 forward", "data": "synthetic",
            "config": {"workload": "qwen05b_layer", "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "kv_tile": T,
                       "S": 256.0, "kv_order": "reverse", "conditions": ["unrotated", "rotated", "centred",
                                                                         "centred_rotated"]},
            "roofline": {"kernel": "attnq_ref_attention (k_ref_attn)", "bound": "alu", "achieved": ref_tflops,
                         "peak": FP64_PEAK_TFLOPS, "unit": "TFLOP/s fp64", "frac": ref_tflops / FP64_PEAK_TFLOPS,
                         "traffic": None, "peak_note": "nominal dense FP64 (no measured FP64 peak)",
                         "ms_per_launch": ms_ref},
            "harm_mean_abs": float(np.mean(np.abs(harm))),
            "cpu_baseline": {"value": dt * 1e3 * (B * Hkv), "unit": "ms per layer (extrapolated from one KV group)",
                             "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"oracle exact attention + four conditions on 1 of {B * Hkv} (batch, KV group)"}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the other four workloads (--config 1..4): parity-test shapes, timed here
# end to end on the GPU and, in the cpu_baseline leg, on the oracle
# ---------------------------------------------------------------------------

def _event_ms(fn, warmup, steps, stream):
    """Mean device time of fn() over `steps` calls after `warmup` calls (CUDA events)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def _graph_ms(fn, warmup, steps, stream):
    """Mean device time of one replay of a CUDA graph holding fn()'s launches
    (captured once after `warmup` direct calls): the same kernels without the
    per-call host work, for workloads whose kernels last a few microseconds."""
    import torch
    for _ in range(max(1, warmup)):
        fn()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    return _event_ms(g.replay, 2, steps, stream)


def nonsink_in_mask(N: int, k_sink: int) -> int:
    """In-mask keys j >= k_sink summed over the N query rows of one causal head."""
    r = np.arange(N, dtype=np.int64)
    return int(np.maximum(r + 1 - k_sink, 0).sum())


def _dev_tensor(a, dev):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(dev)


def _common_line(metric, value, unit, args, hib, dtype, config, **extra):
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": hib, "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": config}
    line.update(extra)
    return line


def run_config1(args):
    """Sink probe: B=1, H=1, N=256, d=64, KV tile 64, fp32 inputs with 4 sink
    keys at delta = 7, no rotation; one step = prepare + forward at S = 1 +
    forward at S = 256 (forward KV order).  Launch-bound at this size."""
    import torch

    import precision_attention_numerics_gb300 as aq
    import synth
    wl = synth.WORKLOADS["sink_probe"]
    B, H, N, d, T = wl["B"], wl["Hq"], wl["N"], wl["d"], wl["kv_tile"]
    dev = torch.device("cuda")
    aq.load_library()
    q, k, v = synth.sink_probe_inputs()
    Q, K, V = (_dev_tensor(a, dev) for a in (q, k, v))
    desc = aq.AttnqDesc(B, H, H, N, d, aq.ATTNQ_F32, aq.ATTNQ_VT_LAYOUT)
    bufs = aq.alloc_prepared(desc, device=dev)
    Os = {S: torch.empty((B, H, N, d), dtype=torch.float32, device=dev) for S in wl["S"]}
    stream = torch.cuda.current_stream()

    def step():
        aq.attnq_prepare(desc, Q, K, V, bufs.q8, bufs.k8, bufs.v8, bufs.scales, bufs.workspace)
        for S in wl["S"]:
            aq.attnq_fwd(desc, bufs.q8, bufs.k8, bufs.v8, bufs.scales, S, aq.ATTNQ_KV_FORWARD, True, T, Os[S])

    ms_direct = _event_ms(step, args.warmup, args.steps, stream)
    ms = _graph_ms(step, args.warmup, args.steps, stream)
    flops = attn_flops(B, H, N, d) * len(wl["S"])
    # one untimed pass with the underflow counters, and the per-head error
    # against the GPU's FP64 reference
    O_ref = torch.empty((B, H, N, d), dtype=torch.float64, device=dev)
    aq.attnq_ref_attention(desc, Q, K, V, True, O_ref)
    per_s = {}
    outs = {}
    for S in wl["S"]:
        uf = torch.zeros(2 * B * H, dtype=torch.int64, device=dev)
        aq.attnq_fwd(desc, bufs.q8, bufs.k8, bufs.v8, bufs.scales, S, aq.ATTNQ_KV_FORWARD, True, T, Os[S], uf)
        err = torch.empty(B * H, dtype=torch.float64, device=dev)
        aq.attnq_err(desc, Os[S], O_ref, err)
        u = uf.cpu().numpy().astype(np.int64)
        per_s[str(int(S))] = {"log1p_relF_vs_fp64": float(err.cpu().numpy().mean()),
                              "nonsink_underflow_fraction": float(u.sum() / nonsink_in_mask(N, 4) / (B * H)),
                              "underflow_tile0": int(u[0::2].sum()), "underflow_later_tiles": int(u[1::2].sum())}
        outs[S] = (Os[S].cpu().numpy().astype(np.float64).reshape(B * H, N, d), u.reshape(-1, 2))
    st = aq.attnq_device_status()
    if st != 0:
        raise RuntimeError(f"device status {aq.STATUS.get(st, st)}")
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        prep = oracle.prepare(q, k, v, flags=0)
        emus = {S: oracle.attn_quant(prep, (B, H, H, N, d), 0, S, 0, True, T) for S in wl["S"]}
        exact = oracle.attn_exact(q, k, v)
        dt = time.perf_counter() - t0
        parity = {}
        for S in wl["S"]:
            emu, uref = emus[S]
            got, u = outs[S]
            rel = float(np.linalg.norm(got - emu) / np.linalg.norm(emu))
            e_orc = float(oracle.err(emu, exact).mean())
            parity[str(int(S))] = {"relF_vs_emulation": rel, "log1p_relF_oracle": e_orc,
                                   "underflow_oracle": uref.astype(np.int64).sum(axis=0).tolist(),
                                   "underflow_gpu": u.sum(axis=0).tolist()}
        cpu = {"value": dt * 1e3, "unit": "ms per step (prepare + both forwards + exact FP64 attention)",
               "cores": oracle.threads(), "kind": "oracle", "sample": "the whole workload", "parity": parity}
    cfg = {"workload": "sink_probe", "B": B, "H": H, "N": N, "d": d, "kv_tile": T, "in_dtype": "f32",
           "delta": wl["deltas"][0], "S": list(wl["S"]), "kv_order": "forward", "rotate": False, "center_k": False,
           "step": "attnq_prepare + attnq_fwd (S=1) + attnq_fwd (S=256)", "l2": "inputs fit in L2 (launch-bound size)",
           "launch": "one CUDA graph replay per step (ms_per_step_direct: the same calls made directly)"}
    line = _common_line("sink probe step time (launch-bound)", ms * 1e3, "us per step", args, False, "e4m3", cfg,
                        ms_per_step=ms, ms_per_step_direct=ms_direct, tflops=flops / (ms * 1e-3) / 1e12,
                        per_S=per_s, cpu_baseline=cpu,
                        gpu_launches=args.steps * (2 + len(wl["S"])))
    print(json.dumps(line), flush=True)
    return 0


def run_config2(args):
    """P-cast isolation sweep: B=1, H=8, N=4096, d=128, KV tile 128, fp32 Q/K/V
    with 4 sink keys at delta = 0..12, only P cast (attnq_fwd_ponly), forward
    and reverse x S in {1, 256, 448}: 78 runs and 13 FP64 references (GPU).
    Reports the output MSE against FP64 and the non-sink underflow fraction of
    every run, the P-cast page's four qualitative results (section 4) as
    measured values, and in the cpu_baseline leg the oracle's emulation of the
    whole sweep (its time, its MSE and counts, and the closed form F(delta, S))."""
    import torch

    import precision_attention_numerics_gb300 as aq
    import synth
    wl = synth.WORKLOADS["pcast_sweep"]
    B, H, N, d, T = wl["B"], wl["Hq"], wl["N"], wl["d"], wl["kv_tile"]
    deltas, Ss, orders = wl["deltas"], wl["S"], (aq.ATTNQ_KV_FORWARD, aq.ATTNQ_KV_REVERSE)
    oname = {aq.ATTNQ_KV_FORWARD: "fwd", aq.ATTNQ_KV_REVERSE: "rev"}
    dev = torch.device("cuda")
    aq.load_library()
    stream = torch.cuda.current_stream()
    nonsink = nonsink_in_mask(N, 4) * B * H

    def sweep_at(n_tokens, delta_list, runs):
        """GPU P-only runs; returns {(delta, order, S): (mse, uf0, uf1, O)}."""
        desc = aq.AttnqDesc(B, H, H, n_tokens, d, aq.ATTNQ_F32, 0, None)
        res = {}
        for delta in delta_list:
            q, k, v = synth.pcast_sweep_inputs(delta, n_tokens)
            Q, K, V = (_dev_tensor(a, dev) for a in (q, k, v))
            O_ref = torch.empty((B, H, n_tokens, d), dtype=torch.float64, device=dev)
            aq.attnq_ref_attention(desc, Q, K, V, True, O_ref)
            ref = O_ref.cpu().numpy()
            for order, S in runs:
                O = torch.empty((B, H, n_tokens, d), dtype=torch.float32, device=dev)
                uf = torch.zeros(2 * B * H, dtype=torch.int64, device=dev)
                aq.attnq_fwd_ponly(desc, Q, K, V, S, order, True, T, O, uf)
                o = O.cpu().numpy().astype(np.float64)
                u = uf.cpu().numpy().astype(np.int64).reshape(-1, 2)
                res[(delta, order, S)] = (float(np.mean((o - ref) ** 2)), int(u[:, 0].sum()), int(u[:, 1].sum()), o)
        return res

    runs = [(o, S) for o in orders for S in Ss]
    t0 = time.perf_counter()
    res = sweep_at(N, deltas, runs)
    sweep_s = time.perf_counter() - t0
    # the kernel's own time for one run (delta = 7, reverse, S = 256)
    desc = aq.AttnqDesc(B, H, H, N, d, aq.ATTNQ_F32, 0, None)
    q, k, v = synth.pcast_sweep_inputs(7.0)
    Q, K, V = (_dev_tensor(a, dev) for a in (q, k, v))
    O = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    ms_run = _event_ms(lambda: aq.attnq_fwd_ponly(desc, Q, K, V, 256.0, aq.ATTNQ_KV_REVERSE, True, T, O),
                       args.warmup, args.steps, stream)
    st = aq.attnq_device_status()
    if st != 0:
        raise RuntimeError(f"device status {aq.STATUS.get(st, st)}")
    table = []
    for delta in deltas:
        for order, S in runs:
            mse, u0, u1, _ = res[(delta, order, S)]
            table.append({"delta": delta, "order": oname[order], "S": S, "mse": mse,
                          "underflow_fraction": (u0 + u1) / nonsink, "underflow_tile0": u0, "underflow_later": u1})

    def mse(delta, order, S):
        return res[(delta, order, S)][0]

    F, R = aq.ATTNQ_KV_FORWARD, aq.ATTNQ_KV_REVERSE
    # P-cast page section 4: (1) forward S=1 vs the optimised configurations
    # near delta = 7; (2) forward S=256 vs forward S=448; (3) reverse+256 vs
    # forward+256 in the collapse regime; (4) the gain's growth with N
    gain_n = {}
    for n_tokens in (1024, 2048, 4096):
        r = res if n_tokens == N else sweep_at(n_tokens, (7.0,), [(F, 1.0), (R, 256.0), (F, 256.0)])
        gain_n[str(n_tokens)] = r[(7.0, F, 1.0)][0] / r[(7.0, R, 256.0)][0]
    qual = {
        "fwd_S1_over_rev_S256_mse_at_delta": {str(int(x)): mse(x, F, 1.0) / mse(x, R, 256.0) for x in (6.0, 7.0, 8.0)},
        "fwd_S1_over_fwd_S256_mse_at_delta": {str(int(x)): mse(x, F, 1.0) / mse(x, F, 256.0) for x in (6.0, 7.0, 8.0)},
        "fwd_S256_mse_below_fwd_S448_pct": {str(int(x)): 100.0 * (1.0 - mse(x, F, 256.0) / mse(x, F, 448.0))
                                            for x in deltas},
        "rev_S256_over_fwd_S256_mse": {str(int(x)): mse(x, R, 256.0) / mse(x, F, 256.0) for x in deltas},
        "fwd_S1_over_rev_S256_mse_by_N_at_delta7": gain_n,
    }
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        from oracle import closed_forms as cf
        t0 = time.perf_counter()
        orc = {}
        for delta in deltas:
            q, k, v = synth.pcast_sweep_inputs(delta)
            exact = oracle.attn_exact(q, k, v)
            for order, S in runs:
                emu, uref = oracle.attn_ponly(q, k, v, S, order, True, T)
                orc[(delta, order, S)] = (emu, uref.astype(np.int64), exact)
        dt = time.perf_counter() - t0
        worst_rel, worst_cnt = 0.0, 0.0
        for row in table:
            order = F if row["order"] == "fwd" else R
            key = (row["delta"], order, row["S"])
            emu, uref, exact = orc[key]
            o = res[key][3].reshape(emu.shape)
            rel = float(np.max(np.linalg.norm(o - emu, axis=(1, 2)) / np.linalg.norm(emu, axis=(1, 2))))
            worst_rel = max(worst_rel, rel)
            row["relF_vs_oracle"] = rel
            row["oracle_mse"] = float(np.mean((emu - exact) ** 2))
            row["oracle_underflow_fraction"] = float(uref.sum() / nonsink)
            tot = uref.sum()
            worst_cnt = max(worst_cnt, abs(row["underflow_tile0"] + row["underflow_later"] - tot) / max(tot, 1))
            row["F_closed_form"] = cf.underflow_fraction(row["delta"], row["S"]) if row["order"] == "fwd" else None
        cpu = {"value": dt, "unit": "s for the whole sweep (78 emulations + 13 exact FP64 attentions)",
               "cores": oracle.threads(), "kind": "oracle", "sample": "the whole sweep",
               "parity": {"max_relF_vs_oracle": worst_rel, "max_rel_count_diff": worst_cnt}}
    if args.report_md:
        _write_sweep_md(args.report_md, table, qual, ms_run, sweep_s, cpu, N)
    cfg = {"workload": "pcast_sweep", "B": B, "H": H, "N": N, "d": d, "kv_tile": T, "in_dtype": "f32",
           "deltas": list(deltas), "S": list(Ss), "kv_order": ["forward", "reverse"], "mode": "P-only",
           "step": "one attnq_fwd_ponly run (delta 7, reverse, S=256)", "l2": "inputs 50 MB (fit in L2)"}
    line = _common_line("P-cast sweep: MSE and non-sink underflow fraction per (delta, order, S)",
                        attn_flops(B, H, N, d) / (ms_run * 1e-3) / 1e12, "TFLOP/s (fp32 SIMT, one run)", args, True,
                        "f32 scores, e4m3 P", cfg, ms_per_run=ms_run, sweep_wall_s=sweep_s, qualitative=qual,
                        table=table, cpu_baseline=cpu, gpu_launches=args.steps)
    print(json.dumps(line), flush=True)
    return 0


def _write_sweep_md(path, table, qual, ms_run, sweep_s, cpu, N):
    cols = ("delta", "order", "S", "mse", "oracle_mse", "underflow_fraction", "oracle_underflow_fraction",
            "F_closed_form", "underflow_tile0", "underflow_later", "relF_vs_oracle")
    lines = [f"# P-cast isolation sweep (N = {N}, 8 heads, d = 128, KV tile 128, fp32 Q/K/V, only P cast)", "",
             "Command: `python bench.py --config 2 --report-md <this file>`", "",
             f"GPU: one attnq_fwd_ponly run {ms_run:.3f} ms; the whole sweep (78 runs, 13 FP64 references, "
             f"host copies and MSE on the host) {sweep_s:.1f} s wall.", ""]
    if cpu:
        lines += [f"Oracle: the whole sweep in {cpu['value']:.1f} s on {cpu['cores']} host threads; "
                  f"GPU vs oracle: max per-head rel-F {cpu['parity']['max_relF_vs_oracle']:.2e}, "
                  f"max relative count difference {cpu['parity']['max_rel_count_diff']:.2e}.", ""]
    lines += ["MSE: mean over all outputs of (O - O_FP64)^2.  Underflow fraction: in-mask non-sink P (key >= 4) "
              "with P*S > 0 cast to code 0, over all in-mask non-sink pairs; tile 0 / later tiles are the counts. "
              "F: the page's closed form Phi(delta + delta_4 - 10 ln 2 - ln S) (forward order only).", "",
              "| " + " | ".join(cols) + " |", "|" + "---|" * len(cols)]
    for r in table:
        cells = []
        for c in cols:
            x = r.get(c)
            if x is None:
                cells.append("")
            elif isinstance(x, float) and c not in ("delta", "S"):
                cells.append(f"{x:.4g}")
            else:
                cells.append(str(x))
        lines.append("| " + " | ".join(cells) + " |")
    lines += ["", "Qualitative results of the page's section 4, measured here (reported, not gated):", "",
              "```", json.dumps(qual, indent=1), "```", ""]
    with open(path, "w") as f:
        f.write("\n".join(lines))


def run_config34(args, name):
    """Qwen-shaped layers (qwen05b: 24 layers, 14/2 heads, d=64; qwen15b: 28
    layers, 12/2 heads, d=128; B=3, N=1024, S=256 reverse), four conditions
    each.  Timed: prepare + forward of every layer and condition (the FP8
    path, TFLOP/s), and the four-condition harm report per layer (FP64
    reference + four prepare/forward/error passes).  Reported: each
    condition's mean per-head log1p rel-F against FP64 and the number of heads
    rotation harms; in the cpu_baseline leg the oracle's whole-workload time
    and the largest per-head error difference from it."""
    import torch

    import precision_attention_numerics_gb300 as aq
    import synth
    wl = synth.WORKLOADS[name]
    B, Hq, Hkv, N, d, T, L = wl["B"], wl["Hq"], wl["Hkv"], wl["N"], wl["d"], wl["kv_tile"], wl["layers"]
    if args.layers:
        L = min(L, args.layers)
    dev = torch.device("cuda")
    aq.load_library()
    stream = torch.cuda.current_stream()
    signs_np = synth.qwen_signs(name)
    signs = torch.from_numpy(signs_np).to(dev)
    inputs = [synth.qwen_layer_inputs(name, layer) for layer in range(L)]
    dev_in = [tuple(_dev_tensor(a, dev) for a in x) for x in inputs]
    conds = list(synth.CONDITIONS.items())
    descs = [aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16,
                          (1 if r else 0) | (2 if c else 0) | aq.ATTNQ_VT_LAYOUT, signs) for _, (r, c) in conds]
    bufs = [aq.alloc_prepared(ds, device=dev) for ds in descs]
    O = torch.empty((B, Hq, N, d), dtype=torch.float32, device=dev)

    def fp8_step():
        for Q, K, V in dev_in:
            for ds, bf in zip(descs, bufs):
                aq.attnq_prepare(ds, Q, K, V, bf.q8, bf.k8, bf.v8, bf.scales, bf.workspace)
                aq.attnq_fwd(ds, bf.q8, bf.k8, bf.v8, bf.scales, 256.0, aq.ATTNQ_KV_REVERSE, True, T, O)

    ms_fp8_direct = _event_ms(fp8_step, args.warmup, args.steps, stream)
    ms_fp8 = _graph_ms(fp8_step, args.warmup, args.steps, stream)
    flops = attn_flops(B, Hq, N, d) * L * len(conds)
    rdesc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16, 0, signs)
    ws = torch.empty(aq.attnq_harm_workspace(rdesc), dtype=torch.uint8, device=dev)
    errs = torch.empty((L, 4, B * Hq), dtype=torch.float64, device=dev)

    def harm_all():
        for layer, (Q, K, V) in enumerate(dev_in):
            aq.attnq_harm_report(rdesc, Q, K, V, 256.0, aq.ATTNQ_KV_REVERSE, T, ws, errs[layer])

    ms_harm = _event_ms(harm_all, 1, max(1, min(args.steps, 3)), stream)
    st = aq.attnq_device_status()
    if st != 0:
        raise RuntimeError(f"device status {aq.STATUS.get(st, st)}")
    e = errs.cpu().numpy()                       # [L, 4, B*Hq]
    per_head = e.reshape(L, 4, B, Hq).mean(axis=2)  # mean over the batch ("texts")
    harm = per_head[:, 1] - per_head[:, 0]       # rotated - unrotated, per (layer, head)
    summary = {cname: float(per_head[:, i].mean()) for i, (cname, _) in enumerate(conds)}
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        worst = 0.0
        for layer, (q, k, v) in enumerate(inputs):
            exact = oracle.attn_exact(q, k, v)
            for i, (_, (r, c)) in enumerate(conds):
                fl = (1 if r else 0) | (2 if c else 0)
                prep = oracle.prepare(q, k, v, flags=fl, signs=signs_np)
                emu, _ = oracle.attn_quant(prep, (B, Hq, Hkv, N, d), fl, 256.0, 1, True, T)
                e_orc = oracle.err(emu, exact)
                worst = max(worst, float(np.max(np.abs(e[layer, i] - e_orc) / e_orc)))
        dt = time.perf_counter() - t0
        cpu = {"value": dt, "unit": f"s for all {L} layers (exact FP64 + four conditions)", "cores": oracle.threads(),
               "kind": "oracle", "sample": "the whole workload",
               "parity": {"max_rel_err_diff_per_head": worst, "bar": 0.05}}
    cfg = {"workload": name, "layers": L, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "kv_tile": T, "S": 256.0,
           "kv_order": "reverse", "in_dtype": "bf16", "out_dtype": "f32", "conditions": [c for c, _ in conds],
           "step": "attnq_prepare + attnq_fwd for every layer and condition", "l2": "no flush (layers rotate through L2)",
           "launch": "one CUDA graph replay per step (ms_per_step_direct: the same calls made directly)"}
    line = _common_line("causal FP8 attention fwd TFLOP/s over all layers and conditions; per-head log1p rel-F vs FP64",
                        flops / (ms_fp8 * 1e-3) / 1e12, "TFLOP/s", args, True, "e4m3", cfg,
                        ms_per_step=ms_fp8, ms_per_step_direct=ms_fp8_direct,
                        tflops_direct=flops / (ms_fp8_direct * 1e-3) / 1e12, harm_report_ms_per_layer=ms_harm / L,
                        mean_log1p_relF=summary, heads=int(L * Hq),
                        heads_harmed_by_rotation=int(np.sum(harm > 0)), cpu_baseline=cpu,
                        gpu_launches=args.steps * L * len(conds) * 3)
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch

    import precision_attention_numerics_gb300 as aq
    import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    aq.load_library()
    B, Hq, Hkv, N, d, T = WL["B"], WL["Hq"], WL["Hkv"], WL["N"], WL["d"], WL["kv_tile"]
    S = WL["S"]
    flags = aq.ATTNQ_ROTATE | aq.ATTNQ_CENTER_K | aq.ATTNQ_VT_LAYOUT
    if args.scales == "tile":
        flags |= aq.ATTNQ_TILE_SCALES
    i8 = args.qk == "int8"
    if i8:
        flags |= aq.ATTNQ_I8QK
    q_np, k_np, v_np = make_inputs(replica_seed(rank))
    signs_np = synth.hadamard_signs(17, d)
    dev = torch.device("cuda", local)
    # pinned host copies (end-to-end leg) and device-resident inputs
    Qh = torch.from_numpy(q_np).view(torch.bfloat16).pin_memory()
    Kh = torch.from_numpy(k_np).view(torch.bfloat16).pin_memory()
    Vh = torch.from_numpy(v_np).view(torch.bfloat16).pin_memory()
    Q, K, V = Qh.to(dev), Kh.to(dev), Vh.to(dev)
    signs = torch.from_numpy(signs_np).to(dev)
    desc = aq.AttnqDesc(B, Hq, Hkv, N, d, aq.ATTNQ_BF16, flags, signs, args.stat_len)
    bufs = aq.alloc_prepared(desc, device=dev)
    O = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=dev)
    Oh = torch.empty((B, Hq, N, d), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream(dev)

    def step():
        aq.attnq_prepare(desc, Q, K, V, bufs.q8, bufs.k8, bufs.v8, bufs.scales, bufs.workspace)
        aq.attnq_fwd(desc, bufs.q8, bufs.k8, bufs.v8, bufs.scales, S, aq.ATTNQ_KV_REVERSE, True, T, O)

    for _ in range(args.warmup):
        step()
    st = aq.attnq_device_status()
    if st != 0:
        raise RuntimeError(f"device status {aq.STATUS.get(st, st)} after warm-up")

    # ---- device-resident timed region, with per-call events for the roofline
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for s in range(args.steps):
            e0, e1, e2 = ev[s]
            e0.record(stream)
            aq.attnq_prepare(desc, Q, K, V, bufs.q8, bufs.k8, bufs.v8, bufs.scales, bufs.workspace)
            e1.record(stream)
            aq.attnq_fwd(desc, bufs.q8, bufs.k8, bufs.v8, bufs.scales, S, aq.ATTNQ_KV_REVERSE, True, T, O)
            e2.record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary()
    elapsed = start.elapsed_time(end) / 1e3
    prep_ms = sorted(e0.elapsed_time(e1) for e0, e1, _ in ev)
    fwd_ms = sorted(e1.elapsed_time(e2) for _, e1, e2 in ev)
    t_prep = sum(prep_ms) / args.steps / 1e3
    t_fwd = sum(fwd_ms) / args.steps / 1e3
    st = aq.attnq_device_status()
    if st != 0:
        raise RuntimeError(f"device status {aq.STATUS.get(st, st)} in the timed region")
    elapsed = max_over_ranks(elapsed, dist, dev)

    # ---- end-to-end through the C ABI's host-buffer pipeline: every step copies
    # its Q, K, V in from pinned host memory and its O back out; the copies of
    # step s+1's inputs and step s-1's output overlap step s's kernels
    e2e_elapsed = float("nan")
    e2e_clocks = None
    if not args.no_e2e:
        del bufs  # the pipeline keeps its own device buffers in its workspace
        compute, copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        pws = torch.empty(aq.attnq_host_pipeline_workspace(desc, aq.ATTNQ_BF16), dtype=torch.uint8, device=dev)

        def e2e_run(n):
            aq.attnq_attention_host(desc, [Qh] * n, [Kh] * n, [Vh] * n, S, aq.ATTNQ_KV_REVERSE, True, T, [Oh] * n,
                                    aq.ATTNQ_BF16, pws, compute, copy_in, copy_out)

        e2e_run(min(args.warmup, 2))
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as e2e_clk:
            s0.record(compute)
            e2e_run(args.steps)
            s1.record(compute)
            torch.cuda.synchronize()
        e2e_clocks = e2e_clk.summary()
        e2e_elapsed = s0.elapsed_time(s1) / 1e3
        st = aq.attnq_device_status(compute.cuda_stream)
        if st != 0:
            raise RuntimeError(f"device status {aq.STATUS.get(st, st)} in the end-to-end run")
        del pws
    h2d = (Qh.numel() + Kh.numel() + Vh.numel()) * 2
    d2h = Oh.numel() * 2

    flops_step = attn_flops(B, Hq, N, d)
    value = replica_value(flops_step, args.steps, world, elapsed)
    e2e_value = replica_value(flops_step, args.steps, world, e2e_elapsed)
    peaks = load_peaks()
    # The timed region is well under a second at full clocks, so the burst
    # peaks apply.  FP8: this GPU's own dense E4M3 GEMM rate, measured here
    # after the timed region; twice the bf16 burst figure (the nominal
    # 4.5 : 2.25 ratio) only if that measurement is unavailable.
    fp8_meas = measure_fp8_peak(dev) if not args.no_fp8_peak else {"tflops": None, "error": "skipped"}
    if fp8_meas.get("tflops"):
        fp8_peak, fp8_src = fp8_meas["tflops"], f"measured here: {fp8_meas['method']}"
    else:
        fp8_peak = 2.0 * peaks["bf16"]
        fp8_src = (f"{peaks['source']} bf16 burst {peaks['bf16']} x 2 (nominal fp8:bf16 ratio; FP8 GEMM "
                   f"not measured: {fp8_meas.get('error')})")
    # INT8-QK: half the flops (Q K^T) on the bf16 path, half (P V) on fp8, so
    # the step's tensor peak is 1 / (0.5 / bf16 + 0.5 / fp8)
    mma_peak = 1.0 / (0.5 / peaks["bf16"] + 0.5 / fp8_peak) if i8 else fp8_peak
    fwd_tflops = flops_step / t_fwd / 1e12
    prep_bytes = prepare_bytes(B, Hq, Hkv, N, d, qk_code_bytes=2 if i8 else 1)
    prep_gbs = prep_bytes / t_prep / 1e9
    fwd_hash = kernel_source_hash(["attn_fwd.cu", "ptx.cuh"])
    full_size = (B, Hq, Hkv) == (2, 32, 8)  # the captures are of the full workload
    # traffic is recorded per kernel and per workload variant
    tag = ("_i8" if i8 else "") + ("_tile" if args.scales == "tile" else "") + (f"_p{args.stat_len}" if args.stat_len else "")
    prep_hash = kernel_source_hash(["prepare.cu", "ptx.cuh"])

    line = None
    if rank == 0:
        # per-head error against FP64 on a row sample (oracle, outside the timed region)
        import oracle
        rows = np.unique(np.array([0, 1, 127, 4095, N // 2 - 1, N // 2, N - 1], dtype=np.int64))
        bh = sorted({h for h in (0, B * Hq // 2 - 1, B * Hq // 2 + 5, B * Hq - 1) if 0 <= h < B * Hq})
        Og = O.view(B * Hq, N, d)[bh][:, rows].float().cpu().numpy().astype(np.float64)
        exact = oracle.attn_exact(q_np, k_np, v_np, bh_list=bh, rows=rows)
        rel = np.linalg.norm(Og - exact, axis=(1, 2)) / np.linalg.norm(exact, axis=(1, 2))
        err_sample = {"mean_log1p_relF": float(np.mean(np.log1p(rel))), "heads": bh,
                      "rows": rows.tolist(), "reference": "oracle exact FP64 attention"}
        cpu = None
        if not args.no_cpu_baseline:
            rows_s = sample_rows(args.cpu_rows)
            dt, fl, thr = oracle_sample(q_np, k_np, v_np, signs_np, rows_s, stat_len=args.stat_len,
                                        extra_flags=oracle.I8QK if i8 else 0)
            t_prep_g, t_emu = oracle_sample.split
            full_s = extrapolated_oracle_step(t_prep_g, t_emu, fl)
            cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                   "sample": (f"oracle prepare of one (batch, KV group) (4 query heads, 1 KV head) + quantised "
                              f"emulation of {len(rows_s)} query rows in [N/2, N) of those heads; "
                              f"{dt:.1f} s of CPU time"),
                   "extrapolated_step_s": full_s,
                   "extrapolated_note": (f"extrapolated: prepare {t_prep_g:.2f} s per (batch, KV group) x "
                                         f"{B * Hkv} groups + emulation {t_emu:.2f} s x causal pairs of the whole "
                                         f"step / of the sample"),
                   "extrapolated_speedup_of_gpu_step": full_s / (elapsed / args.steps)}
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8-qk/e4m3-pv" if i8 else "e4m3", "data": "synthetic",
            "config": {"workload": "long_context" if (B, Hq, Hkv) == (2, 32, 8) else "long_context_reduced", **WL, "rotate": True, "center_k": True, "scales": "per-tile (128 tokens)" if args.scales == "tile" else "per (batch, head)",
                       "statistics": f"first {args.stat_len} tokens" if args.stat_len else "full sequence",
                       "qk_codes": "int8 (held in bf16)" if i8 else "e4m3", "in_dtype": "bf16",
                       "out_dtype": "bf16", "step": "attnq_prepare + attnq_fwd",
                       "l2": "inputs 805 MB per step > 129 MB L2; no flush",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            # the whole step's TFLOP/s against the same tensor peak as the roofline
            "pct_fp8_peak": 100.0 * value / world / mma_peak,
            "fp8_gemm_peak": fp8_meas,
            "roofline": {"kernel": "attnq_fwd (k_attn_fwd<128,128>)", "bound": "tensor", "achieved": fwd_tflops,
                         "peak": mma_peak, "unit": "TFLOP/s", "frac": fwd_tflops / mma_peak,
                         "traffic": ncu_traffic("k_attn_fwd" + tag, fwd_hash) if full_size else None,
                         "peak_note": ((f"1 / (0.5 / bf16 burst {peaks['bf16']} + 0.5 / fp8 {fp8_peak:.1f}): Q K^T on "
                                        f"the bf16 path, P V on fp8; fp8 {fp8_src}") if i8 else
                                       f"fp8 dense, burst: {fp8_src}"),
                         "flops_per_launch": flops_step, "ms_per_launch": t_fwd * 1e3,
                         "ms_median": statistics.median(fwd_ms), "ms_best": fwd_ms[0],
                         # the dense datasheet figure, for context (GB300: 4.5 PFLOP/s FP8, 2.25 bf16)
                         "datasheet": {"peak": DATASHEET_MMA_TFLOPS["int8" if i8 else "e4m3"],
                                       "frac": fwd_tflops / DATASHEET_MMA_TFLOPS["int8" if i8 else "e4m3"]}},
            "roofline_prepare": {"kernel": "attnq_prepare (all passes)", "bound": "hbm", "achieved": prep_gbs,
                                 "peak": peaks["hbm"], "unit": "GB/s", "frac": prep_gbs / peaks["hbm"],
                                 "traffic": ncu_traffic("attnq_prepare" + tag, prep_hash) if full_size else None,
                                 "bytes_per_launch": prep_bytes, "ms_per_launch": t_prep * 1e3,
                                 "ms_median": statistics.median(prep_ms), "ms_best": prep_ms[0]},
            "err_vs_fp64": err_sample,
            "cpu_baseline": cpu,
            "e2e": None if args.no_e2e else {
                "value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_elapsed / args.steps * 1e3, "clocks": e2e_clocks},
            "clocks": clocks,
            "device": device_info(dev),
            "gpu_launches": args.steps * launches_per_step(flags),
        }
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=3072)
    ap.add_argument("--ref-rows", type=int, default=96)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--no-fp8-peak", action="store_true",
                    help="skip the FP8 GEMM peak measurement (profiling runs; the roofline then uses 2 x bf16)")
    ap.add_argument("--scales", choices=["slice", "tile"], default="slice",
                    help="Q/K scales per (batch, head) (the timed workload) or per 128-token tile")
    ap.add_argument("--qk", choices=["e4m3", "int8"], default="e4m3",
                    help="Q/K code format: E4M3 (the timed workload) or INT8 (INT8-QK / FP8-PV)")
    ap.add_argument("--stat-len", type=int, default=0,
                    help="causal-prefix statistics: mean key and slice scales over the first P tokens (0: all N)")
    ap.add_argument("--B", type=int, default=WL["B"], help="smaller batch for profiling captures")
    ap.add_argument("--Hq", type=int, default=WL["Hq"])
    ap.add_argument("--Hkv", type=int, default=WL["Hkv"])
    ap.add_argument("--report", choices=["step", "harm"], default="step",
                    help="harm: time the four-condition harm report on a Qwen-0.5B-shaped layer instead")
    ap.add_argument("--config", type=int, choices=[1, 2, 3, 4, 5], default=5,
                    help="workload: 1 sink probe, 2 P-cast sweep, 3/4 Qwen-0.5B/1.5B-shaped layers, "
                         "5 long context (the default line)")
    ap.add_argument("--layers", type=int, default=0, help="configs 3/4: first L layers only (0: all)")
    ap.add_argument("--report-md", default="", help="config 2: also write the sweep table as markdown here")
    args = ap.parse_args()
    WL.update(B=args.B, Hq=args.Hq, Hkv=args.Hkv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.config != 5:
        torch_dev = int(os.environ.get("LOCAL_RANK", "0"))
        import torch
        torch.cuda.set_device(torch_dev)
        return {1: run_config1, 2: run_config2, 3: lambda a: run_config34(a, "qwen05b"),
                4: lambda a: run_config34(a, "qwen15b")}[args.config](args)
    if args.report == "harm":
        return run_harm(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
