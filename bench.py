"""Benchmark of the MXAttention MXFP4 forward hot path on GB300.

One step = the whole hot path over one batch of synthetic input:
mxattn_quantize_qkv (Q and K rotated and quantized, V quantized: one launch)
and mxattn_forward -- two kernel launches on one stream, inputs resident in HBM.

Default workload: the video-DiT shaped configuration B=1, H=40, N=32760
(21x30x52 latent tokens), d=128, non-causal, seeded synthetic bf16 Q, K, V
(standard normal with 4 outlier channels x20 in Q and K). The 1.0 GB of inputs
is larger than the 129 MB L2, so no flush is needed between steps.

Prints one JSON line (metric: TFLOPS = 4*B*H*N*N*d per step / time).
  --impl reference  times the float64 CPU oracle on the host cores instead,
                    each step a bounded sample of the same workload.
Multi-GPU (torchrun, one rank per GPU): every rank runs its own copy of the
workload (the path shards by independent heads; no collective touches the
data), timing is the max over ranks, and value is the aggregate.
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

METRIC = "MXFP4 attention fwd TFLOPS and % of GB300 dense FP4 peak (Wan-shaped N=32760)"
UNIT = "TFLOPS"
FP4_OVER_BF16_NOMINAL = 13.5 / 2.25  # nominal dense FP4 / BF16 tensor rate on GB300
NOMINAL_FP4_TFLOPS = 13500.0  # nominal dense FP4 tensor rate of one GB300


# DRAM bytes of one forward launch from an ncu capture (dram__bytes_read.sum,
# dram__bytes_write.sum) of the full Wan-shaped launch (B*H = 40, N = 32760;
# the 671 MB fp32 output is 5x the L2, so at most the L2's dirty residue at
# exit goes uncounted), with a fingerprint of the kernel source it was taken
# on. `traffic` is reported (scaled by B*H) only while the source still has
# that fingerprint; otherwise it is null.
FWD_TRAFFIC_CAPTURE = {
    "fingerprint": "29121bc444881720",
    "bh": 40, "n": 32760,
    "read_bytes": 268373504, "write_bytes": 614174464,
}
FWD_SOURCES = ("attn_mxfp4.cu", "sm103_ptx.cuh", "internal.h")


def kernel_fingerprint() -> str:
    """sha256 of the forward kernel's sources with comments and blank space removed."""
    import hashlib
    import re

    h = hashlib.sha256()
    for name in FWD_SOURCES:
        with open(os.path.join(ROOT, "mxfp4_precision_attention_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(name.encode())
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def fwd_traffic(bh: int, n: int):
    """(read, write) DRAM bytes of one forward launch at B*H = bh, N = n, from the
    capture above, or None if the kernel source or N differs from the capture's."""
    c = FWD_TRAFFIC_CAPTURE
    if c["fingerprint"] != kernel_fingerprint() or n != c["n"]:
        return None
    return c["read_bytes"] * bh / c["bh"], c["write_bytes"] * bh / c["bh"]


def fwd_algorithmic_bytes(bh: int, n: int, out_bytes: int = 4) -> int:
    """The forward's own bytes: Q^, K^, V^ codes and scale atoms read once, O written once."""
    nt = (n + 127) // 128
    codes = 2 * bh * n * 64 + bh * 128 * ((n + 31) // 32 * 32) // 2
    return codes + 3 * bh * nt * 512 + bh * n * 128 * out_bytes


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

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
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(w, rank: int) -> int:
    """Seed of rank `rank`'s replica: every rank runs the whole workload on its own inputs."""
    return w.seed + rank


def max_over_ranks(x: float, device) -> float:
    """The maximum of `x` over all ranks of the default process group (x itself
    without one). `device` is where the collective's tensor lives: the GPU for
    NCCL, the CPU for gloo."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, flops_per_step: float, steps: int, seconds: float) -> float:
    """Whole-job TFLOPS: every rank's steps over the slowest rank's time."""
    return world * flops_per_step * steps / seconds / 1e12


def cpu_oracle_sample(w, budget_rows: int, seed: int = 0):
    """Time the oracle on a bounded sample of workload `w`: per sampled head, its
    K and V quantized in full plus up to N query rows through the forward, over
    as many heads as `budget_rows` needs. Returns (seconds, flops, description,
    threads, rows)."""
    import numpy as np

    import oracle
    from mxfp4_precision_attention_gb300 import workloads as W

    oracle.build()
    rows_left = max(1, int(budget_rows))
    nheads = (rows_left + w.N - 1) // w.N
    dt, flops, rows_done = 0.0, 0.0, 0
    for hh in range(nheads):
        q, k, v = W.generate(w, device="cpu", B=1, H=1, seed=w.seed + 1000 * seed + hh)
        qb, kb, vb = (W.as_u16(t).reshape(1, w.N, 128) for t in (q, k, v))
        rng = np.random.default_rng(seed * 7919 + hh)
        nr = min(rows_left, w.N)
        toks = np.sort(rng.choice(w.N, size=nr, replace=False))
        t0 = time.perf_counter()
        qc, qs = oracle.rotate_quantize_qk(qb[:, toks])
        kc, ks = oracle.rotate_quantize_qk(kb)
        vc, vs = oracle.quantize_v(vb)
        qc_full = np.zeros((1, w.N, 128), dtype=np.uint8)
        qs_full = np.full((1, w.N, 4), 127, dtype=np.uint8)
        qc_full[:, toks], qs_full[:, toks] = qc, qs
        rows = np.stack([np.zeros_like(toks), toks], axis=1)
        oracle.forward(qc_full, qs_full, kc, ks, vc, vs, rows, vraw_u16=vb, causal=w.causal)
        dt += time.perf_counter() - t0
        if w.causal:
            flops += float(sum(4.0 * (int(t) + 1) * 128 for t in toks))
        else:
            flops += 4.0 * len(toks) * w.N * 128
        rows_left -= nr
        rows_done += nr
    desc = (f"{nheads} head(s) of {w.name}: per head rotate+quantize the sampled Q rows and all {w.N} K tokens, "
            f"quantize all V, float64 forward for the sampled rows against all keys ({rows_done} rows in total)")
    return dt, flops, desc, oracle.num_threads(), rows_done


def cpu_extrapolation(w, seconds: float, flops: float, rows: int) -> dict:
    """Rows per second of the sample and a linear extrapolation of the sample's
    rate (FLOP per second) to the whole workload."""
    return {"rows_per_s": rows / seconds, "extrapolated_full_workload_s": w.flops / (flops / seconds),
            "extrapolation": "linear in FLOP from the sample's rate"}


# The other seeded workloads, each timed in the same run as the headline line
# (parity-test configurations, reported beside it; the tiny 512-token case is
# launch-bound and left out).
PER_WORKLOAD = ("lognormal_4096", "wan_32760", "hunyuan_118800", "causal_lm_8192")


def time_workload(mx, W, w, stream, fp4_peak: float, hbm: float, cpu_s: float, reps: int = 5) -> dict:
    """Forward and one-launch quantizer of workload `w`, CUDA events on `stream`
    (3 warm-up launches, then the mean of `reps`), with its roofline fraction and,
    if cpu_s > 0, the oracle timed on a bounded sample of the same workload."""
    import torch

    B, H, N = w.B, w.H, w.N
    q, k, v = W.generate(w, device="cuda")
    dev = q.device
    qcn, qsn = mx.qk_layout_sizes(B, H, N)
    vcn, vsn = mx.v_layout_sizes(B, H, N)
    bufs = [torch.empty(n, dtype=torch.uint8, device=dev) for n in (qcn, qsn, qcn, qsn, vcn, vsn)]
    out = torch.empty((B, H, N, 128), dtype=torch.float32, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with torch.cuda.stream(stream):
        for rep in range(3 + reps):
            if rep == 3: ev[0].record(stream)
            mx.mxattn_quantize_qkv(q, k, v, out=tuple(bufs), stream=stream)
        ev[1].record(stream)
        for rep in range(3 + reps):
            if rep == 3: ev[2].record(stream)
            mx.mxattn_forward(*bufs, v, B, H, N, causal=w.causal, out=out, stream=stream)
        ev[3].record(stream)
    torch.cuda.synchronize()
    mx.mxattn_check(stream)
    q_ms = ev[0].elapsed_time(ev[1]) / reps
    f_ms = ev[2].elapsed_time(ev[3]) / reps
    e = B * H * N * 128
    qb = 3 * e * 2 + 2 * (qcn + qsn) + vcn + vsn
    tf = w.flops / (f_ms * 1e-3) / 1e12
    res = {"B": B, "H": H, "N": N, "causal": w.causal, "forward_ms": f_ms, "tflops": tf, "frac": tf / fp4_peak,
           "quantize_qkv_ms": q_ms, "quantizer_gbs": qb / (q_ms * 1e-3) / 1e9,
           "quantizer_frac_of_hbm": qb / (q_ms * 1e-3) / 1e9 / hbm,
           "step_tflops": w.flops / ((f_ms + q_ms) * 1e-3) / 1e12}
    del q, k, v, bufs, out
    torch.cuda.empty_cache()
    if cpu_s > 0:
        dt0, _, _, _, _ = cpu_oracle_sample(w, 64)
        rows = int(max(8, min(200000, cpu_s / max(dt0 / 64, 1e-6))))
        dt, fl, desc, thr, nr = cpu_oracle_sample(w, rows, seed=3)
        res["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
                               "sample": desc, "seconds": dt, **cpu_extrapolation(w, dt, fl, nr)}
    return res


def run_reference(args, w):
    world, rank, _ = _dist()
    if rank != 0:
        return
    # calibrate the sample so that one step costs ~ args.ref_step_s seconds
    dt, fl, _, _, _ = cpu_oracle_sample(w, 256)
    per_row = max(dt / 256, 1e-6)
    rows = int(max(8, min(200000, args.ref_step_s / per_row)))
    for i in range(args.warmup):
        cpu_oracle_sample(w, max(4, rows // 8), seed=100 + i)
    times, flops, nrows = [], [], 0
    for i in range(args.steps):
        dt, fl, desc, thr, nr = cpu_oracle_sample(w, rows, seed=i)
        times.append(dt)
        flops.append(fl)
        nrows += nr
    total_t, total_f = sum(times), sum(flops)
    value = total_f / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": 128, "causal": w.causal,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": desc,
                         **cpu_extrapolation(w, total_t, total_f, nrows)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import mxfp4_precision_attention_gb300 as mx
    from mxfp4_precision_attention_gb300 import workloads as W

    mx.load()
    hbm, bf16, bf16_sus, peak_src = _peaks()
    fp4_peak = bf16 * FP4_OVER_BF16_NOMINAL
    B, H, N = w.B, w.H, w.N
    q, k, v = W.generate(w, device="cuda", seed=rank_seed(w, rank))
    qcn, qsn = mx.qk_layout_sizes(B, H, N)
    vcn, vsn = mx.v_layout_sizes(B, H, N)
    dev = q.device
    qc = torch.empty(qcn, dtype=torch.uint8, device=dev)
    qs = torch.empty(qsn, dtype=torch.uint8, device=dev)
    kc = torch.empty(qcn, dtype=torch.uint8, device=dev)
    ks = torch.empty(qsn, dtype=torch.uint8, device=dev)
    vc = torch.empty(vcn, dtype=torch.uint8, device=dev)
    vs = torch.empty(vsn, dtype=torch.uint8, device=dev)
    out = torch.empty((B, H, N, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream()
    n_events = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_events)]

    def step(i=None):
        e = ev[i] if i is not None else None
        if e: e[0].record(stream)
        mx.mxattn_quantize_qkv(q, k, v, out=(qc, qs, kc, ks, vc, vs), stream=stream)
        if e: e[1].record(stream)
        mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, B, H, N, causal=w.causal, out=out, stream=stream)
        if e: e[2].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    mx.mxattn_check(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    mx.mxattn_check(stream)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
    if world > 1:
        torch.distributed.barrier()
    qkv_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(n_events))
    fwd_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(n_events))
    flops = w.flops
    value = job_value(world, flops, args.steps, total_ms * 1e-3)
    fwd_tflops = flops / (fwd_ms * 1e-3) / 1e12
    e = B * H * N * 128
    qkv_bytes = 2 * (e * 2 + qcn + qsn) + e * 2 + vcn + vsn

    # the three single-tensor quantizer calls, for comparison with the one launch (not part of the step)
    single = None
    with torch.cuda.stream(stream):
        s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for rep in range(4):
            if rep == 3: s_ev[0].record(stream)
            mx.mxattn_rotate_quantize_qk(q, qc, qs, stream=stream)
            mx.mxattn_rotate_quantize_qk(k, kc, ks, stream=stream)
            if rep == 3: s_ev[1].record(stream)
            mx.mxattn_quantize_v(v, vc, vs, stream=stream)
            if rep == 3: s_ev[2].record(stream)
    torch.cuda.synchronize()
    mx.mxattn_check(stream)
    single = {"rotate_quantize_qk_x2_ms": s_ev[0].elapsed_time(s_ev[1]), "quantize_v_ms": s_ev[1].elapsed_time(s_ev[2])}

    # the forward writing bf16 instead of fp32 (not part of the step, whose output is fp32)
    o16 = torch.empty((B, H, N, 128), dtype=torch.bfloat16, device=dev)
    b_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        for rep in range(4):
            if rep == 1: b_ev[0].record(stream)
            mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, B, H, N, causal=w.causal, out=o16, stream=stream,
                              out_dtype=torch.bfloat16)
        b_ev[1].record(stream)
    torch.cuda.synchronize()
    mx.mxattn_check(stream)
    fwd_bf16out_ms = b_ev[0].elapsed_time(b_ev[1]) / 3
    del o16

    # the BF16 comparison path on the same inputs (not part of the step)
    bf16_path = None
    if not args.no_bf16:
        with torch.cuda.stream(stream):
            for _ in range(2):
                mx.mxattn_forward_bf16(q, k, v, causal=w.causal, out=out, stream=stream)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for _ in range(3):
                mx.mxattn_forward_bf16(q, k, v, causal=w.causal, out=out, stream=stream)
            b1.record(stream)
        torch.cuda.synchronize()
        mx.mxattn_check(stream)
        bms = b0.elapsed_time(b1) / 3
        bt = flops / (bms * 1e-3) / 1e12
        bf16_path = {"kernel": "bf16_fwd_kernel (tcgen05 kind::f16)", "ms": bms, "tflops": bt,
                     "frac_of_bf16_peak": bt / bf16, "mxfp4_speedup": bms / fwd_ms}
        # context: the library BF16 attention on the same tensors (torch SDPA, bf16 output)
        try:
            import torch.nn.functional as F

            with torch.cuda.stream(stream):
                for _ in range(2):
                    F.scaled_dot_product_attention(q, k, v, is_causal=w.causal)
                l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                l0.record(stream)
                for _ in range(3):
                    F.scaled_dot_product_attention(q, k, v, is_causal=w.causal)
                l1.record(stream)
            torch.cuda.synchronize()
            lms = l0.elapsed_time(l1) / 3
            bf16_path["library_sdpa"] = {"api": "torch.nn.functional.scaled_dot_product_attention (bf16)",
                                         "ms": lms, "tflops": flops / (lms * 1e-3) / 1e12,
                                         "mxfp4_speedup": lms / fwd_ms}
        except Exception as ex:  # no fused backend for this GPU / torch build
            bf16_path["library_sdpa"] = {"unavailable": str(ex)[:200]}

    # the NVFP4 comparison path on the same inputs (not part of the step): its
    # quantizers (amax pass + tiles, per tensor) and the kind::mxf4nvf4 forward
    nvfp4_path = None
    if not args.no_nvfp4:
        with torch.cuda.stream(stream):
            n_ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            for rep in range(3):
                if rep == 2: n_ev[0].record(stream)
                qt = mx.mxattn_nvfp4_quantize_qk(q, stream=stream)
                kt = mx.mxattn_nvfp4_quantize_qk(k, stream=stream)
                vt = mx.mxattn_nvfp4_quantize_v(v, stream=stream)
                if rep == 2: n_ev[1].record(stream)
            for rep in range(5):
                if rep == 2: n_ev[2].record(stream)
                mx.mxattn_nvfp4_forward(qt, kt, vt, v, B, H, N, causal=w.causal, placement=1, out=out, stream=stream)
            n_ev[3].record(stream)
        torch.cuda.synchronize()
        mx.mxattn_check(stream)
        nq_ms = n_ev[0].elapsed_time(n_ev[1])
        nf_ms = n_ev[2].elapsed_time(n_ev[3]) / 3
        nt = flops / (nf_ms * 1e-3) / 1e12
        nvfp4_path = {"kernel": "mxfp4_fwd_kernel NVFP4 instantiation (tcgen05 kind::mxf4nvf4 scale_vec::4X, UE4M3)",
                      "placement": "direct (the baseline)", "forward_ms": nf_ms, "tflops": nt,
                      "frac_of_fp4_peak": nt / fp4_peak, "quantize_ms": nq_ms, "mxfp4_speedup": nf_ms / fwd_ms}
        del qt, kt, vt

    # the dense FP4 MMA rate of this GPU (not part of the step): the tensor-core
    # probe's back-to-back kind::mxf4 M128 K64 MMAs, N = 256 and the forward's
    # own N = 128, for about a second each
    mma_probe = None
    if not args.no_mma_probe:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mma_probe = {"kernel": "mxf4_mma_rate_kernel (tcgen05 kind::mxf4 M128 Nn K64 back to back, one CTA per SM)",
                     "nominal_dense_fp4_tflops": NOMINAL_FP4_TFLOPS, "forward_tflops": fwd_tflops}
        for n in (256, 128):
            p_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            with torch.cuda.stream(stream):
                mx.mxattn_mxf4_mma_rate(2000, n=n, stream=stream)
                p_ev[0].record(stream)
                mx.mxattn_mxf4_mma_rate(20000, n=n, stream=stream)
                p_ev[1].record(stream)
            torch.cuda.synchronize()
            mx.mxattn_check(stream)
            per_iter_ms = p_ev[0].elapsed_time(p_ev[1]) / 20000
            iters = int(min(1 << 27, max(20000, args.mma_probe_s * 1e3 / per_iter_ms)))
            probe_clocks = ClockSampler(local)
            probe_clocks.start()
            with torch.cuda.stream(stream):
                p_ev[0].record(stream)
                pfl = mx.mxattn_mxf4_mma_rate(iters, n=n, stream=stream)
                p_ev[1].record(stream)
            torch.cuda.synchronize()
            pclk = probe_clocks.stop()
            mx.mxattn_check(stream)
            pms = p_ev[0].elapsed_time(p_ev[1])
            pt = pfl / (pms * 1e-3) / 1e12
            mhz = pclk.get("sm_mhz")
            mma_probe[f"n{n}"] = {
                "tflops": pt, "ms": pms, "iters_per_cta": iters, "clocks": pclk,
                "frac_of_nominal": pt / NOMINAL_FP4_TFLOPS,
                "flop_per_clock_per_sm": pt * 1e12 / (sms * mhz * 1e6) if mhz else None,
                "forward_frac": fwd_tflops / pt}

    # end to end through the host-buffer entry point (pinned host memory)
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        outh = torch.empty((B, H, N, 128), dtype=torch.float32).pin_memory()
        del q, k, v, qc, qs, kc, ks, vc, vs, out
        torch.cuda.empty_cache()
        ws = torch.empty(mx.mxattn_workspace_bytes(B, H, N), dtype=torch.uint8, device=dev)
        mx.mxattn_attention_host(qh, kh, vh, w.causal, outh, ws, stream=stream)
        steps_e2e = max(1, args.steps)
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(steps_e2e):
            mx.mxattn_attention_host(qh, kh, vh, w.causal, outh, ws, stream=stream)
        dt = max_over_ranks(time.perf_counter() - t0, dev)
        e2e = {"value": job_value(world, flops, steps_e2e, dt), "unit": UNIT,
               "h2d_bytes_per_step": 3 * e * 2, "d2h_bytes_per_step": e * 4, "steps": steps_e2e,
               "api": "mxattn_attention_host (pinned host buffers, copies inside the timed region)"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        dt0, _, _, _, _ = cpu_oracle_sample(w, 256)
        rows = int(max(8, min(200000, args.cpu_budget_s / max(dt0 / 256, 1e-6))))
        dt, fl, desc, thr, nr = cpu_oracle_sample(w, rows, seed=1)
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": desc,
               "seconds": dt, **cpu_extrapolation(w, dt, fl, nr)}

    per_workload = None
    if rank == 0 and not args.no_per_workload:
        per_workload = {}
        for pname in PER_WORKLOAD:
            if pname == w.name:
                continue
            per_workload[pname] = time_workload(mx, W, W.WORKLOADS[pname], stream, fp4_peak, hbm,
                                                cpu_s=0 if args.no_cpu_baseline else args.per_workload_cpu_s)

    traffic = fwd_traffic(B * H, N)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4",
            "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": 128, "causal": w.causal,
                       "parallelism": (f"replicas x{world}: every rank runs the whole workload on its own seeded "
                                       "inputs (weak scaling); no collective"),
                       "l2": f"inputs {3 * e * 2 / 1e9:.2f} GB per step vs 129 MB L2; no flush"},
            "roofline": {"bound": "tensor", "achieved": fwd_tflops, "peak": fp4_peak, "unit": "TFLOP/s",
                         "frac": fwd_tflops / fp4_peak,
                         "traffic": None if traffic is None else traffic[0] + traffic[1],
                         "traffic_read": None if traffic is None else traffic[0],
                         "traffic_write": None if traffic is None else traffic[1],
                         "algorithmic_bytes": fwd_algorithmic_bytes(B * H, N),
                         "traffic_note": ("DRAM bytes per launch (ncu dram__bytes_read/write.sum of the full 40-head "
                                          "launch of the same kernel source, scaled by B*H); writes still dirty in L2 "
                                          "at kernel exit are not counted"),
                         "kernel": "mxfp4_fwd_kernel",
                         "peak_source": f"{peak_src} bf16 {bf16:.1f} TF/s x nominal fp4/bf16 ratio {FP4_OVER_BF16_NOMINAL:g}"},
            "breakdown_ms": {"quantize_qkv": qkv_ms, "forward": fwd_ms},
            "forward_out_bf16_ms": fwd_bf16out_ms,
            "quantizer": {"kernel": "quantize_qkv_roles_kernel (one launch for Q, K, V)",
                          "algorithmic_bytes": qkv_bytes, "gbs": qkv_bytes / (qkv_ms * 1e-3) / 1e9,
                          "frac_of_hbm": qkv_bytes / (qkv_ms * 1e-3) / 1e9 / hbm, "hbm_peak": hbm,
                          "single_calls": single},
            "gpu_launches": 2 * args.steps,
            "per_workload": per_workload,
            "bf16_path": bf16_path,
            "nvfp4_path": nvfp4_path,
            "fp4_mma_probe": mma_probe,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# Table 3 of the paper (section 5.4), top to bottom, then TFS:
# (name, scale rule of Q/K/V/P~, rotate, placement of l)
ABLATION = [
    ("full (rotation + PNQ + UOS)", 0, True, 0),
    ("without UOS (OCP)", 1, True, 0),
    ("without UOS, PNQ (OCP + direct l)", 1, True, 1),
    ("plain OCP MXFP4 (no rotation, direct l)", 1, False, 1),
    ("rotation + PNQ + TFS", 2, True, 0),
]


def _e2m1_lut(device):
    import torch

    return torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], device=device)


def _atom_rows(device):
    """[128 rows, 4 blocks] -> byte offset in a 512-byte scale atom (include/mxattn.h)."""
    import torch

    r = torch.arange(128, device=device)[:, None]
    k = torch.arange(4, device=device)[None, :]
    return (r % 32) * 16 + (r // 32) * 4 + k


def _dequant_qk(codes, scales, BH, N):
    """Q/K codes [BH][N][64] and scale atoms -> float32 [BH, N, 128]."""
    import torch

    lut = _e2m1_lut(codes.device)
    c = codes.view(BH, N, 64).long()
    vals = torch.stack([lut[c & 15], lut[c >> 4]], -1).view(BH, N, 128)
    NT = (N + 127) // 128
    sb = scales.view(BH, NT, 512)[:, :, _atom_rows(codes.device)].reshape(BH, NT * 128, 4)[:, :N]
    return vals * torch.exp2(sb.float() - 127).repeat_interleave(32, -1)


def _dequant_v(codes, scales, BH, N):
    """V codes [BH][128][Npad/2] and scale atoms -> float32 [BH, N, 128]."""
    import torch

    lut = _e2m1_lut(codes.device)
    npad = (N + 31) // 32 * 32
    c = codes.view(BH, 128, npad // 2).long()
    vals = torch.stack([lut[c & 15], lut[c >> 4]], -1).view(BH, 128, npad)[:, :, :N]
    NT = (N + 127) // 128
    sb = scales.view(BH, NT, 512)[:, :, _atom_rows(codes.device)]          # [BH, NT, 128 ch, 4 blocks]
    sb = sb.permute(0, 2, 1, 3).reshape(BH, 128, NT * 4).repeat_interleave(32, -1)[:, :, :N]
    return (vals * torch.exp2(sb.float() - 127)).transpose(1, 2)


def run_qmax_sweep(mx, W, names):
    """Section 5.5.1: for every head and tensor (rotated Q, rotated K, V), the Q_max in
    6.00 .. 8.00 (steps of 0.05) that minimizes the block quantizer's MSE."""
    import torch

    grid = [round(6.0 + 0.05 * i, 2) for i in range(41)]
    H128 = torch.ones(1, 1, device="cuda")
    while H128.shape[0] < 128:
        H128 = torch.cat([torch.cat([H128, H128], 1), torch.cat([H128, -H128], 1)], 0)
    res = {}
    for wname in names:
        w = W.WORKLOADS[wname]
        q, k, v = W.generate(w, device="cuda")
        B, H, N = w.B, w.H, w.N
        BH = B * H
        out = {}
        for tname, x, rot in (("Q", q, True), ("K", k, True), ("V", v, False)):
            ref = x.float().reshape(BH, N, 128)
            if rot:
                ref = (ref @ H128) * (128 ** -0.5)
            mse = torch.empty(len(grid), BH, device="cuda")
            for gi, qm in enumerate(grid):
                if rot:
                    c, sc = mx.mxattn_quantize_qk_ex(x, rule=3, qmax=qm)
                    d = _dequant_qk(c, sc, BH, N)
                else:
                    c, sc = mx.mxattn_quantize_v_ex(x, rule=3, qmax=qm)
                    d = _dequant_v(c, sc, BH, N)
                mse[gi] = ((d - ref) ** 2).mean(dim=(1, 2))
                del c, sc, d
            best = [grid[i] for i in mse.argmin(0).tolist()]
            hist = {str(g): best.count(g) for g in sorted(set(best))}
            rel = (mse / mse[grid.index(7.25)]).mean(1).tolist()
            out[tname] = {"heads": BH, "argmin_counts": hist, "frac_at_7.25": best.count(7.25) / BH,
                          "mean_mse_rel_to_7.25": {str(g): rel[grid.index(g)] for g in (6.0, 6.5, 7.0, 7.2, 7.25, 7.3, 7.5, 8.0)}}
        res[wname] = out
        del q, k, v
        torch.cuda.empty_cache()
    return res


def rowsum_parts_gpu(mx, Pb, rule: int):
    """Section 5.5.2 row-sum diagnostic on the GPU: the bf16 rows ``Pb [R, npad]``
    (npad a multiple of 128, padding zero) quantized in 32-key blocks by the
    library's Q/K quantizer (rotation off) under ``rule``. Returns float64
    ``[R, 5]``: sum Q(P), then the zeroing, saturation (P / 2^e above 6, e the
    block's scale exponent from the quantizer), downward- and upward-rounding
    parts of sum(Q(P) - P)."""
    import torch

    R, npad = Pb.shape
    rows = R * npad // 128
    x = Pb.reshape(1, 1, rows, 128)
    c, sc = mx.mxattn_quantize_qk_ex(x, rule=rule, rotate=False)
    Qp = _dequant_qk(c, sc, 1, rows).reshape(R, npad).double()
    Pr = Pb.double()
    NT = (rows + 127) // 128
    e = (sc.view(1, NT, 512)[:, :, _atom_rows(sc.device)].reshape(1, NT * 128, 4)[:, :rows].long() - 127)
    e = e.repeat_interleave(32, -1).reshape(R, npad).double()
    d = Qp - Pr
    pos = Pr > 0
    zero = (Qp == 0) & pos
    sat = (Pr * torch.exp2(-e) > 6) & pos & ~zero
    down = (d < 0) & pos & ~zero & ~sat
    up = (d > 0) & pos
    return torch.stack([Qp.sum(1)] + [(d * m).sum(1) for m in (zero, sat, down, up)], 1)


def materialized_p(W, w, rows_per_workload: int, seed: int = 4321):
    """Softmax rows P = softmax(QK^T / sqrt(d)) (float64, exact S from the bf16
    Q and K; causal rows masked) for up to four sampled heads of `w`, and the
    same rows rounded to bf16 and zero-padded to a multiple of 128 keys."""
    import torch

    q, k, _ = W.generate(w, device="cuda")
    B, H, N = w.B, w.H, w.N
    g = torch.Generator().manual_seed(seed)
    heads = torch.randperm(B * H, generator=g)[: min(4, B * H)].tolist()
    per = max(1, rows_per_workload // len(heads))
    qf, kf = q.reshape(B * H, N, 128), k.reshape(B * H, N, 128)
    Ps = []
    for h in heads:
        ii = torch.randint(0, N, (per,), generator=g).cuda()
        s = (qf[h, ii].double() @ kf[h].double().T) / 128 ** 0.5
        if w.causal:
            s = s.masked_fill(torch.arange(N, device="cuda")[None, :] > ii[:, None], -float("inf"))
        Ps.append(torch.softmax(s, 1))
    P = torch.cat(Ps)
    npad = (N + 127) // 128 * 128
    Pb = torch.zeros((P.shape[0], npad), dtype=torch.bfloat16, device="cuda")
    Pb[:, :N] = P.to(torch.bfloat16)
    return P, Pb


def run_rowsum_diagnostic(mx, W, names, rows_per_workload=256):
    """Section 5.5.2 on synthetic heads: materialize P = softmax(S) for sampled rows
    (exact S from the bf16 Q, K), round it to bf16, quantize it in 32-key MXFP4
    blocks with the library's quantizer (rotation off), and report the mean row sum
    of the quantized P, the row-sum error split into zeroing, saturation, downward
    and upward rounding, and the row sums by attention entropy."""
    import torch

    out = {}
    for wname in names:
        w = W.WORKLOADS[wname]
        P, Pb = materialized_p(W, w, rows_per_workload)
        R = P.shape[0]
        ent = -(P * torch.log(P.clamp_min(1e-300))).sum(1)
        res = {}
        for rname, rule in (("UOS", 0), ("OCP", 1)):
            parts = rowsum_parts_gpu(mx, Pb, rule)
            rs = parts[:, 0]
            bins = {}
            for lo, hi in ((0, 1), (1, 3), (3, 5), (5, 1e9)):
                m = (ent >= lo) & (ent < hi)
                if m.any():
                    bins[f"entropy [{lo}, {hi if hi < 1e9 else 'inf'})"] = {
                        "rows": int(m.sum()), "mean_rowsum": rs[m].mean().item(),
                        "frac_below_1": (rs[m] < 1).double().mean().item()}
            res[rname] = {"mean_rowsum": rs.mean().item(), "min_rowsum": rs.min().item(),
                          "max_rowsum": rs.max().item(),
                          "error_parts": {name: parts[:, i + 1].mean().item() for i, name in
                                          enumerate(("zeroing", "saturation", "rounding_down", "rounding_up"))},
                          "by_entropy": bins}
        out[wname] = {"rows": R, "mean_entropy": ent.mean().item(), "results": res}
        del P, Pb
        torch.cuda.empty_cache()
    return out


def run_accuracy(args):
    """Accuracy of the ablation variants and the BF16 path against exact
    softmax attention (Eq. 1, float64 on the host) on sampled rows of every
    workload, plus the mean row sum of the normalized attention under direct
    placement (V = 1 makes the output the row sum). Prints one JSON line."""
    import torch

    import mxfp4_precision_attention_gb300 as mx
    from mxfp4_precision_attention_gb300 import workloads as W

    mx.load()
    names = args.accuracy_workloads.split(",") if args.accuracy_workloads else list(W.WORKLOADS)
    table = {}
    for wname in names:
        w = W.WORKLOADS[wname]
        q, k, v = W.generate(w, device="cuda")
        B, H, N = w.B, w.H, w.N
        g = torch.Generator().manual_seed(1234)
        heads = torch.randperm(B * H, generator=g)[: min(4, B * H)].tolist()
        per_head = max(1, args.accuracy_rows // len(heads))
        rows = [(h, int(i)) for h in heads for i in torch.randint(0, N, (per_head,), generator=g)]
        qf, kf, vf = (t.reshape(B * H, N, 128) for t in (q, k, v))
        ref = []
        for h, i in rows:  # exact attention for the sampled rows (float64, host)
            kk = kf[h].double().cpu()
            s = (qf[h, i].double().cpu() @ kk.T) / 128 ** 0.5
            if w.causal:
                s[i + 1:] = -float("inf")
            ref.append(torch.softmax(s, 0) @ vf[h].double().cpu())
        ref = torch.stack(ref)
        hh = torch.tensor([r[0] for r in rows])
        ii = torch.tensor([r[1] for r in rows])

        def score(out):
            o = out.reshape(B * H, N, 128)[hh.to(out.device), ii.to(out.device)].double().cpu()
            cos = torch.nn.functional.cosine_similarity(o, ref, dim=1).mean().item()
            rel = ((o - ref).norm() / ref.norm()).item()
            return {"cosine": cos, "rel_l2": rel, "max_abs": (o - ref).abs().max().item()}

        res = {}
        for name, rule, rotate, placement in ABLATION:
            qc, qs = mx.mxattn_quantize_qk_ex(q, rule=rule, rotate=rotate)
            kc, ks = mx.mxattn_quantize_qk_ex(k, rule=rule, rotate=rotate)
            vc, vs = mx.mxattn_quantize_v_ex(v, rule=rule)
            out = mx.mxattn_forward_ex(qc, qs, kc, ks, vc, vs, v, B, H, N, causal=w.causal, p_rule=rule,
                                       placement=placement)
            mx.mxattn_check()
            res[name] = score(out)
            if placement == 1:
                ones = torch.ones_like(v)
                oc, os_ = mx.mxattn_quantize_v_ex(ones, rule=rule)
                rs = mx.mxattn_forward_ex(qc, qs, kc, ks, oc, os_, ones, B, H, N, causal=w.causal, p_rule=rule,
                                          placement=placement)[..., 0]
                res[name]["rowsum_mean"] = rs.mean().item()
                res[name]["rowsum_min"] = rs.min().item()
        # the NVFP4 baseline (section 5.2: direct l) and NVFP4 with PNQ
        qt, kt, vt = mx.mxattn_nvfp4_quantize_qk(q), mx.mxattn_nvfp4_quantize_qk(k), mx.mxattn_nvfp4_quantize_v(v)
        for label, placement in (("NVFP4 (direct l, the baseline)", 1), ("NVFP4 + PNQ", 0)):
            out = mx.mxattn_nvfp4_forward(qt, kt, vt, v, B, H, N, causal=w.causal, placement=placement)
            mx.mxattn_check()
            res[label] = score(out)
            if placement == 1:
                ones = torch.ones_like(v)
                ot = mx.mxattn_nvfp4_quantize_v(ones)
                rs = mx.mxattn_nvfp4_forward(qt, kt, ot, ones, B, H, N, causal=w.causal, placement=1)[..., 0]
                res[label]["rowsum_mean"] = rs.mean().item()
                res[label]["rowsum_min"] = rs.min().item()
        del qt, kt, vt
        res["bf16 path"] = score(mx.mxattn_forward_bf16(q, k, v, causal=w.causal))
        mx.mxattn_check()
        table[wname] = {"rows": len(rows), "results": res}
        del q, k, v
        torch.cuda.empty_cache()
    sweep = run_qmax_sweep(mx, W, [n for n in ("lognormal_4096", "wan_32760", "hunyuan_118800") if n in names])
    rowsum = run_rowsum_diagnostic(mx, W, names)
    print(json.dumps({"accuracy": table, "qmax_sweep": sweep, "rowsum_diagnostic": rowsum,
                      "reference": "exact softmax attention (Eq. 1), float64 on the host",
                      "data": "synthetic"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="wan_32760")
    ap.add_argument("--heads", type=int, default=None, help="override H (smaller profiling cases)")
    ap.add_argument("--n", type=int, default=None, help="override N (smaller profiling cases)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-bf16", action="store_true", help="skip the BF16 comparison-path timing")
    ap.add_argument("--no-nvfp4", action="store_true", help="skip the NVFP4 comparison-path timing")
    ap.add_argument("--no-mma-probe", action="store_true", help="skip the dense FP4 MMA rate probe")
    ap.add_argument("--mma-probe-s", type=float, default=1.0, help="seconds of back-to-back MMAs in the probe")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-per-workload", action="store_true", help="skip the other workloads' lines")
    ap.add_argument("--per-workload-cpu-s", type=float, default=6.0, help="oracle seconds per other workload")
    ap.add_argument("--ref-step-s", type=float, default=8.0)
    ap.add_argument("--accuracy", action="store_true",
                    help="accuracy of the ablation variants vs exact attention instead of timing")
    ap.add_argument("--accuracy-workloads", default=None, help="comma-separated workload names (default: all)")
    ap.add_argument("--accuracy-rows", type=int, default=256, help="sampled query rows per workload")
    args = ap.parse_args()
    if args.accuracy:
        run_accuracy(args)
        return
    from mxfp4_precision_attention_gb300 import workloads as W

    w = W.WORKLOADS[args.workload]
    if args.heads is not None or args.n is not None:
        import dataclasses

        w = dataclasses.replace(w, H=args.heads or w.H, N=args.n or w.N,
                                name=f"{w.name}[H={args.heads or w.H},N={args.n or w.N}]")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
