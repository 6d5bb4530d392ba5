"""Benchmark of the CPR Gated DeltaNet layer on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one CPR prefill / training forward of the trainer-shaped workload (1 sequence
x 10,240 tokens, H=16, dk=dv=128, C=64, bf16 q/k/v, fp32 state), inputs resident in HBM,
L2 flushed between steps.  The JSON line also carries, each with its own rate and
roofline:
  - decode: the rollout-decode workload (256 sequences x 1 token, prior lengths
    U[1,4096], steps/s);
  - continuation: the rollout prefill resumed at seeded positions;
  - rollout_prefill: the 5 x 2,048 packed rollout prefill in one call;
  - varlen_stress: 32 packed sequences of log-uniform lengths (H=32), prefill and then
    128 decode steps;
  - tiny: the fp32 case's prefill and decode-step latency;
  - train_fwd_bwd: the trainer's forward and backward (cpr_gdn_backward) at 1 x 10,240;
  - pik: the deterministic K-split product (one GPU only);
  - fp32_peak_probe: the FP32-pipe peak measured on this GPU by the committed probe;
plus the end-to-end number through the C ABI with host buffers, and the fp64 CPU oracle
timed on this machine's cores.  Under torchrun every rank runs the same workload on its
own GPU (independent problems: weak scaling, no collective on the data path); rank 0
prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CPR-GDN prefill tokens/s, decode steps/s per layer; % of roofline; 1 GB300"
# FP32 pipe: 152 SMs x 128 FP32 lanes x 2 flop (FMA) x 2.07 GHz (maximum SM clock)
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
L2_BYTES = 129 * 1024 * 1024
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture
# of the kernel as it now stands: k23_chain_and_intra at trainer_fwd, k4_decode_step at
# rollout_decode, kb23_chain_and_grads_tc at the trainer's forward + backward.  Reset to
# None whenever the kernel changes.
TRAFFIC_K23_TRAINER_FWD = 531.102976e6 + 194.182912e6
TRAFFIC_K4_ROLLOUT_DECODE = 267.595520e6 + 208.146688e6
TRAFFIC_KB23_TRAINER = 834.262528e6 + 391.001600e6


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = str(gpu_index)
        try:  # nvidia-smi numbering can differ from CUDA's: select the GPU by UUID
            u = str(torch.cuda.get_device_properties(gpu_index).uuid)
            self.gpu = u if u.startswith("GPU-") else f"GPU-{u}"
        except Exception:
            pass
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
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

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------------------------
# algorithmic work (per the method, independent of the kernels' own bookkeeping)
# ------------------------------------------------------------------------------------

def prefill_algorithmic(T, N, H, dk, dv, n_chunks, elem=2):
    """Bytes and FP32 flops of one prefill: q,k,v read, o written, g,beta read, every
    boundary state written, final states written; 7*dk*dv flops per token-head (S k: 2,
    alpha S + u k^T: 3, S q: 2)."""
    bytes_ = T * H * (2 * dk + dv) * elem + T * H * dv * elem + 2 * T * H * 4
    bytes_ += n_chunks * H * dk * dv * 4 + N * H * dk * dv * 4
    flops_intra = 7 * dk * dv * T * H
    return bytes_, flops_intra


def decode_algorithmic(B, H, dk, dv, C, n_resync, elem=2):
    """Bytes of one decode step: state read + write, token q,k,v,g,beta read, o written,
    the token's ring slot written; per resync: the ring chunk and S_b read, S_b and the
    state written."""
    per = 2 * dk * dv * 4 + (2 * dk + dv) * elem + 8 + dv * elem + (dk + dv) * elem + 8
    res = C * (dk + dv) * elem + 8 * C + dk * dv * 4 + 2 * dk * dv * 4
    return B * H * per + n_resync * H * res


# ------------------------------------------------------------------------------------

def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def _max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(dist):
    if dist is not None:
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def weak_scaling_rate(world: int, units_per_rank: float, ms_max: float) -> float:
    """Whole-job rate: every rank processed units_per_rank; the job took the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


def cpu_baseline_oracle(x_cpu, C, target_s=12.0):
    """The fp64 oracle as it stands, on this host's cores, over whole copies of the
    workload until about target_s seconds have run.  Returns (tokens/s, threads, sample)."""
    import numpy as np

    import oracle

    arrs = [np.ascontiguousarray(x_cpu[k].double().numpy()) for k in ("q", "k", "v", "g", "beta")]
    cu = x_cpu["cu_seqlens"].numpy()
    T = int(cu[-1])
    reps, t_total = 0, 0.0
    while t_total < target_s and reps < 50:
        t0 = time.perf_counter()
        oracle.recurrent(*arrs, cu, C, boundaries=True)
        t_total += time.perf_counter() - t0
        reps += 1
    return T * reps / t_total, oracle.max_threads(), f"{reps} full run(s) of the {T}-token workload"


def run_reference(args):
    """--impl reference: the fp64 CPU oracle on the same workload, metric and unit."""
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:  # the CPU oracle runs once, on rank 0; other ranks exit without work
        return
    import numpy as np

    import oracle
    from linear_attention_cpr_gb300 import inputs

    w = inputs.workload("trainer_fwd")
    x = inputs.prefill_inputs(w)
    arrs = [np.ascontiguousarray(x[k].double().numpy()) for k in ("q", "k", "v", "g", "beta")]
    T_s = 2048  # one step = the first 2,048 tokens of the sequence, all 16 heads
    sub = [a[:T_s] for a in arrs]
    for _ in range(args.warmup):
        oracle.recurrent(*sub, [0, T_s], w.C)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.recurrent(*sub, [0, T_s], w.C)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = T_s / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "trainer_fwd: 1 x 10,240 tokens, H=16, dk=dv=128, C=64",
                       "sample": f"first {T_s} tokens x 16 heads per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"first {T_s} tokens of the 10,240-token sequence, 16 heads, per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_fp32_peak(dev):
    """FP32-pipe peak of this GPU from the committed probe (csrc/probe_peaks.cu): scalar
    FFMA and paired f32x2 FMA over every SM, the larger of the two, in TFLOP/s."""
    import ctypes

    from linear_attention_cpr_gb300 import build

    lib = ctypes.CDLL(build.PROBE_LIB)
    lib.cpr_probe_fp32.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, threads, iters = sms * 8, 256, 20000
    sink = torch.empty(blocks * threads, dtype=torch.float32, device=dev)
    ms = ctypes.c_float(0.0)
    best = {}
    for paired in (0, 1):
        vals = []
        for _ in range(4):
            rc = lib.cpr_probe_fp32(paired, blocks, threads, iters, ctypes.c_void_p(sink.data_ptr()),
                                    ctypes.byref(ms), None)
            if rc != 0:
                return None
            vals.append(ms.value)
        flops = blocks * threads * iters * 16 * 2 * (2 if paired else 1)
        best["ffma2" if paired else "ffma"] = flops / (min(vals[1:]) * 1e-3) / 1e12
    return {"tflops": max(best.values()), "ffma": best["ffma"], "ffma2": best["ffma2"],
            "how": f"{blocks} CTAs x {threads} threads x {iters} rounds of 16 independent FMA chains"}


def time_prefill(cpr, w, x, dev, steps, warmup, dist, flush, p32_meas=None):
    """Time one workload's prefill through the C ABI (inputs resident, L2 flushed between
    steps outside the events) with the per-kernel events of the profiling hook.  Returns
    the line's fields: ms per step, kernel times, tokens/s, roofline of k23 (FP32 bound)."""
    T, H, dk, dv, C, N = w.total_tokens, w.H, w.dk, w.dv, w.C, len(w.seqlens)
    n_chunks = cpr.cpr_gdn_num_chunks(x["cu_seqlens"].cpu(), C)
    out = torch.empty(T, H, dv, dtype=w.dtype, device=dev)
    st = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    bnd = torch.empty(max(n_chunks, 1), H, dk, dv, dtype=torch.float32, device=dev)
    ws = torch.empty(cpr.cpr_gdn_prefill_workspace_size(T, N, H, dk, dv, C), dtype=torch.uint8, device=dev)

    def prefill():
        cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, out=out, state_out=st,
                            boundary_states=bnd, workspace=ws)

    for _ in range(warmup):
        prefill()
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    kern = {"chunk_index": [], "chunk_prep": [], "chain_and_intra": []}
    step_ms = []
    _barrier(dist)
    cpr.cpr_gdn_set_profile_events(ev)
    for _ in range(steps):
        flush.zero_()
        prefill()
        ev[3].synchronize()
        step_ms.append(ev[0].elapsed_time(ev[3]))
        for i, name in enumerate(kern):
            kern[name].append(ev[i].elapsed_time(ev[i + 1]))
    cpr.cpr_gdn_set_profile_events(None)
    _barrier(dist)
    ms_max = _max_over_ranks(dist, statistics.fmean(step_ms))
    kern_ms = {k: statistics.fmean(v) for k, v in kern.items()}
    alg_bytes, flops = prefill_algorithmic(T, N, H, dk, dv, n_chunks, elem=2 if w.dtype == torch.bfloat16 else 4)
    achieved = flops / (kern_ms["chain_and_intra"] / 1e3) / 1e12
    roof = {"kernel": "k23_chain_and_intra", "bound": "alu", "achieved": achieved, "peak": FP32_PEAK_TFLOPS,
            "unit": "TFLOP/s", "frac": achieved / FP32_PEAK_TFLOPS, "traffic": None,
            "peak_kind": "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz", "flops_per_launch": flops}
    if p32_meas:
        roof["peak_measured"] = p32_meas["tflops"]
        roof["frac_of_measured"] = achieved / p32_meas["tflops"]
    hbm_peak, _ = _peaks()
    t_roof_ms = max(alg_bytes / (hbm_peak * 1e9), flops / (FP32_PEAK_TFLOPS * 1e12)) * 1e3
    return {"ms_per_step": ms_max, "value": weak_scaling_rate(dist.get_world_size() if dist else 1, T, ms_max),
            "unit": "tokens/s", "steps": steps, "kernels_ms": kern_ms, "algorithmic_bytes": alg_bytes,
            "t_roof_ms": t_roof_ms, "frac_of_t_roof": t_roof_ms / ms_max, "roofline": roof, "n_chunks": n_chunks,
            "gpu_launches": 3 * steps}


def time_decode_steps(cpr, w, state, ring, pos0, dev, steps, warmup, dist, flush, hbm_peak):
    """Time `steps` decode steps of a workload's sequences from a prefilled state and ring,
    one step per timed region (events of the profiling hook), L2 flushed between steps when
    the resident state is smaller than L2.  Returns the line's fields."""
    B, H, dk, dv, C = len(w.seqlens), w.H, w.dk, w.dv, w.C
    toks = [inputs_decode(w, s, dev) for s in range(min(steps, 64))]
    pos = pos0.clone().to(dev)
    out = torch.empty(B, H, dv, dtype=w.dtype, device=dev)
    dws = torch.empty(cpr.cpr_gdn_decode_workspace_size(B, H, dk, dv, C), dtype=torch.uint8, device=dev)
    small = B * H * dk * dv * 4 < L2_BYTES

    def step(s):
        t = toks[s % len(toks)]
        cpr.cpr_gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], state, ring, pos, C, out=out, workspace=dws)
        pos.add_(1)

    for s in range(warmup):
        step(s)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    step_ms, k4 = [], []
    n_res = 0
    pos_host = pos0.clone().cpu() + warmup
    _barrier(dist)
    cpr.cpr_gdn_set_profile_events(ev)
    for s in range(warmup, warmup + steps):
        n_res += int(((pos_host % C) == C - 1).sum())
        pos_host += 1
        if small:
            flush.zero_()
        step(s)
        ev[2].synchronize()
        step_ms.append(ev[0].elapsed_time(ev[2]))
        k4.append(ev[0].elapsed_time(ev[1]))
    cpr.cpr_gdn_set_profile_events(None)
    _barrier(dist)
    assert cpr.cpr_gdn_device_status(dws) == 0
    ms = _max_over_ranks(dist, statistics.fmean(step_ms))
    k4_ms = statistics.fmean(k4)
    bytes_step = decode_algorithmic(B, H, dk, dv, C, n_res / steps, elem=2 if w.dtype == torch.bfloat16 else 4)
    step_only = decode_algorithmic(B, H, dk, dv, C, 0, elem=2 if w.dtype == torch.bfloat16 else 4)
    ach = step_only / (k4_ms / 1e3) / 1e9
    world = dist.get_world_size() if dist else 1
    return {"metric": "decode steps/s per layer", "value": 1e3 / ms * world, "unit": "steps/s", "ms_per_step": ms,
            "steps": steps, "kernels_ms": {"step_with_concurrent_resync": k4_ms},
            "resyncs_per_step": n_res / steps, "l2": "flushed between steps" if small else "state larger than L2",
            "roofline": {"kernel": "k4_decode_step", "bound": "hbm", "achieved": ach, "peak": hbm_peak,
                         "unit": "GB/s", "frac": ach / hbm_peak, "traffic": None, "bytes_per_launch": step_only},
            "t_roof_ms": bytes_step / (hbm_peak * 1e9) * 1e3,
            "frac_of_t_roof": bytes_step / (hbm_peak * 1e9) * 1e3 / ms, "gpu_launches": 2 * steps}


def inputs_decode(w, s, dev):
    from linear_attention_cpr_gb300 import inputs

    return inputs.decode_inputs(w, s, device=dev)


def backward_algorithmic(n_chunks, H, dk, dv, C):
    """FP32-equivalent flops of one backward as its kernels evaluate it, per (chunk, head) with
    n = C tokens (multiply-adds x 2):
      chunk maps: K K^T, Q K^T, W, Qt (4 n^2 d), M^T and C_b (2 n d^2), T (n^3 / 6);
      reverse chain: dS M^T (dk^2 dv);
      chunk gradients: 10 products of n^2 d (K K^T, Q K^T, U, dPm, Pm^T dO, dQK K, dQK^T Q,
      dT, T^T dU, (dKK + dKK^T) K), 5 of n d^2 (K S_b^T, dO S_b, diag(d) K dS^T, U dS,
      T^T dU S_b), 2 of n^3 (T^T dT, X T^T) and T (n^3 / 6)."""
    d = dk
    maps = 4 * C * C * d + 2 * C * d * d + C ** 3 // 6
    chain = dk * dk * dv
    grads = 10 * C * C * d + 5 * C * d * d + 2 * C ** 3 + C ** 3 // 6
    return {"chunk_maps": 2 * maps * n_chunks * H, "reverse_chain": 2 * chain * n_chunks * H,
            "chunk_grads": 2 * grads * n_chunks * H}


def run_train_fwd_bwd(args, cpr, inputs, dev, dist, world, flush, p32_meas):
    """Trainer forward + backward at 1 x 10,240 tokens (H=16, d=128, C=64): cpr_gdn_prefill
    then cpr_gdn_backward on the same batch (the forward's boundary states are the saved
    states), upstream gradients dL/do seeded, L2 flushed between steps."""
    w = inputs.workload("trainer_fwd")
    xc = inputs.prefill_inputs(w)
    x = {k: v.to(dev) for k, v in xc.items()}
    T, H, dk, dv, C, N = w.total_tokens, w.H, w.dk, w.dv, w.C, len(w.seqlens)
    n_chunks = cpr.cpr_gdn_num_chunks(xc["cu_seqlens"], C)
    gen = torch.Generator().manual_seed(7)
    d_out = torch.randn(T, H, dv, generator=gen).to(w.dtype).to(dev)
    out = torch.empty(T, H, dv, dtype=w.dtype, device=dev)
    st = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    bnd = torch.empty(n_chunks, H, dk, dv, dtype=torch.float32, device=dev)
    ws = torch.empty(cpr.cpr_gdn_prefill_workspace_size(T, N, H, dk, dv, C), dtype=torch.uint8, device=dev)
    bws = torch.empty(cpr.cpr_gdn_backward_workspace_size(T, N, H, dk, dv, C), dtype=torch.uint8, device=dev)
    grads = {"dq": torch.empty(T, H, dk, device=dev), "dk": torch.empty(T, H, dk, device=dev),
             "dv": torch.empty(T, H, dv, device=dev), "dg": torch.empty(T, H, device=dev),
             "dbeta": torch.empty(T, H, device=dev), "d_state_in": torch.empty(N, H, dk, dv, device=dev)}

    def fwd():
        cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, out=out, state_out=st,
                            boundary_states=bnd, workspace=ws)

    def bwd():
        cpr.cpr_gdn_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, bnd, d_out,
                             grads=grads, workspace=bws)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0 and cpr.cpr_gdn_device_status(bws) == 0
    steps = max(3, min(args.steps, 30))
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    # the backward's events: k0 | chunk maps | (chain) | chain and gradients; at this shape the
    # reverse chain and the chunk gradients are one launch, so they are timed together
    total, fwd_ms, kern = [], [], {"chunk_maps": [], "chain_and_grads": []}
    _barrier(dist)
    for _ in range(steps):
        flush.zero_()
        e[0].record()
        fwd()
        e[1].record()
        cpr.cpr_gdn_set_profile_events(ev)
        bwd()
        cpr.cpr_gdn_set_profile_events(None)
        ev[4].synchronize()
        total.append(e[0].elapsed_time(ev[4]))
        fwd_ms.append(e[0].elapsed_time(e[1]))
        kern["chunk_maps"].append(ev[1].elapsed_time(ev[2]))
        kern["chain_and_grads"].append(ev[2].elapsed_time(ev[4]))
    _barrier(dist)
    ms = _max_over_ranks(dist, statistics.fmean(total))
    kern_ms = {k: statistics.fmean(v) for k, v in kern.items()}
    flops = backward_algorithmic(n_chunks, H, dk, dv, C)
    _, f_fwd = prefill_algorithmic(T, N, H, dk, dv, n_chunks)
    f_cg = flops["reverse_chain"] + flops["chunk_grads"]
    ach = f_cg / (kern_ms["chain_and_grads"] / 1e3) / 1e12
    roof = {"kernel": "kb23_chain_and_grads_tc", "bound": "alu", "achieved": ach, "peak": FP32_PEAK_TFLOPS,
            "unit": "TFLOP/s", "frac": ach / FP32_PEAK_TFLOPS, "traffic": TRAFFIC_KB23_TRAINER,
            "flops_per_launch": f_cg,
            "peak_kind": "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz; FP32-equivalent work (the kernels "
                         "run the products as bf16 hi/lo splits on the tensor cores)"}
    if p32_meas:
        roof["peak_measured"] = p32_meas["tflops"]
        roof["frac_of_measured"] = ach / p32_meas["tflops"]
    t_roof = (f_fwd + sum(flops.values())) / (FP32_PEAK_TFLOPS * 1e12) * 1e3
    line = {"metric": "trainer forward + backward tokens/s per layer", "value": weak_scaling_rate(world, T, ms),
            "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "workload": f"trainer_fwd + backward: 1 x {T} tokens, H={H}, dk=dv={dk}, C={C}, bf16 q/k/v/dO, "
                        "fp32 gradients",
            "forward_ms": statistics.fmean(fwd_ms), "backward_kernels_ms": kern_ms,
            "backward_flops": flops, "t_roof_ms": t_roof, "frac_of_t_roof": t_roof / ms, "roofline": roof,
            "gpu_launches": 6 * steps}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = backward_cpu_baseline(xc, d_out.cpu(), C)
    return line


def backward_cpu_baseline(xc, d_out, C, heads=2):
    """The oracle's forward (C, host threads) and WY-chunked adjoint (fp64, numpy) on the
    first `heads` heads of the trainer sequence; tokens/s of forward + backward scaled to
    all heads."""
    import numpy as np

    import oracle
    from oracle import backward

    H = xc["q"].shape[1]
    sub = {k: np.ascontiguousarray(xc[k][:, :heads].double().numpy()) for k in ("q", "k", "v", "g", "beta")}
    cu = xc["cu_seqlens"].numpy()
    t0 = time.perf_counter()
    oracle.recurrent(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], cu, C, boundaries=True)
    backward.wy_chunked_backward(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], cu,
                                 d_out[:, :heads].double().numpy(), C)
    sec = time.perf_counter() - t0
    T = int(cu[-1])
    return {"value": T * heads / H / sec, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"forward + backward of heads 0..{heads - 1} of the {T}-token sequence ({sec:.1f} s), "
                      f"scaled to {H} heads"}


def run_extra_workloads(args, cpr, inputs, dev, dist, world, flush, p32_meas, hbm_peak):
    """The other configurations of the layer, each with its own line: the one-shot rollout
    prefill (5 x 2,048 packed), the varlen stress batch (prefill, then 128 decode steps) and
    the tiny fp32 case (latency in microseconds)."""
    res = {}
    steps = max(3, min(args.steps, 50))
    # rollout prefill: the five sequences in one packed call
    w = inputs.workload("rollout_prefill")
    xc = inputs.prefill_inputs(w)
    x = {k: v.to(dev) for k, v in xc.items()}
    line = time_prefill(cpr, w, x, dev, steps, args.warmup, dist, flush, p32_meas)
    line.update({"metric": "rollout prefill tokens/s per layer",
                 "workload": f"rollout_prefill: 5 x 2,048 tokens packed in one call, H={w.H}, dk=dv={w.dk}, "
                             f"C={w.C}, bf16 q/k/v"})
    if world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample = cpu_baseline_oracle(xc, w.C, target_s=5.0)
        line["cpu_baseline"] = {"value": v_cpu, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    res["rollout_prefill"] = line
    del x
    # varlen stress: prefill of the packed batch, then decode steps of every sequence
    w = inputs.workload("varlen_stress")
    xc = inputs.prefill_inputs(w)
    x = {k: v.to(dev) for k, v in xc.items()}
    line = time_prefill(cpr, w, x, dev, steps, args.warmup, dist, flush, p32_meas)
    line.update({"metric": "varlen prefill tokens/s per layer",
                 "workload": f"varlen_stress: {len(w.seqlens)} sequences, log-uniform lengths in [64, 8192], "
                             f"{w.total_tokens} tokens, H={w.H}, dk=dv={w.dk}, C={w.C}, bf16 q/k/v"})
    if world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample = cpu_baseline_oracle(xc, w.C, target_s=3.0)
        line["cpu_baseline"] = {"value": v_cpu, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    _, st, bnd, _ = cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], w.C)
    ring = cpr.cpr_gdn_ring_from_prefill(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], w.C, bnd, st)
    pos0 = torch.tensor(w.seqlens, dtype=torch.int32)
    dec = time_decode_steps(cpr, w, st, ring, pos0, dev, w.decode_steps, args.warmup, dist, flush, hbm_peak)
    dec["workload"] = (f"varlen_stress decode: {len(w.seqlens)} sequences x 1 token after the prefill, H={w.H}, "
                       f"dk=dv={w.dk}, C={w.C}, {w.decode_steps} steps")
    line["decode"] = dec
    res["varlen_stress"] = line
    del x, st, bnd, ring
    # tiny fp32: latency of one prefill and of one decode step
    w = inputs.workload("tiny")
    xc = inputs.prefill_inputs(w)
    x = {k: v.to(dev) for k, v in xc.items()}
    line = time_prefill(cpr, w, x, dev, steps, args.warmup, dist, flush, p32_meas)
    pre = {k: v[:w.total_tokens - 1] for k, v in x.items() if k != "cu_seqlens"}
    cu_pre = inputs.cu_seqlens_of([w.total_tokens - 1]).to(dev)
    _, st, bnd, _ = cpr.cpr_gdn_prefill(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], cu_pre, w.C)
    ring = cpr.cpr_gdn_ring_from_prefill(pre["k"], pre["v"], pre["g"], pre["beta"], cu_pre, w.C, bnd, st)
    dec = time_decode_steps(cpr, w, st, ring, torch.tensor([w.total_tokens - 1], dtype=torch.int32), dev, steps,
                            args.warmup, dist, flush, hbm_peak)
    res["tiny"] = {"metric": "tiny fp32 latency per layer", "workload": "tiny: 1 x 256 tokens, H=2, dk=dv=32, "
                   "C=16, fp32 q/k/v (latency-bound: no roofline fraction)",
                   "prefill_us": 1e3 * line["ms_per_step"], "prefill_kernels_us":
                   {k: 1e3 * v for k, v in line["kernels_ms"].items()},
                   "decode_step_us": 1e3 * dec["ms_per_step"], "steps": steps,
                   "gpu_launches": line["gpu_launches"] + dec["gpu_launches"]}
    return res



def run_ours(args):
    import linear_attention_cpr_gb300 as cpr
    from linear_attention_cpr_gb300 import build, inputs

    dist, rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    cpr.load_library()
    hbm_peak, hbm_kind = _peaks()
    gen_dev = torch.Generator(device=dev)
    if args.only_pik:  # the deterministic K-split product alone (profiling and quick checks)
        if world > 1:
            raise SystemExit("--only-pik runs on one GPU only")
        line = run_pik(args, cpr, inputs, dev, dist, world)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    # ---------------- prefill: trainer-forward shape ----------------
    w = inputs.workload(args.workload)
    x_cpu = inputs.prefill_inputs(w)
    x = {k: v.to(dev) for k, v in x_cpu.items()}
    T, H, dk, dv, C, N = w.total_tokens, w.H, w.dk, w.dv, w.C, len(w.seqlens)
    n_chunks = cpr.cpr_gdn_num_chunks(x_cpu["cu_seqlens"], C)
    out = torch.empty(T, H, dv, dtype=w.dtype, device=dev)
    st = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    bnd = torch.empty(n_chunks, H, dk, dv, dtype=torch.float32, device=dev)
    ws = torch.empty(cpr.cpr_gdn_prefill_workspace_size(T, N, H, dk, dv, C), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def prefill():
        cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, out=out, state_out=st,
                            boundary_states=bnd, workspace=ws)

    for _ in range(args.warmup):
        prefill()
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    kern = {"chunk_index": [], "chunk_prep": [], "chain_and_intra": []}
    step_ms = []
    _barrier(dist)
    with ClockSampler(local) as clocks:
        cpr.cpr_gdn_set_profile_events(ev)
        for _ in range(args.steps):
            flush.zero_()  # L2 flush between steps (outside the events)
            prefill()
            ev[3].synchronize()
            step_ms.append(ev[0].elapsed_time(ev[3]))
            for i, name in enumerate(kern):
                kern[name].append(ev[i].elapsed_time(ev[i + 1]))
        cpr.cpr_gdn_set_profile_events(None)
        _barrier(dist)
    ms = statistics.fmean(step_ms)
    ms_max = _max_over_ranks(dist, ms)
    value = weak_scaling_rate(world, T, ms_max)
    kern_ms = {k: statistics.fmean(v) for k, v in kern.items()}
    alg_bytes, flops_intra = prefill_algorithmic(T, N, H, dk, dv, n_chunks)
    intra_ms = kern_ms["chain_and_intra"]
    achieved = flops_intra / (intra_ms / 1e3) / 1e12
    roofline = {"kernel": "k23_chain_and_intra", "bound": "alu", "achieved": achieved, "peak": FP32_PEAK_TFLOPS,
                "unit": "TFLOP/s", "frac": achieved / FP32_PEAK_TFLOPS,
                "traffic": TRAFFIC_K23_TRAINER_FWD if w.name == "trainer_fwd" else None,
                "peak_kind": "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz",
                "flops_per_launch": flops_intra}
    t_roof_ms = max(alg_bytes / (hbm_peak * 1e9), flops_intra / (FP32_PEAK_TFLOPS * 1e12)) * 1e3

    # ---------------- end to end through the C ABI with host buffers ----------------
    pin = {k: v.pin_memory() for k, v in x_cpu.items()}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    st_h = torch.empty(st.shape, dtype=st.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = out_h.numel() * out_h.element_size() + st_h.numel() * st_h.element_size()
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for it in range(args.warmup + args.steps):
        flush.zero_()
        e_a.record()
        for k in x:
            x[k].copy_(pin[k], non_blocking=True)
        prefill()
        out_h.copy_(out, non_blocking=True)
        st_h.copy_(st, non_blocking=True)
        e_b.record()
        e_b.synchronize()
        if it >= args.warmup:
            e2e_ms.append(e_a.elapsed_time(e_b))
    e2e_val = weak_scaling_rate(world, T, _max_over_ranks(dist, statistics.fmean(e2e_ms)))

    # ---------------- decode: rollout shape ----------------
    decode = None
    if not args.no_decode and not args.no_rollout_decode:
        decode = run_decode(args, cpr, inputs, dev, hbm_peak, dist, world)
    continuation = run_continuation(args, cpr, inputs, dev, hbm_peak, dist, world) if not args.no_decode else None
    # the K-split product is a one-GPU leg: under torchrun it is left out on every rank
    pik_line = run_pik(args, cpr, inputs, dev, dist, world) if not args.no_pik and world == 1 else None

    p32_meas = measure_fp32_peak(dev)
    if p32_meas:
        roofline["peak_measured"] = p32_meas["tflops"]
        roofline["frac_of_measured"] = roofline["achieved"] / p32_meas["tflops"]
    extra = None if args.no_extra else run_extra_workloads(args, cpr, inputs, dev, dist, world, flush, p32_meas,
                                                           hbm_peak)
    train = None if args.no_train else run_train_fwd_bwd(args, cpr, inputs, dev, dist, world, flush, p32_meas)

    # ---------------- CPU oracle baseline (rank 0, N = 1 only) ----------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample = cpu_baseline_oracle(x_cpu, C)
        cpu = {"value": v_cpu, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}

    launches = 3 * args.steps
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{w.name}: {N} x {T} tokens, H={H}, dk=dv={dk}, C={C}, bf16 q/k/v, fp32 state",
                       "l2": "flushed between timed steps (2 x L2 buffer written)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roofline,
            "prefill": {"kernels_ms": kern_ms, "algorithmic_bytes": alg_bytes, "t_roof_ms": t_roof_ms,
                        "frac_of_t_roof": t_roof_ms / ms_max, "hbm_peak_gbs": hbm_peak, "hbm_peak_kind": hbm_kind},
            "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches + (decode["gpu_launches"] if decode else 0) +
                            (continuation["gpu_launches"] if continuation else 0) +
                            (pik_line["gpu_launches"] if pik_line else 0) +
                            (sum(v["gpu_launches"] + (v.get("decode") or {}).get("gpu_launches", 0)
                                 for v in extra.values()) if extra else 0) +
                            (train["gpu_launches"] if train else 0),
            "clocks": clocks.summary(),
            "decode": decode,
            "continuation": continuation,
            "pik": pik_line,
            "rollout_prefill": extra["rollout_prefill"] if extra else None,
            "varlen_stress": extra["varlen_stress"] if extra else None,
            "tiny": extra["tiny"] if extra else None,
            "train_fwd_bwd": train,
            "fp32_peak_probe": p32_meas,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_decode(args, cpr, inputs, dev, hbm_peak, dist, world):
    w = inputs.workload("rollout_decode")
    if args.decode_context:  # shorter prior contexts (profiling): the same positions modulo C
        w.seqlens = [(int(L) - 1) % args.decode_context + 1 for L in w.seqlens]
    B, H, dk, dv, C = len(w.seqlens), w.H, w.dk, w.dv, w.C
    x = inputs.prefill_inputs(w, device=dev)  # prior context, drawn on the device
    n_chunks = cpr.cpr_gdn_num_chunks(inputs.cu_seqlens_of(w.seqlens), C)
    _, st, bnd, ws = cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C,
                                         n_chunks=n_chunks)
    ring = cpr.cpr_gdn_ring_from_prefill(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, bnd, st)
    del x, bnd, ws
    torch.cuda.empty_cache()
    state = st
    n_steps = args.decode_steps
    toks = [inputs.decode_inputs(w, s, device=dev) for s in range(n_steps)]
    pos0 = torch.tensor(w.seqlens, dtype=torch.int32)
    pos = pos0.to(dev)
    out = torch.empty(B, H, dv, dtype=w.dtype, device=dev)
    dws = torch.empty(cpr.cpr_gdn_decode_workspace_size(B, H, dk, dv, C), dtype=torch.uint8, device=dev)

    def step(s):
        t = toks[s % n_steps]
        cpr.cpr_gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], state, ring, pos, C, out=out, workspace=dws)
        pos.add_(1)

    warm = max(3, args.warmup)
    for s in range(warm):
        step(s)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    step_ms, k4, k5 = [], [], []
    n_res = 0
    _barrier(dist)
    cpr.cpr_gdn_set_profile_events(ev)
    for s in range(warm, warm + n_steps):
        p_host = pos0 + s
        n_res += int(((p_host % C) == C - 1).sum())
        step(s)
        ev[2].synchronize()
        step_ms.append(ev[0].elapsed_time(ev[2]))
        k4.append(ev[0].elapsed_time(ev[1]))
        k5.append(ev[1].elapsed_time(ev[2]))
    cpr.cpr_gdn_set_profile_events(None)
    _barrier(dist)
    assert cpr.cpr_gdn_device_status(dws) == 0
    ms = _max_over_ranks(dist, statistics.fmean(step_ms))
    k4_ms = statistics.fmean(k4)
    bytes_step = decode_algorithmic(B, H, dk, dv, C, n_res / n_steps)
    step_only = decode_algorithmic(B, H, dk, dv, C, 0)
    ach = step_only / (k4_ms / 1e3) / 1e9
    # end to end: the step's tokens from pinned host memory, the outputs back
    pin = [{k: v.cpu().pin_memory() for k, v in t.items()} for t in toks[:8]]
    dbuf = {k: v.clone() for k, v in toks[0].items()}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pin[0].values())
    d2h = out_h.numel() * out_h.element_size()
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e = []
    for s in range(64):
        e_a.record()
        for k in dbuf:
            dbuf[k].copy_(pin[s % 8][k], non_blocking=True)
        cpr.cpr_gdn_decode(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["g"], dbuf["beta"], state, ring, pos, C, out=out,
                           workspace=dws)
        pos.add_(1)
        out_h.copy_(out, non_blocking=True)
        e_b.record()
        e_b.synchronize()
        e2e.append(e_a.elapsed_time(e_b))
    e2e_ms = _max_over_ranks(dist, statistics.fmean(e2e[4:]))
    return {
        "metric": "decode steps/s per layer", "value": 1e3 / ms * world, "unit": "steps/s",
        "ms_per_step": ms, "steps": n_steps, "workload": f"rollout_decode: B={B}, H={H}, dk=dv={dk}, C={C}, "
        + (f"prior lengths U[1,4096] capped at {args.decode_context} (profiling)" if args.decode_context
           else "prior lengths U[1,4096]") + ", state resident (> L2)",
        "kernels_ms": {"step_with_concurrent_resync": k4_ms, "join": statistics.fmean(k5)},
        "resyncs_per_step": n_res / n_steps,
        "roofline": {"kernel": "k4_decode_step", "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                     "frac": ach / hbm_peak, "traffic": TRAFFIC_K4_ROLLOUT_DECODE, "bytes_per_launch": step_only},
        "t_roof_ms": bytes_step / (hbm_peak * 1e9) * 1e3,
        "frac_of_t_roof": bytes_step / (hbm_peak * 1e9) * 1e3 / ms,
        "e2e": {"value": 1e3 / e2e_ms * world, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * n_steps,
    }


def run_continuation(args, cpr, inputs, dev, hbm_peak, dist, world):
    """Continuation prefill: the rollout_prefill sequences (5 x 2,048), each resumed at a
    seeded position in [1, 2047] with the state and ring a prefill of its first part left;
    the continuation of the rest is timed (state and ring restored outside the events)."""
    w = inputs.workload("rollout_prefill")
    H, dk, dv, C = w.H, w.dk, w.dv, w.C
    x = inputs.prefill_inputs(w, device=dev)
    lens = list(w.seqlens)
    gen = torch.Generator().manual_seed(w.seed + 17)
    splits = [int(torch.randint(1, L, (1,), generator=gen)) for L in lens]
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    keys = ("q", "k", "v", "g", "beta")

    def pack(parts):
        p = {k: torch.cat([t[k] for t in parts], 0).contiguous() for k in keys}
        p["cu_seqlens"] = inputs.cu_seqlens_of([t["q"].shape[0] for t in parts]).to(dev)
        return p

    seqs = [{k: x[k][cu[n]:cu[n + 1]] for k in keys} for n in range(len(lens))]
    first = pack([{k: t[k][:s] for k in keys} for t, s in zip(seqs, splits)])
    second = pack([{k: t[k][s:] for k in keys} for t, s in zip(seqs, splits)])
    _, st1, bnd1, _ = cpr.cpr_gdn_prefill(first["q"], first["k"], first["v"], first["g"], first["beta"],
                                          first["cu_seqlens"], C)
    ring0 = cpr.cpr_gdn_ring_from_prefill(first["k"], first["v"], first["g"], first["beta"], first["cu_seqlens"], C,
                                          bnd1, st1)
    pos0 = torch.tensor(splits, dtype=torch.int32, device=dev)
    n_chunks = cpr.continue_chunks(second["cu_seqlens"].cpu(), splits, C)
    T2 = second["q"].shape[0]
    out = torch.empty(T2, H, dv, dtype=w.dtype, device=dev)
    bnd = torch.empty(max(n_chunks, 1), H, dk, dv, dtype=torch.float32, device=dev)
    ws = torch.empty(cpr.cpr_gdn_prefill_workspace_size(T2, len(lens), H, dk, dv, C), dtype=torch.uint8, device=dev)
    state = st1.clone()
    ring = ring0.clone()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    def call():
        cpr.cpr_gdn_prefill_continue(second["q"], second["k"], second["v"], second["g"], second["beta"],
                                     second["cu_seqlens"], pos0, C, state, ring, out=out, boundary_states=bnd,
                                     workspace=ws)

    def restore():
        state.copy_(st1)
        for a, b in zip((ring.S_b, ring.k, ring.v, ring.g, ring.beta),
                        (ring0.S_b, ring0.k, ring0.v, ring0.g, ring0.beta)):
            a.copy_(b)

    for _ in range(args.warmup):
        restore()
        call()
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ms = []
    steps = max(3, min(args.steps, 50))
    _barrier(dist)
    for _ in range(steps):
        restore()
        flush.zero_()
        e0.record()
        call()
        e1.record()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    _barrier(dist)
    ms_max = _max_over_ranks(dist, statistics.fmean(ms))
    _, flops = prefill_algorithmic(T2, len(lens), H, dk, dv, n_chunks)
    t_roof = flops / (FP32_PEAK_TFLOPS * 1e12) * 1e3
    return {
        "metric": "continuation prefill tokens/s per layer", "value": weak_scaling_rate(world, T2, ms_max),
        "unit": "tokens/s", "ms_per_step": ms_max, "steps": steps,
        "workload": f"rollout_prefill resumed: 5 x 2,048 tokens, H={H}, dk=dv={dk}, C={C}, bf16; each sequence "
                    f"resumed at a seeded position (first parts {splits}), {T2} tokens continued",
        "t_roof_ms": t_roof, "frac_of_t_roof": t_roof / ms_max,
        "gpu_launches": 6 * steps,
    }


def _bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 8192^3, burst)"
    return 1900.0, "fallback"


def pik_cpu_baseline(x, w, rows=512):
    """The pik oracle's exact product (fp64, numpy) timed on the host cores for the first
    `rows` rows of X against all of W; reported in the product's own unit."""
    from oracle import pik

    xs = x[:rows].float().cpu().double().numpy()
    ws = w.float().cpu().double().numpy()
    pik.gemm_exact(xs[:8], ws)  # warm the BLAS threads
    t0 = time.perf_counter()
    pik.gemm_exact(xs, ws)
    sec = time.perf_counter() - t0
    flops = 2.0 * xs.shape[0] * ws.shape[0] * ws.shape[1]
    return {"value": flops / sec / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {xs.shape[0]} rows of X against all of W ({sec:.2f} s)"}


def run_pik(args, cpr, inputs, dev, dist, world):
    """Deterministic K-split product (pik): Y = X W^T with M = N = K = 8,192 and eight
    leaves, as one call over the whole tree, and as two rank calls of four leaves each plus
    the combine of their roots (the same bits); and the product under a four-leaf contract.  The operands (2 x 128 MB) and the result
    (256 MB) exceed L2, so no flush is needed between calls."""
    M = N = K = args.pik_size
    L = 8
    x, w = inputs.gemm_operands(M, N, K, seed=0, device=dev)
    y = torch.empty(M, N, dtype=torch.float32, device=dev)
    parts = torch.empty(2, M, N, dtype=torch.float32, device=dev)
    ws = torch.empty(cpr.cpr_pik_workspace_size(), dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def whole():
        cpr.cpr_pik_gemm(x, w, L, out=y, workspace=ws)

    def whole4():
        cpr.cpr_pik_gemm(x, w, 4, out=y, workspace=ws)

    def two_ranks():
        cpr.cpr_pik_gemm(x, w, L, (0, 4), out=parts[0], workspace=ws)
        cpr.cpr_pik_gemm(x, w, L, (4, 8), out=parts[1], workspace=ws)
        cpr.cpr_pik_combine(parts, out=y)

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        _barrier(dist)
        ms = []
        for _ in range(steps):
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        _barrier(dist)
        return _max_over_ranks(dist, statistics.fmean(ms))

    steps = max(3, min(args.steps, 20))
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = pik_cpu_baseline(x, w)
    ms = timed(whole, steps)
    ms2 = timed(two_ranks, steps)
    ms4 = timed(whole4, steps)
    assert cpr.cpr_gdn_device_status(ws) == 0
    flops = 2.0 * M * N * K
    tf = flops / (ms * 1e-3) / 1e12
    peak, kind = _bf16_peak()
    return {
        "metric": "pik deterministic K-split GEMM TFLOP/s", "value": tf * world, "unit": "TFLOP/s",
        "ms_per_call": ms, "steps": steps,
        "workload": f"Y = X W^T, M = N = K = {M}, bf16 operands, fp32 accumulation and result, {L} leaves",
        "roofline": {"kernel": "k_pik_leaves", "bound": "tensor", "achieved": tf, "peak": peak, "peak_kind": kind,
                     "unit": "TFLOP/s", "frac": tf / peak, "traffic": None, "flops_per_launch": flops},
        "cpu_baseline": cpu,
        "two_ranks_ms": ms2, "four_leaves_ms": ms4, "four_leaves_tflops": flops / (ms4 * 1e-3) / 1e12,
        "gpu_launches": 5 * steps,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="trainer_fwd")
    ap.add_argument("--decode-steps", type=int, default=512)
    ap.add_argument("--decode-context", type=int, default=0,
                    help="cap the rollout_decode prior contexts at this many tokens (a multiple of C, for "
                         "profiling: the state and the step are unchanged, the prior prefill smaller)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pik", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the rollout_prefill, varlen_stress and tiny lines")
    ap.add_argument("--no-train", action="store_true", help="skip the train_fwd_bwd line")
    ap.add_argument("--no-rollout-decode", action="store_true",
                    help="skip the rollout_decode leg (its prior prefill holds tens of GB); the continuation still runs")
    ap.add_argument("--only-pik", action="store_true")
    ap.add_argument("--pik-size", type=int, default=8192, help="M = N = K of the pik product (a multiple of 512)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
