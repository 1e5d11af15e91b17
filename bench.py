"""Throughput of the tensor-parallel MLP block (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--sweep]

One step = one training pass of the block over one batch: tp_mlp_forward
(training) followed by tp_mlp_backward, i.e. every kernel of the path
(GEMM1+GeLU, GEMM2 + shard sum, dH GEMM + GeLU', column sums, the two
weight-gradient GEMMs, dX GEMM + shard sum, and the LayerNorm kernels when the
workload has pre-LN).  Algorithmic work: 12 T h f flops per step (forward
4 T h f), whatever the shard count.  Inputs are seeded synthetic tensors of
the workload's shapes, resident in device memory before timing starts.
Where the weights alone exceed the 129 MB L2 (GPT-3-13B, 8.3B, BLOOM MLP
blocks; the GPT-3-13B attention block) no flush is inserted between steps;
otherwise a 256 MiB write evicts L2 before every timed step, outside the
step's events (config "l2" says which).

``--workload attn_gpt3_13b`` (or another ``attn_*`` workload) times the
head-parallel attention block instead: one step = tp_attn_forward (training)
+ tp_attn_backward (Q/K/V projection, attention core, output projection +
shard sum, and their gradients); algorithmic work 24 T h^2 for the
projections plus 12 d per unmasked (query, key) pair for the attention core.

``--fp8`` times the FP8 (E4M3) forward of an MLP workload instead (weights
quantized once before timing; per step: quantize Xn, GEMM1 + GeLU, quantize
Y, GEMM2 + shard sum; 4 T h f flops), against twice the measured bf16 peak.
``--fp8 --train`` times the FP8 training step (that forward keeping what the
backward needs, then the FP8 backward; 12 T h f flops).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on a bounded token slice of the same workload instead.  With
WORLD_SIZE > 1 (torchrun) every rank runs an independent replica on its own
GPU; ranks meet only at a barrier and a max-reduce of the timings (gloo), no
collective touches the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TP-MLP fwd+bwd TFLOP/s and tokens/s on 1 GB300, % of dense bf16 peak"
METRIC_FP8 = ("TP-MLP FP8 (E4M3) forward TFLOP/s and tokens/s on 1 GB300, "
              "% of dense fp8 peak")
METRIC_FP8_TRAIN = ("TP-MLP FP8 (E4M3) fwd+bwd TFLOP/s and tokens/s on 1 "
                    "GB300, % of dense fp8 peak")
METRIC_ATTN = ("TP-attention fwd+bwd TFLOP/s and tokens/s on 1 GB300, "
               "% of dense bf16 peak")
DEFAULT_WORKLOAD = "gpt3_13b"

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum)
# from full-size ncu captures, keyed by workload then kernel, with the hash of
# the kernel sources the capture was taken on ("gemm": the pair GEMM,
# "attn": the attention core).  Reported as null once the source has changed
# or for a workload without a capture.  The captures' commands and per-launch
# figures are kept with the other ncu summaries under profiles/.
_G, _A = "73fa3dd9ac5d98d6", "6f5294747167f930"
NCU_TRAFFIC = {
    # GPT-3-13B-shaped MLP step (T=8192, h=5120, f=20480, t=8)
    "gpt3_13b": {
        "gemm1_gelu": (1811.8e6, "gemm", _G),
        "gemm2_shardsum": (2255.5e6, "gemm", _G),
        "gemm_dh_gelu_bwd": (1812.7e6, "gemm", _G),
        "gemm_wgrad_dB": (2499.1e6, "gemm", _G),
        "gemm_wgrad_dA": (2315.8e6, "gemm", _G),
        "gemm_dx_shardsum": (2255.8e6, "gemm", _G),
    },
    # the same layer's FP8 forward
    "gpt3_13b_fp8": {
        "gemm1_gelu_fp8": (557.2e6, "gemm", _G),
        "gemm2_shardsum_fp8": (1151.1e6, "gemm", _G),
    },
    # the same layer's FP8 training step
    "gpt3_13b_fp8_train": {
        "gemm1_gelu_fp8": (913.6e6, "gemm", _G),
        "gemm2_shardsum_fp8": (1151.7e6, "gemm", _G),
        "gemm_dh_gelu_bwd_fp8": (954.4e6, "gemm", _G),
        "gemm_wgrad_dB_fp8": (971.3e6, "gemm", _G),
        "gemm_wgrad_dA_fp8": (894.5e6, "gemm", _G),
        "gemm_dx_shardsum_fp8": (1150.3e6, "gemm", _G),
    },
    # Megatron-8.3B-shaped pre-LN MLP step (T=8192, h=3072, f=12288, t=8)
    "megatron_8p3b": {
        "gemm1_ln_gelu": (697.4e6, "gemm", _G),
        "gemm2_shardsum": (828.7e6, "gemm", _G),
        "gemm_dh_gelu_bwd": (639.6e6, "gemm", _G),
        "gemm_wgrad_dB": (913.9e6, "gemm", _G),
        "gemm_wgrad_dA": (737.5e6, "gemm", _G),
        "gemm_dx_shardsum": (870.7e6, "gemm", _G),
    },
    # GPT-3-13B-shaped attention block (4 x 2048 tokens, 40 heads of 128)
    "attn_gpt3_13b": {
        "gemm_qkv": (924.9e6, "gemm", _G),
        "gemm_out_shardsum": (367.3e6, "gemm", _G),
        "gemm_wgrad_dWo": (619.6e6, "gemm", _G),
        "gemm_dctx": (366.9e6, "gemm", _G),
        "gemm_wgrad_dWqkv": (1756.4e6, "gemm", _G),
        "gemm_dx_shardsum": (1710.2e6, "gemm", _G),
        "attn_fwd": (311.4e6, "attn", _A),
        "attn_bwd_dq": (495.7e6, "attn", _A),
        "attn_bwd_dkdv": (483.0e6, "attn", _A),
    },
    # Megatron-8.3B-shaped pre-LN attention block (8 x 1024 tokens, 32 heads
    # of 96)
    "attn_megatron_8p3b": {
        "gemm_ln_qkv": (384.3e6, "gemm", _G),
        "gemm_out_shardsum": (105.9e6, "gemm", _G),
        "gemm_wgrad_dWo": (171.8e6, "gemm", _G),
        "gemm_dctx": (107.4e6, "gemm", _G),
        "gemm_wgrad_dWqkv": (554.6e6, "gemm", _G),
        "gemm_dx_shardsum": (667.8e6, "gemm", _G),
        "attn_fwd": (177.3e6, "attn", _A),
        "attn_bwd_dq": (293.4e6, "attn", _A),
        "attn_bwd_dkdv": (279.0e6, "attn", _A),
    },
}
_SRC_FILES = {"gemm": ("gemm_tc2.cu", "gemm_common.cuh", "ptx.cuh", "common.cuh"),
              "attn": ("attn_fwd.cu", "attn_bwd.cu", "attn_common.cuh")}


def traffic_of(workload, kernel):
    entry = NCU_TRAFFIC.get(workload, {}).get(kernel)
    if entry is None:
        return None
    nbytes, group, sha = entry
    return nbytes if _src_sha(_SRC_FILES[group]) == sha else None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return (p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                p["hbm_gbs"], "measured")
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


def _kernel_peak(region_s, peak_b, peak_s):
    """The dense peak a kernel inside the timed step is held to: the burst
    figure (a GEMM timed alone) unless the timed region lasts a second or
    more, the length of the sustained figure's own loop under the power cap,
    whatever clock the region's samples show."""
    if region_s < SUSTAINED_REGION_S:
        return peak_b, "burst"
    return peak_s, "sustained"


def e2e_overlapped(torch, stream, steps, h_in, h_out, d_in, d_out, compute):
    """End to end with the host copies overlapped with the compute: step i's
    inputs go up on one side stream while step i - 1 computes, its results
    come down on another while step i + 1 computes, through two device
    buffer slots.  d_in[s] / d_out[s] are slot s's device tensors (in the
    order of h_in / h_out, pinned host tensors); compute(s) enqueues one
    step on `stream` from d_in[s] into d_out[s].  Every step still moves
    all of its inputs up and all of its results down.  Returns ms per step
    (CUDA events on `stream`, from before the first upload to after the
    last download)."""
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    done, fetched = [None, None], [None, None]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)

    def upload(i):
        s = i % 2
        with torch.cuda.stream(up):
            if done[s] is not None:       # the slot's previous step has
                up.wait_event(done[s])    # finished reading its inputs
            for h, dv in zip(h_in, d_in[s]):
                dv.copy_(h, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(up)
        return ev

    nxt = upload(0)
    for i in range(steps):
        s = i % 2
        stream.wait_event(nxt)
        if fetched[s] is not None:        # its previous results are down
            stream.wait_event(fetched[s])
        compute(s)
        ev = torch.cuda.Event()
        ev.record(stream)
        done[s] = ev
        if i + 1 < steps:
            nxt = upload(i + 1)
        with torch.cuda.stream(down):
            down.wait_event(ev)
            for h, dv in zip(h_out, d_out[s]):
                h.copy_(dv, non_blocking=True)
            f = torch.cuda.Event()
            f.record(down)
            fetched[s] = f
    for f in fetched:
        if f is not None:
            stream.wait_event(f)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def _src_sha(files=_SRC_FILES["gemm"]):
    """Hash of the kernel sources a traffic figure depends on."""
    h = hashlib.sha256()
    for name in files:
        path = os.path.join(ROOT, "tensor_transformer_mlp_tcgen05_gb300",
                            "csrc", name)
        with open(path, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# Idle pause before each timed region (the device-timed steps, the two
# end-to-end runs and the cuBLAS context), each followed by a few untimed
# steps, so that every region starts warm from the same power state instead
# of the later ones inheriting the power-capped clock of the earlier ones.
SETTLE_S = 1.0
# Timed regions at least this long are held to the sustained peak.
SUSTAINED_REGION_S = 1.0


def settle(torch):
    torch.cuda.synchronize()
    time.sleep(SETTLE_S)


# GB300's L2; a workload whose weights fit in it is timed with a flush
# (a 256 MiB write) before every timed step.
L2_BYTES = 129 * 10 ** 6


def l2_flusher(torch, weight_bytes):
    """None when the weights alone exceed L2 (then every step streams more
    than L2 holds); otherwise a callable that writes a 256 MiB buffer on the
    current stream, evicting what the last step left in L2."""
    if weight_bytes > L2_BYTES:
        return None
    buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    return buf.zero_


def l2_note(flush):
    return ("inputs larger than L2 (no flush)" if flush is None else
            "L2 flushed (256 MiB write) before each timed step, the flush "
            "not timed; end-to-end runs not flushed")


def timed_steps(torch, stream, step, steps, flush=None):
    """Run `steps` steps with a CUDA event on `stream` before each and after
    the last; returns (mean ms per step over the whole region, per-step
    median / min / max in ms).  With `flush`, it runs before every step
    between the step's own pair of events, and the mean is over the steps'
    own times."""
    if flush is not None:
        ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush()
            ev0[i].record(stream)
            step()
            ev1[i].record(stream)
        torch.cuda.synchronize()
        per = [ev0[i].elapsed_time(ev1[i]) for i in range(steps)]
        stats = {"median": round(statistics.median(per), 4),
                 "min": round(min(per), 4), "max": round(max(per), 4)}
        return sum(per) / steps, stats
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record(stream)
    for i in range(steps):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    stats = {"median": round(statistics.median(per), 4),
             "min": round(min(per), 4), "max": round(max(per), 4)}
    return evs[0].elapsed_time(evs[-1]) / steps, stats


# ------------------------------------------------------------ clocks ----

class ClockSampler:
    """nvidia-smi sampling every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def begin(self):
        """Marks the start of the timed region: the summary keeps the
        samples from here to stop() (all of them if none falls inside)."""
        self.t0 = time.monotonic()

    def stop(self):
        if self.proc is None:
            return None
        t1 = time.monotonic()
        time.sleep(0.15)                  # the sample taken at the end
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        lines = [ln for t, ln in self.lines
                 if self.t0 is None or self.t0 <= t <= t1 + 0.12]
        for ln in lines or [ln for _, ln in self.lines]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "power_w_max": max(pw) if pw else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------- distributed ----

def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int) -> float:
    """Max of a float over ranks (gloo, host side); identity for world 1."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ oracle ----

def oracle_sample(w, inp, tokens, mode="erf"):
    """Time the fp64 oracle's forward + backward on the first `tokens` rows."""
    from oracle import mlp as O
    f64 = lambda t: None if t is None else t[:tokens].double().numpy() \
        if t.dim() == 2 and t.shape[0] == w.tokens else t.double().numpy()
    X, dZ = f64(inp["X"]), f64(inp["dZ"])
    A, B = inp["A"].double().numpy(), inp["B"].double().numpy()
    gamma, beta = f64(inp["gamma"]), f64(inp["beta"])
    t0 = time.perf_counter()
    fwd = O.forward(X, A, B, f64(inp["b1"]), f64(inp["b2"]), gamma, beta, mode=mode)
    if w.backward:
        O.backward(dZ, X, A, B, fwd, gamma, mode)
    return time.perf_counter() - t0


def oracle_tokens(w):
    """Token slice sized for roughly 10-30 s of fp64 work on the host."""
    per_token = (12.0 if w.backward else 4.0) * w.hidden * w.ffn
    return int(max(16, min(w.tokens, 1.5e12 / per_token)))


# -------------------------------------------------------------- ours ----

def run_ours(args, w, rank, world, local_rank):
    import torch
    from tensor_transformer_mlp_tcgen05_gb300 import binding as Bn
    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    inp = W.make_inputs(w, seed=0)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    m = TensorParallelMLP(w.hidden, w.ffn, w.shards, w.tokens, dtype=w.dtype,
                          layernorm=w.layernorm, residual=args.residual,
                          ln_prologue=not args.ln_standalone)
    stream = torch.cuda.current_stream()
    T = w.tokens
    Z = torch.empty((T, w.hidden), dtype=w.torch_dtype, device=dev)
    grads = {}

    def step(Xd=None, dZd=None):
        Xd = d["X"] if Xd is None else Xd
        dZd = d["dZ"] if dZd is None else dZd
        m.forward(Xd, d["A"], d["B"], d["b1"], d["b2"], d["gamma"], d["beta"],
                  training=w.backward, out=Z)
        if w.backward:
            m.backward(dZd, Xd, d["A"], d["B"], d["gamma"], bias_grads=True,
                       out=grads)

    for _ in range(args.warmup):
        step()
    if m.check() != 0:
        raise RuntimeError("device status after warm-up: "
                           + Bn.tp_mlp_last_detail())
    torch.cuda.synchronize()

    # Bitwise run-to-run identity of every output (two consecutive steps).
    snap = {"Z": Z.clone(), **{k: v.clone() for k, v in grads.items()}}
    step()
    torch.cuda.synchronize()
    identical = all(torch.equal(snap[k], (Z if k == "Z" else grads[k]))
                    for k in snap)

    # ---- timed region: K steps, events on the launching stream ----
    Bn.tp_mlp_set_timing(m.handle, True)
    Bn.tp_mlp_timing_reset(m.handle)
    flush = l2_flusher(torch, 4 * w.hidden * w.ffn)   # weight bytes
    settle(torch)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.25)
    for _ in range(3):            # back from the pause, untimed
        step()
    torch.cuda.synchronize()
    Bn.tp_mlp_timing_reset(m.handle)
    barrier(world)
    torch.cuda.synchronize()
    sampler.begin()
    n0 = Bn.tp_mlp_launch_count(m.handle)
    ms, step_ms = timed_steps(torch, stream, step, args.steps, flush)
    barrier(world)
    clocks = sampler.stop()
    launches = Bn.tp_mlp_launch_count(m.handle) - n0
    if m.check() != 0:
        raise RuntimeError("device status after timing: " + Bn.tp_mlp_last_detail())
    kernels = Bn.tp_mlp_timing_get(m.handle)
    Bn.tp_mlp_set_timing(m.handle, False)
    ms_max = max_over_ranks(ms, world)

    # ---- end to end: pinned host inputs in, results out, every step ----
    hX = inp["X"].pin_memory()
    hdZ = inp["dZ"].pin_memory() if w.backward else None
    hZ = torch.empty_like(inp["X"]).pin_memory()
    hdX = torch.empty_like(inp["X"]).pin_memory() if w.backward else None
    Xd = torch.empty_like(d["X"])
    dZd = torch.empty_like(d["X"]) if w.backward else None
    h2d = hX.numel() * hX.element_size() * (2 if w.backward else 1)
    d2h = hZ.numel() * hZ.element_size() * (2 if w.backward else 1)

    def e2e_step():
        Xd.copy_(hX, non_blocking=True)
        if w.backward:
            dZd.copy_(hdZ, non_blocking=True)
        step(Xd, dZd)
        hZ.copy_(Z, non_blocking=True)
        if w.backward:
            hdX.copy_(grads["dX"], non_blocking=True)

    # the same with the copies overlapped (two slots, side streams)
    d_in = [[torch.empty_like(d["X"])] + ([torch.empty_like(d["X"])]
                                          if w.backward else [])
            for _ in range(2)]
    d_out = [[torch.empty_like(Z)] + ([torch.empty_like(d["X"])]
                                      if w.backward else [])
             for _ in range(2)]
    slot_grads = [dict(grads, dX=d_out[k][1]) if w.backward else None
                  for k in range(2)]

    def compute(k):
        m.forward(d_in[k][0], d["A"], d["B"], d["b1"], d["b2"], d["gamma"],
                  d["beta"], training=w.backward, out=d_out[k][0])
        if w.backward:
            m.backward(d_in[k][1], d_in[k][0], d["A"], d["B"], d["gamma"],
                       bias_grads=True, out=slot_grads[k])

    h_in = [hX] + ([hdZ] if w.backward else [])
    h_out = [hZ] + ([hdX] if w.backward else [])
    settle(torch)
    e2e_overlapped(torch, stream, 2, h_in, h_out, d_in, d_out, compute)
    barrier(world)
    e2e_ms = max_over_ranks(
        e2e_overlapped(torch, stream, args.steps, h_in, h_out, d_in, d_out,
                       compute), world)
    # the same with the copies serialised on the compute stream
    settle(torch)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e3.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(e2.elapsed_time(e3) / args.steps, world)
    if m.check() != 0:
        raise RuntimeError("device status after the end-to-end runs: "
                           + Bn.tp_mlp_last_detail())

    flops = w.flops_fwd_bwd() if w.backward else w.flops_fwd()
    peak_b, peak_s, hbm, peak_src = _peaks()
    tflops = world * flops / (ms_max * 1e-3) / 1e12
    total_ms = sum(k[2] for k in kernels) or 1.0
    krep = [{"name": n, "launches": c, "avg_ms": round(t / max(c, 1), 4),
             "share": round(t / total_ms, 4)} for n, c, t in kernels]
    krep.sort(key=lambda r: -r["share"])
    top = krep[0]
    roof = None
    gemm_flops = {
        "gemm1_gelu": 2.0 * w.tokens * w.hidden * w.ffn,
        "gemm1_ln_gelu": 2.0 * w.tokens * w.hidden * w.ffn,
        "gemm2_shardsum": 2.0 * w.tokens * w.hidden * w.ffn,
        "gemm_dh_gelu_bwd": 2.0 * w.tokens * w.hidden * w.ffn,
        "gemm_wgrad_dB": 2.0 * w.tokens * w.hidden * w.ffn,
        "gemm_wgrad_dA": 2.0 * w.tokens * w.hidden * w.ffn,
        "gemm_dx_shardsum": 2.0 * w.tokens * w.hidden * w.ffn,
    }
    if top["name"] in gemm_flops:
        ach = gemm_flops[top["name"]] / (top["avg_ms"] * 1e-3) / 1e12
        traffic = traffic_of(w.name, top["name"]) \
            if not (args.tokens or args.shards or args.residual) else None
        pk, pkind = _kernel_peak(ms_max * args.steps / 1e3, peak_b, peak_s)
        roof = {"kernel": top["name"], "bound": "tensor",
                "achieved": round(ach, 1), "peak": pk, "unit": "TFLOP/s",
                "frac": round(ach / pk, 4),
                "peak_kind": f"bf16 {pkind} ({peak_src})",
                "traffic": traffic}

    line = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOP/s",
        "tokens_per_s": round(world * w.tokens / (ms_max * 1e-3), 1),
        "frac_of_peak": round(tflops / (world * peak_b), 4),
        "peak_tflops": peak_b, "peak_kind": f"bf16 burst ({peak_src})",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4), "step_ms": step_ms,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: seeded N(0,1) activations and upstream gradient, "
                f"N(0,{w.w_std}^2) weights",
        "config": {"workload": w.name, "tokens": w.tokens, "batch": w.batch,
                   "seq": w.seq, "hidden": w.hidden, "ffn": w.ffn,
                   "shards": w.shards, "layernorm": w.layernorm,
                   "ln_prologue": bool(w.layernorm and not args.ln_standalone),
                   "residual": bool(args.residual),
                   "pass": "fwd+bwd" if w.backward else "fwd",
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": l2_note(flush),
                   "idle_before_timed_s": SETTLE_S},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "overlapped with the compute (side streams, two "
                          "buffer slots)",
                "serial_value": round(world * flops / (e2e_serial_ms * 1e-3)
                                      / 1e12, 2),
                "serial_ms_per_step": round(e2e_serial_ms, 4)},
        "gpu_launches": launches,
        "bitwise_identical_two_runs": identical,
        "clocks": clocks,
        "roofline": roof,
        "kernels": krep,
    }
    m.close()
    line["spec_peak"] = spec_peak(clocks, tflops / world)
    line["vendor_context"] = vendor_context(w, d, args)
    return line, inp


def spec_peak(clocks, tflops_per_gpu):
    """Clock-based dense peak: SMs x the per-SM bf16 rate measured by the
    library's tensor-core probe (one thread per SM issuing back-to-back
    128 x 256 x 16 MMAs) x the median SM clock seen during the timed region."""
    from tensor_transformer_mlp_tcgen05_gb300 import binding as Bn
    rate, sms = Bn.mma_flops_per_cycle(256)
    mhz = (clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz")
    out = {"flops_per_sm_cycle": round(rate, 1), "sms": sms, "sm_mhz": mhz,
           "what": "SMs x measured flops/SM/cycle x median SM clock"}
    if mhz:
        peak = rate * sms * mhz * 1e6 / 1e12
        out.update(tflops=round(peak, 1), frac=round(tflops_per_gpu / peak, 4))
    return out


def vendor_context(w, d, args):
    """torch bf16 matmul + GeLU (cuBLAS), unsharded, same shapes, autograd
    forward (+ backward), as vendor-library context only."""
    import torch
    import torch.nn.functional as F
    X = d["X"].detach().clone().requires_grad_(w.backward)
    A = d["A"].detach().clone().requires_grad_(w.backward)
    B = d["B"].detach().clone().requires_grad_(w.backward)

    def step():
        Xn = F.layer_norm(X, (w.hidden,), d["gamma"].to(X.dtype),
                          d["beta"].to(X.dtype)) if w.layernorm else X
        Z = F.gelu(Xn @ A) @ B
        if w.backward:
            X.grad = A.grad = B.grad = None
            Z.backward(d["dZ"])
        return Z

    with torch.enable_grad():
        settle(torch)
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        n = max(3, min(args.steps, 20))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    flops = w.flops_fwd_bwd() if w.backward else w.flops_fwd()
    return {"value": round(flops / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": n,
            "what": "torch bf16 matmul + gelu (cuBLAS), unsharded, autograd "
                    + ("fwd+bwd" if w.backward else "fwd")}


def attn_kernel_flops(w):
    """Algorithmic flops per launch of each attention-block kernel."""
    T, h = w.tokens, w.hidden
    core = 2.0 * w.head_dim * w.score_pairs()      # one pair-wise matmul
    return {"gemm_qkv": 6.0 * T * h * h, "gemm_ln_qkv": 6.0 * T * h * h,
            "gemm_out_shardsum": 2.0 * T * h * h,
            "gemm_wgrad_dWo": 2.0 * T * h * h, "gemm_dctx": 2.0 * T * h * h,
            "gemm_wgrad_dWqkv": 6.0 * T * h * h,
            "gemm_dx_shardsum": 6.0 * T * h * h,
            "attn_fwd": 2 * core,          # Q K^T, P V
            "attn_bwd_dkdv": 2 * core,     # dV = P^T dO, dK = dS^T Q
            "attn_bwd_dq": 2 * core}       # dP = dO V^T, dQ = dS K


def run_ours_attn(args, w, rank, world, local_rank):
    import torch
    from tensor_transformer_mlp_tcgen05_gb300 import binding as Bn
    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    from tensor_transformer_mlp_tcgen05_gb300.attention import \
        TensorParallelAttention

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    inp = W.make_attn_inputs(w, seed=0, with_bias=True)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    m = TensorParallelAttention(w.hidden, w.heads, w.shards, w.tokens, w.seq,
                                causal=w.causal, layernorm=w.layernorm,
                                residual=args.residual)
    stream = torch.cuda.current_stream()
    T, h = w.tokens, w.hidden
    Z = torch.empty((T, h), dtype=torch.bfloat16, device=dev)
    grads = {}

    def step(Xd=None, dZd=None):
        Xd = d["X"] if Xd is None else Xd
        dZd = d["dZ"] if dZd is None else dZd
        m.forward(Xd, d["Wqkv"], d["Wo"], d["bqkv"], d["bo"], d["gamma"],
                  d["beta"], training=True, out=Z)
        m.backward(dZd, Xd, d["Wqkv"], d["Wo"], d["gamma"], out=grads)

    for _ in range(args.warmup):
        step()
    if m.check() != 0:
        raise RuntimeError("device status after warm-up: "
                           + Bn.tp_mlp_last_detail())
    torch.cuda.synchronize()
    snap = {"Z": Z.clone(), **{k: v.clone() for k, v in grads.items()}}
    step()
    torch.cuda.synchronize()
    identical = all(torch.equal(snap[k], (Z if k == "Z" else grads[k]))
                    for k in snap)

    Bn.tp_attn_set_timing(m.handle, True)
    Bn.tp_attn_timing_reset(m.handle)
    flush = l2_flusher(torch, 8 * w.hidden * w.hidden)   # weight bytes
    settle(torch)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.25)
    for _ in range(3):            # back from the pause, untimed
        step()
    torch.cuda.synchronize()
    Bn.tp_attn_timing_reset(m.handle)
    barrier(world)
    torch.cuda.synchronize()
    sampler.begin()
    n0 = Bn.tp_attn_launch_count(m.handle)
    ms, step_ms = timed_steps(torch, stream, step, args.steps, flush)
    barrier(world)
    clocks = sampler.stop()
    launches = Bn.tp_attn_launch_count(m.handle) - n0
    if m.check() != 0:
        raise RuntimeError("device status after timing: "
                           + Bn.tp_mlp_last_detail())
    kernels = Bn.tp_attn_timing_get(m.handle)
    Bn.tp_attn_set_timing(m.handle, False)
    ms_max = max_over_ranks(ms, world)

    hX = inp["X"].pin_memory()
    hdZ = inp["dZ"].pin_memory()
    hZ = torch.empty_like(inp["X"]).pin_memory()
    hdX = torch.empty_like(inp["X"]).pin_memory()
    Xd = torch.empty_like(d["X"])
    dZd = torch.empty_like(d["X"])
    h2d = 2 * hX.numel() * hX.element_size()
    d2h = 2 * hZ.numel() * hZ.element_size()

    def e2e_step():
        Xd.copy_(hX, non_blocking=True)
        dZd.copy_(hdZ, non_blocking=True)
        step(Xd, dZd)
        hZ.copy_(Z, non_blocking=True)
        hdX.copy_(grads["dX"], non_blocking=True)

    d_in = [[torch.empty_like(d["X"]), torch.empty_like(d["X"])]
            for _ in range(2)]
    d_out = [[torch.empty_like(Z), torch.empty_like(d["X"])] for _ in range(2)]
    slot_grads = [dict(grads, dX=d_out[k][1]) for k in range(2)]

    def compute(k):
        m.forward(d_in[k][0], d["Wqkv"], d["Wo"], d["bqkv"], d["bo"],
                  d["gamma"], d["beta"], out=d_out[k][0])
        m.backward(d_in[k][1], d_in[k][0], d["Wqkv"], d["Wo"], d["gamma"],
                   out=slot_grads[k])

    settle(torch)
    e2e_overlapped(torch, stream, 2, [hX, hdZ], [hZ, hdX], d_in, d_out,
                   compute)
    barrier(world)
    e2e_ms = max_over_ranks(
        e2e_overlapped(torch, stream, args.steps, [hX, hdZ], [hZ, hdX], d_in,
                       d_out, compute), world)
    # the same with the copies serialised on the compute stream
    settle(torch)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e3.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(e2.elapsed_time(e3) / args.steps, world)
    if m.check() != 0:
        raise RuntimeError("device status after the end-to-end runs: "
                           + Bn.tp_mlp_last_detail())

    flops = w.flops_fwd_bwd()
    peak_b, peak_s, hbm, peak_src = _peaks()
    tflops = world * flops / (ms_max * 1e-3) / 1e12
    total_ms = sum(k[2] for k in kernels) or 1.0
    krep = [{"name": n, "launches": c, "avg_ms": round(t / max(c, 1), 4),
             "share": round(t / total_ms, 4)} for n, c, t in kernels]
    krep.sort(key=lambda r: -r["share"])
    kf = attn_kernel_flops(w)
    for r in krep:
        if r["name"] in kf:
            r["tflops"] = round(kf[r["name"]] / (r["avg_ms"] * 1e-3) / 1e12, 1)
    top = krep[0]
    roof = None
    if top["name"] in kf:
        ach = kf[top["name"]] / (top["avg_ms"] * 1e-3) / 1e12
        traffic = traffic_of(w.name, top["name"]) \
            if not (args.tokens or args.shards or args.residual) else None
        pk, pkind = _kernel_peak(ms_max * args.steps / 1e3, peak_b, peak_s)
        roof = {"kernel": top["name"], "bound": "tensor",
                "achieved": round(ach, 1), "peak": pk, "unit": "TFLOP/s",
                "frac": round(ach / pk, 4),
                "peak_kind": f"bf16 {pkind} ({peak_src})",
                "traffic": traffic}
    line = {
        "metric": METRIC_ATTN, "value": round(tflops, 2), "unit": "TFLOP/s",
        "tokens_per_s": round(world * T / (ms_max * 1e-3), 1),
        "frac_of_peak": round(tflops / (world * peak_b), 4),
        "peak_tflops": peak_b, "peak_kind": f"bf16 burst ({peak_src})",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4), "step_ms": step_ms,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) activations and upstream gradient, "
                f"N(0,{w.w_std}^2) weights, N(0,0.25) biases",
        "config": {"workload": w.name, "tokens": T, "batch": w.batch,
                   "seq": w.seq, "hidden": h, "heads": w.heads,
                   "head_dim": w.head_dim, "shards": w.shards,
                   "causal": w.causal, "layernorm": w.layernorm,
                   "residual": bool(args.residual), "pass": "fwd+bwd",
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": l2_note(flush),
                   "idle_before_timed_s": SETTLE_S},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "overlapped with the compute (side streams, two "
                          "buffer slots)",
                "serial_value": round(world * flops / (e2e_serial_ms * 1e-3)
                                      / 1e12, 2),
                "serial_ms_per_step": round(e2e_serial_ms, 4)},
        "gpu_launches": launches,
        "bitwise_identical_two_runs": identical,
        "clocks": clocks,
        "roofline": roof,
        "kernels": krep,
    }
    m.close()
    return line, inp


def attn_oracle_sample(w, inp, seqs, seq_len=None):
    """Time the fp64 attention oracle's forward + backward on the first
    `seqs` sequences (optionally cut to their first `seq_len` tokens)."""
    from oracle import attention as OA
    S = seq_len or w.seq
    rows = [r for b in range(seqs) for r in range(b * w.seq, b * w.seq + S)]
    f = lambda t: None if t is None else t.double().numpy()
    X, dZ = f(inp["X"][rows]), f(inp["dZ"][rows])
    Wqkv, Wo = f(inp["Wqkv"]), f(inp["Wo"])
    t0 = time.perf_counter()
    fwd = OA.forward(X, Wqkv, Wo, w.heads, S, w.shards, bqkv=f(inp["bqkv"]),
                     bo=f(inp["bo"]), gamma=f(inp["gamma"]),
                     beta=f(inp["beta"]), causal=w.causal)
    OA.backward(dZ, X, Wqkv, Wo, fwd, w.heads, S, w.shards,
                gamma=f(inp["gamma"]), causal=w.causal)
    return time.perf_counter() - t0


def run_cpu_baseline_attn(w, inp):
    secs = attn_oracle_sample(w, inp, 1)
    flops = w.with_(batch=1).flops_fwd_bwd()
    return {"value": round(flops / secs / 1e12, 5), "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first sequence ({w.seq} of {w.tokens} tokens), fp64 "
                      f"fwd+bwd ({secs:.1f} s)"}


def run_reference_attn(args, w):
    """The oracle as the reference arm for an attention workload: each step
    is the first sequence cut to its first 256 tokens, fp64 on the host."""
    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    S = min(256, w.seq)
    ws = w.with_(batch=1, seq=S)
    inp = W.make_attn_inputs(ws, seed=0, with_bias=True)
    for _ in range(args.warmup):
        attn_oracle_sample(ws, inp, 1)
    t = sum(attn_oracle_sample(ws, inp, 1) for _ in range(args.steps))
    sec = t / args.steps
    val = ws.flops_fwd_bwd() / sec / 1e12
    return {
        "impl": "reference", "metric": METRIC_ATTN, "value": round(val, 5),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.tokens, "hidden": w.hidden,
                   "heads": w.heads, "shards": w.shards, "seq": w.seq},
        "cpu_baseline": {"value": round(val, 5), "unit": "TFLOP/s",
                         "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"one sequence of {S} tokens per step, "
                                   "fp64"},
        "e2e": {"value": round(val, 5), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }



def run_ours_fp8(args, w, rank, world, local_rank):
    """FP8 (E4M3) forward of an MLP workload: one step = quantize Xn, GEMM1
    + GeLU (+ amax of Y), quantize Y, GEMM2 + shard sum; the weights are
    packed once before timing.  With --train a step is the FP8 training
    step: that forward keeping H and the transposed codes, then the FP8
    backward (quantize dZ, dH GEMM + GeLU' + amax + db1 partials, quantize
    dH, db2 and db1 sums, dB and dA GEMMs, dX GEMM + shard sum [+ LayerNorm
    backward]).  The bf16 pass of the same workload is timed alongside for
    context."""
    import torch
    from tensor_transformer_mlp_tcgen05_gb300 import binding as Bn
    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    train = bool(args.train)
    inp = W.make_inputs(w, seed=0, need_grad_input=train)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    m = TensorParallelMLP(w.hidden, w.ffn, w.shards, w.tokens, dtype="bf16",
                          layernorm=w.layernorm, residual=args.residual)
    packed = m.pack_fp8_weights(d["A"], d["B"])
    stream = torch.cuda.current_stream()
    T = w.tokens
    Z = torch.empty((T, w.hidden), dtype=torch.bfloat16, device=dev)
    grads = {}

    def step(Xd=None, dZd=None, Zd=None, dXd=None):
        Xd = d["X"] if Xd is None else Xd
        m.forward_fp8(Xd, packed, d["b1"], d["b2"], d["gamma"], d["beta"],
                      out=Z if Zd is None else Zd, train=train)
        if train:
            g = grads if dXd is None else {**grads, "dX": dXd}
            m.backward_fp8(d["dZ"] if dZd is None else dZd, Xd, packed,
                           d["gamma"], bias_grads=True, grads=g)

    for _ in range(args.warmup):
        step()
    if m.check() != 0:
        raise RuntimeError("device status after warm-up: "
                           + Bn.tp_mlp_last_detail())
    if train:  # keep the gradient buffers from here on
        grads.update(m.backward_fp8(d["dZ"], d["X"], packed, d["gamma"],
                                    bias_grads=True))
    torch.cuda.synchronize()
    snap = {"Z": Z.clone(), **{k: v.clone() for k, v in grads.items()}}
    step()
    torch.cuda.synchronize()
    identical = all(torch.equal(snap[k], Z if k == "Z" else grads[k])
                    for k in snap)

    def timed(fn, n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    Bn.tp_mlp_set_timing(m.handle, True)
    Bn.tp_mlp_timing_reset(m.handle)
    flush = l2_flusher(torch, 2 * w.hidden * w.ffn)   # weight bytes
    settle(torch)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.25)
    for _ in range(3):            # back from the pause, untimed
        step()
    torch.cuda.synchronize()
    Bn.tp_mlp_timing_reset(m.handle)
    barrier(world)
    torch.cuda.synchronize()
    sampler.begin()
    n0 = Bn.tp_mlp_launch_count(m.handle)
    ms, step_ms = timed_steps(torch, stream, step, args.steps, flush)
    barrier(world)
    clocks = sampler.stop()
    launches = Bn.tp_mlp_launch_count(m.handle) - n0
    if m.check() != 0:
        raise RuntimeError("device status after timing: " + Bn.tp_mlp_last_detail())
    kernels = Bn.tp_mlp_timing_get(m.handle)
    Bn.tp_mlp_set_timing(m.handle, False)
    ms_max = max_over_ranks(ms, world)

    # the bf16 pass of the same workload, for context
    bgrads = {}

    def step_bf16():
        m.forward(d["X"], d["A"], d["B"], d["b1"], d["b2"], d["gamma"],
                  d["beta"], training=train, out=Z)
        if train:
            m.backward(d["dZ"], d["X"], d["A"], d["B"], d["gamma"],
                       bias_grads=True, out=bgrads)
    for _ in range(3):
        step_bf16()
    bf16_ms = timed(step_bf16, args.steps)

    hX = inp["X"].pin_memory()
    hZ = torch.empty_like(inp["X"]).pin_memory()
    Xd = torch.empty_like(d["X"])
    hdZ = inp["dZ"].pin_memory() if train else None
    hdX = torch.empty_like(inp["X"]).pin_memory() if train else None
    dZd = torch.empty_like(d["X"]) if train else None

    def e2e_step():
        Xd.copy_(hX, non_blocking=True)
        if train:
            dZd.copy_(hdZ, non_blocking=True)
        step(Xd, dZd)
        hZ.copy_(Z, non_blocking=True)
        if train:
            hdX.copy_(grads["dX"], non_blocking=True)

    nio = 2 if train else 1
    d_in = [[torch.empty_like(d["X"]) for _ in range(nio)] for _ in range(2)]
    d_out = [[torch.empty_like(Z) for _ in range(nio)] for _ in range(2)]
    h_in = [hX] + ([hdZ] if train else [])
    h_out = [hZ] + ([hdX] if train else [])

    def compute(k):
        step(d_in[k][0], d_in[k][1] if train else None, d_out[k][0],
             d_out[k][1] if train else None)

    settle(torch)
    e2e_overlapped(torch, stream, 2, h_in, h_out, d_in, d_out, compute)
    barrier(world)
    e2e_ms = max_over_ranks(
        e2e_overlapped(torch, stream, args.steps, h_in, h_out, d_in, d_out,
                       compute), world)
    # the same with the copies serialised on the compute stream
    settle(torch)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e2e_serial_ms = max_over_ranks(timed(e2e_step, args.steps), world)
    if m.check() != 0:
        raise RuntimeError("device status after the end-to-end runs: "
                           + Bn.tp_mlp_last_detail())

    flops = w.flops_fwd_bwd() if train else w.flops_fwd()
    peak_b, peak_s, hbm, peak_src = _peaks()
    fp8_burst, fp8_sust = 2 * peak_b, 2 * peak_s
    tflops = world * flops / (ms_max * 1e-3) / 1e12
    total_ms = sum(k[2] for k in kernels) or 1.0
    krep = [{"name": n, "launches": c, "avg_ms": round(t / max(c, 1), 4),
             "share": round(t / total_ms, 4)} for n, c, t in kernels]
    krep.sort(key=lambda r: -r["share"])
    gemm = 2.0 * w.tokens * w.hidden * w.ffn
    kf = {k: gemm for k in ("gemm1_gelu_fp8", "gemm2_shardsum_fp8",
                            "gemm_dh_gelu_bwd_fp8", "gemm_wgrad_dB_fp8",
                            "gemm_wgrad_dA_fp8", "gemm_dx_shardsum_fp8")}
    for r in krep:
        if r["name"] in kf:
            r["tflops"] = round(kf[r["name"]] / (r["avg_ms"] * 1e-3) / 1e12, 1)
    top = krep[0]
    roof = None
    if top["name"] in kf:
        ach = kf[top["name"]] / (top["avg_ms"] * 1e-3) / 1e12
        pk, pkind = _kernel_peak(ms_max * args.steps / 1e3, fp8_burst,
                                 fp8_sust)
        roof = {"kernel": top["name"], "bound": "tensor",
                "achieved": round(ach, 1), "peak": pk,
                "unit": "TFLOP/s", "frac": round(ach / pk, 4),
                "peak_kind": f"fp8 = 2 x measured bf16 {pkind} ({peak_src}; "
                             "nominal fp8:bf16 ratio 4.5:2.25)",
                "traffic": traffic_of(w.name + ("_fp8_train" if train
                                                else "_fp8"), top["name"])
                if not (args.tokens or args.shards or args.residual)
                else None}
    line = {
        "metric": METRIC_FP8_TRAIN if train else METRIC_FP8,
        "value": round(tflops, 2), "unit": "TFLOP/s",
        "tokens_per_s": round(world * T / (ms_max * 1e-3), 1),
        "frac_of_peak": round(tflops / (world * fp8_burst), 4),
        "peak_tflops": fp8_burst, "peak_kind": "fp8 (2 x measured bf16 burst)",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4), "step_ms": step_ms,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic: seeded N(0,1) activations, "
                f"N(0,{w.w_std}^2) weights"
                + (f", N(0,{w.dz_std}^2) output gradients" if train else "")
                + "; weights quantized once before timing, activations "
                + ("and gradients " if train else "") + "quantized every step",
        "config": {"workload": w.name, "tokens": T, "batch": w.batch,
                   "seq": w.seq, "hidden": w.hidden, "ffn": w.ffn,
                   "shards": w.shards, "layernorm": w.layernorm,
                   "residual": bool(args.residual),
                   "pass": "fwd+bwd (fp8)" if train else "fwd (fp8)",
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": l2_note(flush),
                   "idle_before_timed_s": SETTLE_S},
        ("bf16_train_step" if train else "bf16_forward"): {
                         "ms_per_step": round(bf16_ms, 4),
                         "value": round(flops / (bf16_ms * 1e-3) / 1e12, 2),
                         "unit": "TFLOP/s"},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": sum(t.numel() * t.element_size()
                                          for t in h_in),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size()
                                          for t in h_out),
                "copies": "overlapped with the compute (side streams, two "
                          "buffer slots)",
                "serial_value": round(world * flops / (e2e_serial_ms * 1e-3)
                                      / 1e12, 2),
                "serial_ms_per_step": round(e2e_serial_ms, 4)},
        "gpu_launches": launches,
        "bitwise_identical_two_runs": identical,
        "clocks": clocks,
        "roofline": roof,
        "kernels": krep,
    }
    m.close()
    return line, inp


def run_cpu_baseline_fp8(w, inp, train=False):
    """The fp64 FP8 oracle's forward (and, with train, backward) on a
    bounded token slice."""
    from oracle import fp8 as OF
    # the weights' quantization (2 h f elements) is a fixed cost of about
    # 15 s per GPT-3-13B-sized matrix; the token slice adds little to it
    tokens = int(max(16, min(w.tokens, 0.1e12 / (4.0 * w.hidden * w.ffn))))
    f = lambda t: None if t is None else t.double().numpy()
    X = f(inp["X"][:tokens])
    t0 = time.perf_counter()
    fwd = OF.forward(X, f(inp["A"]), f(inp["B"]), f(inp["b1"]), f(inp["b2"]),
                     f(inp["gamma"]), f(inp["beta"]))
    if train:
        OF.backward(f(inp["dZ"][:tokens]), X, fwd, f(inp["gamma"]))
    secs = time.perf_counter() - t0
    flops = w.flops_fwd_bwd(tokens) if train else w.flops_fwd(tokens)
    what = "forward + backward" if train else "forward"
    return {"value": round(flops / secs / 1e12, 5), "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {tokens} of {w.tokens} tokens, fp64 FP8 "
                      f"{what} incl. weight quantization ({secs:.1f} s)"}


def run_cpu_baseline(w, inp):
    import numpy as np  # noqa: F401  (BLAS threads are set at import)
    tokens = oracle_tokens(w)
    secs = oracle_sample(w, inp, tokens)
    flops = (w.flops_fwd_bwd(tokens) if w.backward else w.flops_fwd(tokens))
    line = {"value": round(flops / secs / 1e12, 5), "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {tokens} of {w.tokens} tokens, fp64 "
                      f"{'fwd+bwd' if w.backward else 'fwd'} ({secs:.1f} s)"}
    line["one_core"] = oracle_one_core(w, max(16, tokens // 16))
    return line


def oracle_one_core(w, tokens):
    """The same oracle sample on one host thread: a child process started
    with the BLAS and OpenMP thread counts set to 1 before numpy loads,
    on the same seeded inputs (regenerated there), `tokens` rows."""
    code = (
        "import sys, json; sys.path.insert(0, %r); import bench; "
        "from tensor_transformer_mlp_tcgen05_gb300 import workloads as W; "
        "w = W.WORKLOADS[%r].with_(tokens=%d, shards=%d); "
        "inp = W.make_inputs(w, seed=0); "
        "print(json.dumps(bench.oracle_sample(w, inp, %d)))"
        % (ROOT, w.name, w.tokens, w.shards, tokens))
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
              "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS"):
        env[k] = "1"
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env,
                             capture_output=True, text=True, timeout=600)
        secs = float(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: the all-core figure stands
        return {"error": f"{type(e).__name__}: {e}"[:200]}
    flops = (w.flops_fwd_bwd(tokens) if w.backward else w.flops_fwd(tokens))
    return {"value": round(flops / secs / 1e12, 5), "unit": "TFLOP/s",
            "threads": 1, "sample": f"first {tokens} of {w.tokens} tokens "
                                    f"({secs:.1f} s)"}


def run_reference(args, w):
    """The oracle as the reference arm: each step is one bounded token slice
    of the workload through the fp64 CPU oracle, on the host cores."""
    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    tokens = max(16, oracle_tokens(w) // max(1, args.steps + args.warmup) * 2)
    tokens = min(tokens, w.tokens)
    inp = W.make_inputs(w.with_(tokens=tokens), seed=0)
    ws = w.with_(tokens=tokens)
    for _ in range(args.warmup):
        oracle_sample(ws, inp, tokens)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_sample(ws, inp, tokens)
    sec = t / args.steps
    flops = ws.flops_fwd_bwd() if w.backward else ws.flops_fwd()
    val = flops / sec / 1e12
    sample = f"{tokens} of {w.tokens} tokens per step, fp64"
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 5),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.tokens, "hidden": w.hidden,
                   "ffn": w.ffn, "shards": w.shards},
        "cpu_baseline": {"value": round(val, 5), "unit": "TFLOP/s",
                         "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(val, 5), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_sweep(args):
    """BLOOM-shaped token x shard sweep: one JSON line per point (not the
    headline; each point times `steps` fwd+bwd steps after `warmup`)."""
    import torch
    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    from tensor_transformer_mlp_tcgen05_gb300.mlp import TensorParallelMLP
    base = W.WORKLOADS[args.workload]
    tmax = max(W.BLOOM_SWEEP_TOKENS)
    inp = W.make_inputs(base.with_(tokens=tmax), seed=0)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    peak_b = _peaks()[0]
    for t in W.BLOOM_SWEEP_SHARDS:
        for T in W.BLOOM_SWEEP_TOKENS:
            w = base.with_(tokens=T, shards=t)
            m = TensorParallelMLP(w.hidden, w.ffn, t, T)
            X, dZ = d["X"][:T], d["dZ"][:T]
            g = {}

            def step():
                m.forward(X, d["A"], d["B"])
                m.backward(dZ, X, d["A"], d["B"], out=g)

            for _ in range(args.warmup):
                step()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                step()
            e1.record()
            torch.cuda.synchronize()
            if m.check() != 0:
                raise RuntimeError("device status in sweep")
            ms = e0.elapsed_time(e1) / args.steps
            tf = w.flops_fwd_bwd() / (ms * 1e-3) / 1e12
            print(json.dumps({"sweep": w.name, "tokens": T, "shards": t,
                              "ms_per_step": round(ms, 4),
                              "value": round(tf, 1), "unit": "TFLOP/s",
                              "frac_of_peak": round(tf / peak_b, 4)}),
                  flush=True)
            m.close()
            del g


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--shards", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--residual", action="store_true",
                    help="time the residual sub-block X + MLP(LN(X))")
    ap.add_argument("--ln-standalone", action="store_true",
                    help="bf16 MLP with LayerNorm: run the LayerNorm as its "
                         "own launch before GEMM1 instead of GEMM1's fused "
                         "prologue")
    ap.add_argument("--fp8", action="store_true",
                    help="time the FP8 (E4M3) forward of an MLP workload")
    ap.add_argument("--train", action="store_true",
                    help="with --fp8: time the FP8 training step (forward "
                         "+ backward) instead")
    ap.add_argument("--sweep", action="store_true",
                    help="token x shard sweep of the workload (one line per "
                         "point) instead of the headline measurement")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from tensor_transformer_mlp_tcgen05_gb300 import workloads as W
    attn = args.workload in W.ATTN_WORKLOADS
    w = (W.ATTN_WORKLOADS if attn else W.WORKLOADS)[args.workload]
    if args.tokens:
        if attn:
            if args.tokens % w.seq:
                ap.error("--tokens must be a multiple of the sequence length")
            w = w.with_(batch=args.tokens // w.seq)
        else:
            w = w.with_(tokens=args.tokens)
    if args.shards:
        w = w.with_(shards=args.shards)
    rank, world, local_rank = dist_info()

    if args.impl == "reference":
        if rank == 0:
            line = run_reference_attn(args, w) if attn else \
                run_reference(args, w)
            print(json.dumps(line), flush=True)
        return 0
    if attn and (args.sweep or args.fp8):
        ap.error("--sweep and --fp8 are for the MLP workloads")
    if args.train and not args.fp8:
        ap.error("--train goes with --fp8 (the bf16 workloads set their "
                 "own pass)")

    if args.sweep:
        from tensor_transformer_mlp_tcgen05_gb300 import build as b
        b.build()
        run_sweep(args)
        return 0

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    from tensor_transformer_mlp_tcgen05_gb300 import build as b
    if rank == 0:
        b.build()
    barrier(world)
    if attn:
        line, inp = run_ours_attn(args, w, rank, world, local_rank)
    elif args.fp8:
        line, inp = run_ours_fp8(args, w, rank, world, local_rank)
    else:
        line, inp = run_ours(args, w, rank, world, local_rank)
    if rank == 0 and not args.no_cpu_baseline:
        if attn:
            line["cpu_baseline"] = run_cpu_baseline_attn(w, inp)
        elif args.fp8:
            line["cpu_baseline"] = run_cpu_baseline_fp8(w, inp, args.train)
        else:
            line["cpu_baseline"] = run_cpu_baseline(w, inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
