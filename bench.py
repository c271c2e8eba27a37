#!/usr/bin/env python3
"""Benchmark of the Mamba-3 scan on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-decode] [--no-cpu-baseline]

One step = one chunked prefill (m3_scan_fwd) over one batch of the workload,
inputs resident in HBM (1.2 GB for the default workload, larger than the
126 MB L2, so no flush is needed between steps).  Prints ONE JSON line with
prefill tokens/s (tokens = batch * seqlen) as the headline, the roofline of
the prefill kernel against the measured HBM copy bandwidth, an end-to-end
figure through host buffers, the oracle timed on the host cores, and the
decode sweep (m3_step, steps/s and GB/s) measured in the same run.

Under torchrun (N > 1) every rank runs its own copy of the workload (the
(batch, head) sequences are independent: weak scaling, no collective on the
data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_131_b300 import inputs  # noqa: E402

HBM_FALLBACK_GBS = 6400.0

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# prefill kernel from one ncu capture, keyed by workload, with the sha256 prefix
# of the kernel source the counters were taken on: reported only while the
# source is unchanged, else null.  Captured at T = 2048 and scaled x4 to
# T = 8192 (traffic grows with the sequence length).
NCU_TRAFFIC = {
    "m3_siso_bf16_b8h32T8192P64N64": {"bytes": 4 * (239.238144e6 + 48.558336e6),
                                      "source": "selective_state_space_131_b300/csrc/scan_ws.cuh",
                                      "sha256": "5570e514627f945e"},
    # decode: one step of the 1024-step sweep (graph replay), per launch
    "decode_f32_b256h32P64N64_R1": {"bytes": 145.839360e6 + 76.878080e6,
                                    "source": "selective_state_space_131_b300/csrc/step_fast.cuh",
                                    "sha256": "c66af4ad5288320a"},
    "decode_f32_b256h32P64N64_R4": {"bytes": 177.312768e6 + 84.965120e6,
                                    "source": "selective_state_space_131_b300/csrc/step_ring.cuh",
                                    "sha256": "8cd37f266fbcedb5"},
}


def ncu_traffic(workload: str):
    import hashlib
    rec = NCU_TRAFFIC.get(workload)
    if rec is None:
        return None
    try:
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return rec["bytes"] if sha.startswith(rec["sha256"]) else None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": HBM_FALLBACK_GBS}, "fallback"


def scan_bytes(shape: inputs.ScanShape) -> int:
    """Algorithmic bytes of one prefill: every input read once, y and the
    final state written once."""
    b, T, H, P, N, R = shape.batch, shape.seqlen, shape.heads, shape.headdim, shape.dstate, shape.rank
    es = 2 if shape.dtype == "bf16" else 4
    tok = b * T * H
    n = tok * R * P * es * 2            # x read, y written
    n += tok * R * N * es * 2           # B, C
    n += tok * 4                        # dt
    n += tok * 4 if shape.with_lambda else 0
    n += tok * (N // 2) * es if shape.with_theta else 0
    n += H * 4                          # A
    n += b * H * N * P * 4              # final state
    return n


def scan_flops(shape: inputs.ScanShape) -> int:
    """The chunked algorithm's flop count per token and head, R [2Q(N+P) + 4NP],
    at the chunk Q the kernel executes (shape.chunk)."""
    b, T, H, P, N, R, Q = (shape.batch, shape.seqlen, shape.heads, shape.headdim, shape.dstate, shape.rank,
                           shape.chunk)
    return b * T * H * R * (2 * Q * (N + P) + 4 * N * P)


def decode_bytes(shape: inputs.DecodeShape) -> int:
    """Algorithmic bytes of one decode step: state read + written, inputs read
    (x, B, C, theta, dt, lambda, prev B, prev x), y written."""
    b, H, P, N, R = shape.batch, shape.heads, shape.headdim, shape.dstate, shape.rank
    es = 2 if shape.dtype == "bf16" else 4
    u = b * H
    return u * (2 * N * P * 4 + R * P * es * 3 + R * N * es * 3 + (N // 2) * es + 8)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        sm = sorted(r[0] for r in rows)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": rows[0][1], "reasons": reasons, "samples": len(rows)}


def rank_seed(seed: int, rank: int) -> int:
    """Input seed of one rank: every rank draws its own copy of the workload
    (independent (batch, head) sequences, weak scaling, no data exchanged)."""
    return seed + 1000 * rank


def max_over_ranks(ms: float, world: int, device="cpu") -> float:
    """The step time the job is charged: the slowest rank's (all_reduce MAX;
    NCCL on the GPU path, gloo on CPU)."""
    if world <= 1:
        return ms
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, ms: float) -> float:
    """Units per second of the whole job: every rank processes units_per_rank in
    the (max-over-ranks) step time."""
    return world * units_per_rank / (ms * 1e-3)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def oracle_sample(shape: inputs.ScanShape, seed: int, units: int):
    """Inputs of `units` sequences (batch row 0, heads 0..units-1) of the workload."""
    inp = inputs.make_scan_inputs(inputs.ScanShape(**{**shape.__dict__, "batch": 1}), seed)
    hs = list(range(min(units, shape.heads)))
    return {k: (None if v is None else (v[hs] if k == "A" else v[:, :, hs])) for k, v in inp.items()}, len(hs)


def time_cpu_oracle(shape: inputs.ScanShape, sample, n_units: int):
    """The fp64 oracle (as it stands) on a sample of sequences: returns
    (tokens/s equivalent, seconds, threads).  A token is one position of one
    batch row across all heads, so `n_units` sequences count n_units/heads."""
    import oracle
    nthreads = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.scan(sample["x"], sample["dt"], sample["A"], sample["B"], sample["C"], sample["lam"],
                sample["theta"], nthreads=nthreads)
    sec = time.perf_counter() - t0
    tokens = shape.seqlen * n_units / shape.heads
    return tokens / sec, sec, nthreads


def run_reference(args, shape, cfg_name):
    """--impl reference: the oracle on the host cores, a bounded sample per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    # size each step's sample so that warm-up + steps fit the wall budget
    full, _ = oracle_sample(shape, inputs.WORKLOAD_SEEDS[args.workload], args.ref_units)
    one = {k: (None if v is None else (v[:1] if k == "A" else v[:, :, :1])) for k, v in full.items()}
    _, sec1, thr = time_cpu_oracle(shape, one, 1)
    n_steps = args.warmup + args.steps
    units = int(max(1, min(args.ref_units, args.ref_budget_s / max(n_steps, 1) / sec1 * thr)))
    sample = {k: (None if v is None else (v[:units] if k == "A" else v[:, :, :units])) for k, v in full.items()}
    vals = []
    for i in range(n_steps):
        tps, sec, thr = time_cpu_oracle(shape, sample, units)
        if i >= args.warmup:
            vals.append((tps, sec))
    tps = sum(v[0] for v in vals) / len(vals)
    sec = sum(v[1] for v in vals) / len(vals)
    sample = f"batch row 0, heads 0..{units - 1} of {cfg_name}, full T={shape.seqlen} (each step)"
    return {
        "impl": "reference", "metric": "prefill_tokens_per_s", "value": tps, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, the pages' distributions)",
        "config": {"workload": cfg_name, **{k: v for k, v in shape.__dict__.items()}},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def decode_k_bytes(shape: inputs.DecodeShape, k: int) -> int:
    """Algorithmic bytes of one k-token decode launch: state read + written
    once, every token's inputs (x, B, C, theta, dt, lambda) read and y written,
    the previous token's B and x read once."""
    b, H, P, N, R = shape.batch, shape.heads, shape.headdim, shape.dstate, shape.rank
    es = 2 if shape.dtype == "bf16" else 4
    u = b * H
    per_tok = R * P * es * 2 + R * N * es * 2 + (N // 2) * es + 8
    return u * (2 * N * P * 4 + k * per_tok + R * (P + N) * es)


def bench_decode_k(m3, stream, steps: int, rank_seed: int, rank: int, k: int):
    """Multi-token decode of the decode workload: `steps` tokens as steps / k
    m3_step_k launches of k tokens each (the state read and written once per
    launch), captured in one CUDA graph and replayed on `stream`."""
    launches = steps // k
    shape = inputs.DecodeShape(**{**inputs.WORKLOADS[inputs.DECODE].__dict__, "steps": launches * k, "rank": rank})
    dec = inputs.make_decode_inputs(shape, 4 + rank_seed, device="cuda")
    b, H = shape.batch, shape.heads
    lay = lambda a: a[1:].reshape(launches, k, b, H, *a.shape[3:]).transpose(1, 2).contiguous()
    X, DT, Bm, Cm, LAM, TH = (lay(dec[key]) for key in ("x", "dt", "B", "C", "lam", "theta"))
    A, B0, X0 = dec["A"], dec["B"][0], dec["x"][0]
    state = dec["state0"].clone()
    del dec
    Y = torch.empty_like(X)
    dims = m3.scan_dims(X[0], Bm[0], 64)

    # the previous-token slices are gathered once, outside the timed graph
    prevs = [(B0, X0)] + [(Bm[i - 1][:, k - 1].contiguous(), X[i - 1][:, k - 1].contiguous())
                          for i in range(1, launches)]

    def sweep_pre():
        for i in range(launches):
            m3.m3_step_k(state, X[i], DT[i], A, Bm[i], Cm[i], LAM[i], TH[i], prevs[i][0], prevs[i][1], Y[i],
                         stream=stream, dims=dims)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        sweep_pre()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sweep_pre()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if m3.m3_device_status(stream) != m3.M3_OK:
        raise RuntimeError("device status set during the multi-token decode sweep")
    ms = e0.elapsed_time(e1) / (reps * launches)
    nbytes = decode_k_bytes(shape, k)
    del X, DT, Bm, Cm, LAM, TH, Y, state, g, prevs
    torch.cuda.empty_cache()
    return {"workload": inputs.DECODE + f"_R{rank}_k{k}", "tokens_per_launch": k,
            "us_per_launch": ms * 1e3, "tokens_per_s": b * k * 1e3 / ms, "GB_per_s": nbytes / (ms * 1e-3) / 1e9,
            "bytes_per_launch": nbytes, "graph_launches": launches, "entry": "m3_step_k"}


def bench_decode(m3, stream, steps: int, rank_seed: int, rank: int = 1):
    """Decode sweep of the decode workload (fp32, b256 h32 P64 N64, rank R):
    `steps` consecutive m3_step calls captured in one CUDA graph and replayed
    on `stream` (the stream the events are recorded on); returns a dict."""
    shape = inputs.DecodeShape(**{**inputs.WORKLOADS[inputs.DECODE].__dict__, "steps": steps, "rank": rank})
    inp = inputs.make_decode_inputs(shape, 4 + rank_seed, device="cuda")
    state = inp["state0"].clone()
    ys = torch.empty_like(inp["x"][1:])
    dims = m3.step_dims(inp["x"][0], inp["B"][0])

    def sweep():
        for s in range(steps):
            m3.m3_step(state, inp["x"][s + 1], inp["dt"][s + 1], inp["A"], inp["B"][s + 1], inp["C"][s + 1],
                       inp["lam"][s + 1], inp["theta"][s + 1], inp["B"][s], inp["x"][s], ys[s], stream=stream,
                       dims=dims)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        sweep()                      # warm-up (also the first sweep of the state)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sweep()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3
    with torch.cuda.stream(stream):
        g.replay()                   # warm replay
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if m3.m3_device_status(stream) != m3.M3_OK:
        raise RuntimeError("device status set during the decode sweep")
    ms = e0.elapsed_time(e1) / (reps * steps)
    nbytes = decode_bytes(shape)
    del inp, ys, state, g
    torch.cuda.empty_cache()
    return {"workload": inputs.DECODE + f"_R{rank}", "steps_per_s": 1e3 / ms, "us_per_step": ms * 1e3,
            "tokens_per_s": shape.batch * 1e3 / ms, "GB_per_s": nbytes / (ms * 1e-3) / 1e9,
            "bytes_per_step": nbytes, "graph_steps": steps, "launches_per_step": 1}


def time_prefill(m3, stream, shape, seed, dev, steps, warmup, bcnorm=False):
    """Device time (ms) of one prefill of `shape` on resident inputs, CUDA
    events on `stream` around `steps` back-to-back launches (with bcnorm: the
    entry point with the B / C normalisation fused into the prologue)."""
    inp = inputs.make_scan_inputs(shape, seed)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    nd = {k: v.to(dev) for k, v in inputs.make_bcnorm_params(shape.dstate, shape.heads, seed).items()}
    b, T, H, R, P = d["x"].shape
    y = torch.empty_like(d["x"])
    fs = torch.empty(b, H, d["B"].shape[-1], P, device=dev, dtype=torch.float32)
    dims = m3.scan_dims(d["x"], d["B"], shape.chunk)

    def launch():
        if bcnorm:
            m3.m3_scan_fwd_bcnorm(d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], nd["norm_B"],
                                  nd["norm_C"], nd["bias_B"], nd["bias_C"], 1e-6, y, fs, stream=stream, dims=dims)
        else:
            m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], y, fs, stream=stream,
                           dims=dims)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            launch()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            launch()
        e1.record(stream)
    torch.cuda.synchronize()
    if m3.m3_device_status(stream) != m3.M3_OK:
        raise RuntimeError("device status set")
    ms = e0.elapsed_time(e1) / steps
    del d, y, fs
    torch.cuda.empty_cache()
    return ms


def bwd_bytes(shape: inputs.ScanShape) -> int:
    """Algorithmic bytes of one backward pass: the forward's inputs, dy and
    dfinal read once; dx, ddt, dA, dB, dC, dlambda, dtheta written once (the
    workspace of chunk states excluded)."""
    b, T, H, P, N, R = shape.batch, shape.seqlen, shape.heads, shape.headdim, shape.dstate, shape.rank
    es = 2 if shape.dtype == "bf16" else 4
    tok = b * T * H
    per_tok = R * P * es * 2 + R * N * es * 2 + 4 + (4 if shape.with_lambda else 0) + \
        ((N // 2) * es if shape.with_theta else 0)
    n = tok * per_tok * 2           # inputs and their gradients
    n += tok * R * P * es           # dy
    n += b * H * N * P * 4          # dfinal
    n += H * 4 * 2                  # A, dA
    return n


def time_bwd(m3, stream, shape, seed, dev, steps, warmup):
    """Device time (ms) of one m3_scan_bwd of `shape` on resident inputs (CUDA
    events on `stream`), with its workspace bytes."""
    inp = inputs.make_scan_inputs(shape, seed)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    b, T, H, R, P = d["x"].shape
    N = d["B"].shape[-1]
    dy = torch.randn(b, T, H, R, P, generator=g).to(d["x"].dtype).to(dev)
    dfinal = torch.randn(b, H, N, P, generator=g).to(dev)
    dims = m3.scan_dims(d["x"], d["B"], shape.chunk)
    wsb = m3.m3_scan_bwd_workspace_size(dims)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    out = [torch.empty_like(d["x"]), torch.empty_like(d["dt"]), torch.empty_like(d["A"]), torch.empty_like(d["B"]),
           torch.empty_like(d["C"]), torch.empty_like(d["dt"]) if d["lam"] is not None else None,
           torch.empty_like(d["theta"]) if d["theta"] is not None else None]

    def launch():
        m3.m3_scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], dy, dfinal, *out, ws, wsb,
                       stream=stream, dims=dims)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            launch()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            launch()
        e1.record(stream)
    torch.cuda.synchronize()
    if m3.m3_device_status(stream) != m3.M3_OK:
        raise RuntimeError("device status set during the backward")
    ms = e0.elapsed_time(e1) / steps
    del d, dy, dfinal, ws, out
    torch.cuda.empty_cache()
    return ms, wsb


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=inputs.SISO, choices=list(inputs.PREFILL_WORKLOADS))
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-units", type=int, default=32, help="sequences in the oracle sample (cpu_baseline)")
    ap.add_argument("--ref-budget-s", type=float, default=150.0, help="wall budget of the reference arm")
    ap.add_argument("--decode-steps", type=int, default=1024)
    ap.add_argument("--decode-k", type=int, default=8, help="tokens per m3_step_k launch")
    ap.add_argument("--cpu-rows", type=int, default=8, help="batch rows in the oracle's cpu_baseline sample")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="wall time the cpu_baseline repeats for")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling captures)")
    ap.add_argument("--seqlen", type=int, default=0, help="override the workload's seqlen (profiling captures)")
    ap.add_argument("--chunk", type=int, default=0, help="override the workload's chunk (profiling captures)")
    ap.add_argument("--no-other", action="store_true", help="skip the other prefill workloads")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward pass")
    ap.add_argument("--decode-only", action="store_true", help="only the decode sweep (profiling captures)")
    args = ap.parse_args()

    shape = inputs.WORKLOADS[args.workload]
    wseed = inputs.WORKLOAD_SEEDS[args.workload]
    if args.batch or args.seqlen or args.chunk:
        shape = inputs.ScanShape(**{**shape.__dict__, "batch": args.batch or shape.batch,
                                    "seqlen": args.seqlen or shape.seqlen, "chunk": args.chunk or shape.chunk})
    cfg_name = args.workload
    world, rank, local = dist_env()

    if args.impl == "reference":
        out = run_reference(args, shape, cfg_name)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    from selective_state_space_131_b300 import m3scan as m3
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.Stream()
    if args.decode_only:
        for r in (1, 4):
            print(json.dumps(bench_decode(m3, stream, args.decode_steps, rank, rank=r)), flush=True)
            print(json.dumps(bench_decode_k(m3, stream, args.decode_steps, rank, rank=r, k=args.decode_k)),
                  flush=True)
        return 0

    inp = inputs.make_scan_inputs(shape, rank_seed(wseed, rank))
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    b, T, H, R, P = d["x"].shape
    N = d["B"].shape[-1]
    y = torch.empty_like(d["x"])
    fs = torch.empty(b, H, N, P, device=dev, dtype=torch.float32)
    dims = m3.scan_dims(d["x"], d["B"], shape.chunk)
    algo = m3.m3_scan_algorithm(dims)

    def step():
        m3.m3_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["lam"], d["theta"], y, fs, stream=stream,
                       dims=dims)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    torch.cuda.synchronize()
    if m3.m3_device_status(stream) != m3.M3_OK:
        raise RuntimeError("device status set during warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    if m3.m3_device_status(stream) != m3.M3_OK:
        raise RuntimeError("device status set during the timed region")

    tokens = b * T
    value = whole_job_rate(tokens, world, ms)
    peaks, peak_kind = measured_peaks()
    nbytes = scan_bytes(shape)
    achieved = nbytes / (ms * 1e-3) / 1e9
    result = {
        "metric": "prefill_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if shape.dtype == "bf16" else "f32",
        "data": "synthetic (seeded, the pages' input distributions; no dataset)",
        "config": {"workload": cfg_name, "batch": b, "seqlen": T, "heads": H, "headdim": P, "dstate": N,
                   "rank": R, "chunk": shape.chunk, "lambda": shape.with_lambda, "theta": shape.with_theta,
                   "l2": "inputs (%.2f GB) larger than L2; no flush" % (nbytes / 1e9),
                   "algorithm": {0: "sequential_simt", 1: "chunked_tcgen05"}.get(algo, str(algo)),
                   "parallelism": f"weak x{world} (independent sequences per rank)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": (ncu_traffic(cfg_name) if not (args.batch or args.seqlen) else None),
                     "peak_kind": f"{peak_kind} HBM copy bandwidth", "algorithmic_bytes": nbytes,
                     "tensor_tflops": scan_flops(shape) / (ms * 1e-3) / 1e12},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }

    if not args.no_e2e:
        # end to end through the public API with host buffers: m3_scan_fwd_host takes
        # the step's inputs in pinned host memory and returns y and the final state
        # there; it copies them in and out in batch slices, overlapping the copies
        # with the scans (the timed region holds every copy of the step).
        host = {k: (v.pin_memory() if v is not None else None) for k, v in inp.items()}
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        fs_host = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = y_host.numel() * y_host.element_size() + fs_host.numel() * fs_host.element_size()
        e_steps = max(3, min(20, args.steps // 20))
        hdims = m3.scan_dims(host["x"], host["B"], shape.chunk)
        e_slice = 0   # the library's default: an eighth of the batch per slice
        hwsb = m3.m3_scan_fwd_host_workspace_size(hdims, e_slice)
        hws = torch.empty(hwsb, dtype=torch.uint8, device=dev)

        def e2e_step():
            m3.m3_scan_fwd_host(host["x"], host["dt"], host["A"], host["B"], host["C"], host["lam"], host["theta"],
                                y_host, fs_host, hws, hwsb, slice=e_slice, stream=stream, dims=hdims)
        e2e_step()
        torch.cuda.synchronize()
        barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        a1.record(stream)
        barrier()
        ems = a0.elapsed_time(a1) / e_steps
        ems = max_over_ranks(ems, world, dev)
        result["e2e"] = {"value": whole_job_rate(tokens, world, ems), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                         "d2h_bytes_per_step": d2h, "ms_per_step": ems, "steps": e_steps,
                         "entry": "m3_scan_fwd_host", "slice_rows": (b + 7) // 8 if e_slice == 0 else e_slice}
        del hws

    del d, y, fs
    torch.cuda.empty_cache()
    if not args.no_other and rank == 0:
        # the other prefill workloads, same protocol (reported beside the headline)
        other = {}
        for w in inputs.PREFILL_WORKLOADS:
            if w == args.workload:
                continue
            sh = inputs.WORKLOADS[w]
            note = None
            if sh.chunk * sh.rank != 64:
                # the tensor-core kernel's chunk is one 64-row tile: 64 / R tokens (16 at
                # R = 4); the workload's own chunk runs on the chunked CUDA-core kernel
                note = (f"chunk {64 // sh.rank} executed (the 64-row tensor-core tile at R = {sh.rank}); "
                        f"chunk {sh.chunk} runs on the CUDA-core chunked kernel")
                sh = inputs.ScanShape(**{**sh.__dict__, "chunk": 64 // sh.rank})
            wms = time_prefill(m3, stream, sh, inputs.WORKLOAD_SEEDS[w], dev, steps=20, warmup=3)
            wb = scan_bytes(sh)
            other[w] = {
                "ms_per_step": wms, "tokens_per_s": sh.batch * sh.seqlen / (wms * 1e-3),
                "GB_per_s": wb / (wms * 1e-3) / 1e9, "hbm_frac": wb / (wms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "algorithmic_bytes": wb, "chunk": sh.chunk,
                "tensor_tflops": scan_flops(sh) / (wms * 1e-3) / 1e12}
            if note:
                other[w]["note"] = note
        # the timed workload again with the B / C normalisation and biases fused
        # into the prologue (m3_scan_fwd_bcnorm; the parameters add 1 KB per head)
        wms = time_prefill(m3, stream, shape, wseed, dev, steps=20, warmup=3, bcnorm=True)
        wb = scan_bytes(shape)
        other[args.workload + "_bcnorm"] = {
            "ms_per_step": wms, "tokens_per_s": shape.batch * shape.seqlen / (wms * 1e-3),
            "GB_per_s": wb / (wms * 1e-3) / 1e9, "hbm_frac": wb / (wms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "algorithmic_bytes": wb}
        result["other_prefill"] = other

    if not args.no_bwd and rank == 0:
        # the backward pass of the timed workload (training): m3_scan_bwd
        bms, wsb = time_bwd(m3, stream, shape, wseed, dev, steps=10, warmup=3)
        bb = bwd_bytes(shape)
        result["backward"] = {
            "workload": cfg_name, "entry": "m3_scan_bwd", "ms_per_step": bms,
            "tokens_per_s": shape.batch * shape.seqlen / (bms * 1e-3), "GB_per_s": bb / (bms * 1e-3) / 1e9,
            "hbm_frac": bb / (bms * 1e-3) / 1e9 / peaks["hbm_gbs"], "algorithmic_bytes": bb,
            "workspace_bytes": wsb, "launches_per_step": 3,
            "vs_forward": bms / ms}

    if not args.no_decode and rank == 0:
        dec = {}
        for r in (1, 4):
            dr = bench_decode(m3, stream, args.decode_steps, rank, rank=r)
            dr["roofline_frac"] = dr["GB_per_s"] / peaks["hbm_gbs"]
            dr["traffic"] = ncu_traffic(dr["workload"])
            if dr["traffic"]:
                dr["dram_GB_per_s"] = dr["traffic"] / (dr["us_per_step"] * 1e-6) / 1e9
                dr["dram_frac"] = dr["dram_GB_per_s"] / peaks["hbm_gbs"]
            dec[f"R{r}"] = dr
        for r in (1, 4):
            dk = bench_decode_k(m3, stream, args.decode_steps, rank, rank=r, k=args.decode_k)
            dk["roofline_frac"] = dk["GB_per_s"] / peaks["hbm_gbs"]
            dk["tokens_per_s_vs_single_step"] = dk["tokens_per_s"] / dec[f"R{r}"]["tokens_per_s"]
            dec[f"R{r}_k{args.decode_k}"] = dk
        result["decode"] = dec

    if not args.no_cpu_baseline and rank == 0:
        # the oracle on every host core: the workload's first batch rows (all
        # heads, full T), repeated until about args.cpu_seconds of wall time
        import oracle
        full = inputs.make_scan_inputs(shape, wseed)
        rows = max(1, min(shape.batch, args.cpu_rows))
        sample = {k: (None if v is None else (v if k == "A" else v[:rows].contiguous())) for k, v in full.items()}
        del full
        nthreads = oracle.max_threads()
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.scan(sample["x"], sample["dt"], sample["A"], sample["B"], sample["C"], sample["lam"],
                        sample["theta"], nthreads=nthreads)
            reps += 1
            if time.perf_counter() - t0 >= args.cpu_seconds:
                break
        sec = (time.perf_counter() - t0) / reps
        result["cpu_baseline"] = {"value": rows * T / sec, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
                                  "sample": f"batch rows 0..{rows - 1} x all {H} heads x full T={T} of the workload, "
                                            f"{reps} repetition(s), {sec:.2f} s each"}

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
