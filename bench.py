"""Benchmark of the tensor-parallel MLP forward on GB300.

One step = one pass over every forward row of the hot path on the large
workload (T=16384 tokens, D=4096, F=16384, N=8 shards, bf16 operands, fp32
accumulation), with inputs resident in HBM:
    faithful:  H_i = GeLU(X A_i) -> Y_i = H_i B_i -> Y = sum_i Y_i (shard order)
    fused:     H_i = GeLU(X A_i) -> Y = sum_i H_i B_i accumulated on chip
i.e. 2 x 4*T*D*F FLOP. `value` is TFLOP/s over the whole step. Every kernel
is timed with CUDA events on the stream it is launched on.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tpmlp|reference]

--impl reference times the float64 CPU oracle on a bounded sample of the same
workload (host cores). With N > 1 (torchrun), every rank runs its own replica
(the path has no cross-GPU step here) and rank 0 prints one JSON line.
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

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM bytes (read + write) per launch of each kernel of the step on the large
# workload, from one ncu capture of dram__bytes_read.sum + dram__bytes_write.sum
# (one kernel per capture on a reduced token count, scaled to the full launch
# by the tokens it processes; the capture commands are kept with the profiles).
# Valid only for the CUDA sources they were measured on: TRAFFIC_SOURCE_HASH is
# source_hash() of those sources, and a different hash reports null.
TRAFFIC_SOURCE_HASH = "e1d2deb19b01e774"
TRAFFIC_BYTES = {
    "gemm1_gelu(faithful)": 1_231_000_000,
    "gemm2_partials": 3_021_000_000,
    "allreduce": 2_392_000_000,
    "gemm1_gelu(fused)": 1_231_000_000,
    "gemm2_fused_sum": 2_637_000_000,
}


# The sources of the step's kernels and of their launch parameters.
STEP_SOURCES = ["api.cu", "device.cuh", "elementwise.cu", "gemm_common.cuh", "gemm_pair.cu", "gemm_tc.cu", "internal.h"]


def source_hash() -> str:
    import hashlib

    d = os.path.join(ROOT, "tensor_transformer_mlp_column_gb300", "csrc")
    h = hashlib.sha256()
    for f in STEP_SOURCES:
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(kernel: str):
    if source_hash() != TRAFFIC_SOURCE_HASH:
        return None
    return TRAFFIC_BYTES.get(kernel)


METRIC = "TP-MLP fwd TFLOP/s on 1 GB300 (% BF16 peak); partial-sum reduce GB/s (% HBM)"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            hbm = float(d.get("hbm_gbs") or d.get("hbm_GBps") or 0)
            bf = float(d.get("bf16_tflops") or 0)
            bfs = float(d.get("bf16_tflops_sustained") or bf or 0)
            if hbm > 0 and bf > 0:
                return {"hbm_gbs": hbm, "bf16_tflops": bf, "bf16_tflops_sustained": bfs, "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return summarize_clocks(self.lines, getattr(self, "t_begin", 0.0), getattr(self, "t_end", 1e30))


def summarize_clocks(lines, t0: float, t1: float) -> dict:
    """Median and maximum SM clock and the throttle reasons seen in the
    nvidia-smi samples (time, csv line of ClockSampler.FIELDS) taken during
    the timed region [t0, t1] (plus one sampling period)."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ts, ln in lines:
        if not (t0 <= ts <= t1 + 0.15):
            continue
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        for nm, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(nm)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle baseline

def _oracle_worker(target_s: float, reps: int, out_path: str):
    """Runs in a fresh interpreter: times the float64 oracle on token-row samples.

    Inputs are generated once (seeded like the large workload); a 16-row call
    calibrates the rate, then `reps` calls each on as many rows as take about
    target_s seconds are timed.
    """
    import numpy as np
    import torch

    import oracle
    from tpmlp_inputs import WORKLOADS, make_inputs

    w = WORKLOADS["large"]
    inp = make_inputs(w, seed=0)
    X = inp["X"].to(torch.float64).numpy()
    shards = oracle.shard_mlp(inp["A"].to(torch.float64).numpy(), inp["B"].to(torch.float64).numpy(), w.N)
    t0 = time.perf_counter()
    oracle.tp_mlp_rows(X, shards, list(range(16)))
    per_row = (time.perf_counter() - t0) / 16
    rows = int(max(16, min(w.T, target_s / max(per_row, 1e-9))))
    times, check = [], 0.0
    for r in range(reps):
        sel = list(range((r * rows) % (w.T - rows + 1), (r * rows) % (w.T - rows + 1) + rows))
        t0 = time.perf_counter()
        Y = oracle.tp_mlp_rows(X, shards, sel)
        times.append(time.perf_counter() - t0)
        check += float(np.sum(Y))
    json.dump({"seconds": times, "rows": rows, "checksum": check}, open(out_path, "w"))


def _oracle_rows_worker(out_path: str):
    """Runs in a fresh interpreter: the oracle of the block and of attention on
    bounded samples (a few seconds each), for the rows beside the MLP."""
    import torch

    import oracle
    from tpmlp_inputs import ATTN_WORKLOADS, WORKLOADS, make_attn_inputs, make_block_inputs

    res = {}
    w = WORKLOADS["large"]
    inp = make_block_inputs(w, seed=0)
    x = inp["x"][:1024].to(torch.float64).numpy()
    shards = oracle.shard_mlp(inp["A"].to(torch.float64).numpy(), inp["B"].to(torch.float64).numpy(), w.N)
    del inp
    t0 = time.perf_counter()
    oracle.block_mlp(x, shards)
    res["block"] = {"seconds": time.perf_counter() - t0, "rows": 1024}
    del shards
    a = ATTN_WORKLOADS["attn_seq512"]
    ai = make_attn_inputs(a, seed=0)
    f = {k: v.to(torch.float64).numpy() for k, v in ai.items()}
    ash = oracle.shard_attention(f["Wq"], f["Wk"], f["Wv"], f["Wo"], a.heads, a.N)
    t0 = time.perf_counter()
    oracle.tp_attention(f["X"], a.batch, ash, a.heads)
    res["attention"] = {"seconds": time.perf_counter() - t0, "sequences": a.batch}
    json.dump(res, open(out_path, "w"))


def run_oracle(target_s: float, reps: int, cores: int) -> dict:
    out = os.path.join("/tmp", f"tpmlp_oracle_{os.getpid()}.json")
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = f"import bench; bench._oracle_worker({target_s}, {reps}, {out!r})"
    subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, check=True)
    r = json.load(open(out))
    os.remove(out)
    return r


def cpu_baseline(target_s: float = 12.0) -> dict:
    """The oracle as it stands on a bounded sample (token rows of the large workload)."""
    from tpmlp_inputs import WORKLOADS

    w = WORKLOADS["large"]
    cores = len(os.sched_getaffinity(0))
    r = run_oracle(target_s, 1, cores)
    flops = 4.0 * r["rows"] * w.D * w.F
    out = {"value": flops / r["seconds"][0] / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
           "sample": f"{r['rows']} of {w.T} token rows of the large workload, one float64 forward "
                     f"(numpy, {r['seconds'][0]:.1f} s)"}
    # The block's FFN half and head-split attention, timed the same way on small samples.
    path = os.path.join("/tmp", f"tpmlp_oracle_rows_{os.getpid()}.json")
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    subprocess.run([sys.executable, "-c", f"import bench; bench._oracle_rows_worker({path!r})"], cwd=ROOT, env=env,
                   check=True)
    rr = json.load(open(path))
    os.remove(path)
    from tpmlp_inputs import ATTN_WORKLOADS

    a = ATTN_WORKLOADS["attn_seq512"]
    per_seq_flops = a.fwd_flops() / a.batch
    out["rows"] = {
        "block": {"value": round(4.0 * rr["block"]["rows"] * w.D * w.F / rr["block"]["seconds"] / 1e12, 4),
                  "unit": "TFLOP/s", "sample": f"{rr['block']['rows']} token rows of the large workload "
                                               f"({rr['block']['seconds']:.1f} s)"},
        "attention": {"value": round(rr["attention"]["sequences"] * per_seq_flops / rr["attention"]["seconds"] / 1e12,
                                     4),
                      "unit": "TFLOP/s", "sample": f"the seq-512 attention workload, {rr['attention']['sequences']} "
                                                   f"sequences ({rr['attention']['seconds']:.1f} s)"},
    }
    return out


# ------------------------------------------------------------------ GPU arm

def bench_tpmlp(args, rank, world, local_rank):
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import tensor_transformer_mlp_column_gb300 as tp
    from tpmlp_inputs import WORKLOADS, make_inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    if args.T:
        w = w.with_(T=args.T)
    if args.N:
        w = w.with_(N=args.N)
    inp = make_inputs(w, seed=rank)
    X = inp["X"].to(dev)
    A = inp["A"].to(dev)
    B = inp["B"].to(dev)
    sh = tp.tpmlp_shard(A, B, w.N)
    del A, B
    T, D, F, N, Fs = w.T, w.D, w.F, w.N, w.Fs
    H = torch.empty((N, T, Fs), dtype=w.torch_dtype, device=dev)
    Yp = torch.empty((N, T, D), dtype=torch.float32, device=dev)
    Y1 = torch.empty((T, D), dtype=torch.float32, device=dev)
    Y2 = torch.empty((T, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    kernels = ["gemm1_gelu(faithful)", "gemm2_partials", "allreduce", "gemm1_gelu(fused)", "gemm2_fused_sum"]

    def step(evs=None):
        def mark(i):
            if evs is not None:
                evs[i].record(stream)
        mark(0)
        tp.tpmlp_hidden(X, sh, H)
        mark(1)
        tp.tpmlp_partials(H, sh, Yp)
        mark(2)
        tp.tpmlp_allreduce(Yp, Y1)
        mark(3)
        tp.tpmlp_hidden(X, sh, H)
        mark(4)
        tp.tpmlp_fused_sum(H, sh, Y2)
        mark(5)

    clocks = ClockSampler(local_rank)
    clocks.start()  # before the warm-up, so its start-up does not overlap the timed region
    for _ in range(args.warmup):
        step()
    tp.tpmlp_check_status(stream)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark("t_begin")
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(events[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark("t_end")
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    tp.tpmlp_check_status(stream)
    total_ms = t0.elapsed_time(t1)
    per_kernel = {name: [] for name in kernels}
    for evs in events:
        for i, name in enumerate(kernels):
            per_kernel[name].append(evs[i].elapsed_time(evs[i + 1]))
    avg = {k: sum(v) / len(v) for k, v in per_kernel.items()}

    # ---- end to end through the public API, host buffers, copies inside the timed region.
    # Every step uploads its input X from pinned host memory, runs tpmlp_forward in
    # both modes and downloads both results. The copies run on their own streams
    # with double-buffered device tensors, so step k+1's upload and step k's
    # downloads overlap the compute of the neighbouring steps.
    del H, Yp, Y1, Y2
    Xh = inp["X"].pin_memory()
    Yh1 = [torch.empty((T, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    Yh2 = [torch.empty((T, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    Xd = [torch.empty_like(X) for _ in range(2)]
    Yd1 = [torch.empty((T, D), dtype=torch.float32, device=dev) for _ in range(2)]
    Yd2 = [torch.empty((T, D), dtype=torch.float32, device=dev) for _ in range(2)]
    ws_f = torch.empty(tp.tpmlp_workspace_bytes(T, sh, "faithful"), dtype=torch.uint8, device=dev)
    ws_u = torch.empty(tp.tpmlp_workspace_bytes(T, sh, "fused"), dtype=torch.uint8, device=dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, in_free, y1_ready, y2_ready, out_free = ([ev(), ev()] for _ in range(5))

    def e2e_step(k):
        b = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(in_free[b])  # step k-2 has finished reading Xd[b]
            Xd[b].copy_(Xh, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        if k >= 2:
            stream.wait_event(out_free[b])  # step k-2's results have been downloaded
        tp.tpmlp_forward(Xd[b], sh, "faithful", Yd1[b], ws_f, stream)
        y1_ready[b].record(stream)
        tp.tpmlp_forward(Xd[b], sh, "fused", Yd2[b], ws_u, stream)
        y2_ready[b].record(stream)
        in_free[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(y1_ready[b])
            Yh1[b].copy_(Yd1[b], non_blocking=True)
            s_out.wait_event(y2_ready[b])
            Yh2[b].copy_(Yd2[b], non_blocking=True)
            out_free[b].record(s_out)

    for k in range(max(2, min(args.warmup, 3))):
        e2e_step(k)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(2, min(args.steps, 20))
    e0.record(s_in)  # before the first upload
    for k in range(e2e_steps):
        e2e_step(k)
    e1.record(s_out)  # after the last download
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    tp.tpmlp_check_status(stream)
    Yh1, Yh2 = Yh1[0], Yh2[0]

    res = {
        "total_ms": total_ms, "avg": avg, "clocks": clk, "e2e_ms": e2e_ms,
        "h2d": Xh.numel() * Xh.element_size(), "d2h": 2 * Yh1.numel() * 4,
        "launches": 5 * args.steps,
    }
    sh.free()
    return res


def max_over_ranks(values, device):
    """Element-wise MAX of `values` over all ranks of the process group: the
    slowest replica sets the job's time."""
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world: int, flops_per_step_per_rank: float, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank's work divided by the slowest rank's time."""
    return world * flops_per_step_per_rank / (ms_per_step * 1e-3) / 1e12


def bench_gelu(local_rank, peaks):
    """tpmlp_gelu on 1 GiB of input (bf16 and fp32): 2 * n * sizeof(elt) bytes per call."""
    import torch

    import tensor_transformer_mlp_column_gb300 as tp

    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for dt, name in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
        n = (1 << 30) // torch.tensor([], dtype=dt).element_size()
        x = torch.randn(n, device=dev, dtype=torch.float32).to(dt)
        y = torch.empty_like(x)
        for _ in range(3):
            tp.tpmlp_gelu(x, y)
        reps = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            tp.tpmlp_gelu(x, y)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / reps
        gbs = 2.0 * n * x.element_size() / (ms * 1e-3) / 1e9
        out[name] = {"elements": n, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        del x, y
    return out


def bench_small_workloads(local_rank, only=None):
    """Forward time of the GPT-2-small and the sequence-sweep workloads (both
    modes), and the linear fit of forward time against seq for the sweep
    (`only`: that one workload alone, no fit)."""
    import torch

    import tensor_transformer_mlp_column_gb300 as tp
    from tpmlp_inputs import WORKLOADS, make_inputs

    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name in (only,) if only else ("gpt2_small", "seq128", "seq256", "seq512"):
        w = WORKLOADS[name]
        inp = make_inputs(w, seed=0)
        X = inp["X"].to(dev)
        sh = tp.tpmlp_shard(inp["A"].to(dev), inp["B"].to(dev), w.N)
        Y = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
        res = {"T": w.T, "D": w.D, "F": w.F, "N": w.N}
        for mode in ("faithful", "fused"):
            ws = torch.empty(tp.tpmlp_workspace_bytes(w.T, sh, mode), dtype=torch.uint8, device=dev)
            for _ in range(5):
                tp.tpmlp_forward(X, sh, mode, Y, ws)
            reps = 50
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for _ in range(reps):
                tp.tpmlp_forward(X, sh, mode, Y, ws)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / reps
            gms = _time_graph_ms(lambda: tp.tpmlp_forward(X, sh, mode, Y, ws), dev, reps)
            res[mode] = {"ms": round(ms, 4), "TFLOP/s": round(w.fwd_flops() / (ms * 1e-3) / 1e12, 1),
                         "graph_ms": round(gms, 4), "graph_TFLOP/s": round(w.fwd_flops() / (gms * 1e-3) / 1e12, 1)}
        tp.tpmlp_check_status(stream)
        sh.free()
        out[name] = res
    if only:
        return out
    # FFN time against sequence length (batch 8): a least-squares line and its R^2.
    seqs = [128, 256, 512]
    for mode in ("faithful", "fused"):
        ys = [out[f"seq{s}"][mode]["ms"] for s in seqs]
        mx, my = sum(seqs) / 3, sum(ys) / 3
        sxy = sum((x - mx) * (y - my) for x, y in zip(seqs, ys))
        sxx = sum((x - mx) ** 2 for x in seqs)
        slope = sxy / sxx
        ss_res = sum((y - (my + slope * (x - mx))) ** 2 for x, y in zip(seqs, ys))
        ss_tot = sum((y - my) ** 2 for y in ys)
        out[f"seq_sweep_{mode}"] = {"ms_per_unit_seq": round(slope, 6), "intercept_ms": round(my - slope * mx, 4),
                                    "r2": round(1 - ss_res / ss_tot, 5) if ss_tot > 0 else None}
    return out


def bench_backward(args, local_rank, peaks):
    """tpmlp_backward on the fwd+bwd workload (T=8192, D=8192, F=32768, N=8):
    8*T*D*F algorithmic FLOP (plus 2*T*D*F to recompute P = X A_i)."""
    import torch

    import tensor_transformer_mlp_column_gb300 as tp
    from tpmlp_inputs import WORKLOADS, make_inputs

    dev = torch.device("cuda", local_rank)
    w = WORKLOADS["fwd_bwd"]
    if args.T:  # a smaller profiling case of the same shapes
        w = w.with_(T=args.T)
    inp = make_inputs(w, seed=0)
    X, dY = inp["X"].to(dev), inp["dY"].to(dev)
    sh = tp.tpmlp_shard(inp["A"].to(dev), inp["B"].to(dev), w.N)
    del inp
    stream = torch.cuda.current_stream(dev)
    out = {"workload": f"{w.name}: T={w.T} D={w.D} F={w.F} N={w.N} bf16"}
    dX = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
    dA = [torch.empty((w.D, w.Fs), dtype=torch.float32, device=dev) for _ in range(w.N)]
    dB = [torch.empty((w.Fs, w.D), dtype=torch.float32, device=dev) for _ in range(w.N)]
    # Pre-activations saved by a training-mode forward, for the saved-P backward.
    _, P = tp.tpmlp_forward_save(X, sh, "fused")
    for mode, saved in (("faithful", False), ("fused", False), ("faithful", True), ("fused", True)):
        ws = torch.empty(tp.tpmlp_workspace_bytes(w.T, sh, mode, 2 if saved else 1), dtype=torch.uint8, device=dev)

        def run():
            tp.tpmlp_backward(X, dY, sh, mode, dX, dA, dB, ws, P=P if saved else None)

        for _ in range(3):
            run()
        tp.tpmlp_check_status(stream)
        reps = max(3, min(args.steps // 10, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        tp.tpmlp_check_status(stream)
        ms = e0.elapsed_time(e1) / reps
        alg = 8.0 * w.T * w.D * w.F / (ms * 1e-3) / 1e12
        if saved:  # no recompute: all 8*T*D*F FLOP are algorithmic
            out[f"saved_P_{mode}"] = {"ms": round(ms, 3), "TFLOP/s": round(alg, 1),
                                      "frac_bf16": round(alg / peaks["bf16_tflops"], 4)}
        else:
            out[mode] = {"ms": round(ms, 3), "TFLOP/s": round(alg, 1),
                         "TFLOP/s_incl_recompute": round(alg * 10 / 8, 1),
                         "frac_bf16_incl_recompute": round(alg * 10 / 8 / peaks["bf16_tflops"], 4)}
        del ws
    sh.free()
    return out


def _time_ms(fn, dev, stream, reps: int, warm: int = 3) -> float:
    import torch

    for _ in range(warm):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def _time_graph_ms(fn, dev, reps: int) -> float:
    """Mean device time of fn replayed from a CUDA graph of `reps` calls (the
    library's calls only enqueue work, so they capture as they are); the
    graph removes the host's per-call launch and argument costs."""
    import torch

    fn()  # warm: one-time attributes and caches outside the capture
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def bench_block(args, local_rank, peaks):
    """The block's FFN half, out = x + sum_i GeLU(LN(x) A_i) B_i: forward on
    the large workload (T=16384, D=4096, F=16384, N=8) against the plain MLP
    forward, the layer norm alone (2 * T * D * 2 bytes), and the block's
    backward on the fwd+bwd workload (T=8192, D=8192, F=32768, N=8)."""
    import torch

    import tensor_transformer_mlp_column_gb300 as tp
    from tpmlp_inputs import WORKLOADS, make_block_inputs

    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    reps = max(3, min(args.steps // 10, 10))
    out = {}
    w = WORKLOADS["large"]
    inp = make_block_inputs(w, seed=0)
    x = inp["x"].to(dev)
    sh = tp.tpmlp_shard(inp["A"].to(dev), inp["B"].to(dev), w.N)
    del inp
    y = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
    xn = torch.empty_like(x)
    fwd = {"workload": f"{w.name}: T={w.T} D={w.D} F={w.F} N={w.N} bf16"}
    ms = _time_ms(lambda: tp.tpmlp_layer_norm(x, 1e-5, xn), dev, stream, 20)
    gbs = 2.0 * w.T * w.D * 2 / (ms * 1e-3) / 1e9
    fwd["layer_norm"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    for mode in ("faithful", "fused"):
        ws = torch.empty(tp.tpmlp_block_workspace_bytes(w.T, sh, mode, 0), dtype=torch.uint8, device=dev)
        ms_b = _time_ms(lambda: tp.tpmlp_block_forward(x, sh, mode, 1e-5, y, None, ws), dev, stream, reps)
        ms_m = _time_ms(lambda: tp.tpmlp_forward(xn, sh, mode, y, ws), dev, stream, reps)
        tf = w.fwd_flops() / (ms_b * 1e-3) / 1e12
        fwd[mode] = {"ms": round(ms_b, 4), "TFLOP/s": round(tf, 1), "mlp_forward_ms": round(ms_m, 4),
                     "overhead_ms": round(ms_b - ms_m, 4)}
        del ws
    tp.tpmlp_check_status(stream)
    sh.free()
    del x, y, xn
    out["forward"] = fwd
    if args.no_backward:
        return out
    w = WORKLOADS["fwd_bwd"]
    inp = make_block_inputs(w, seed=0, with_dout=True)
    x, dout = inp["x"].to(dev), inp["dout"].to(dev)
    sh = tp.tpmlp_shard(inp["A"].to(dev), inp["B"].to(dev), w.N)
    del inp
    dx = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
    dA = [torch.empty((w.D, w.Fs), dtype=torch.float32, device=dev) for _ in range(w.N)]
    dB = [torch.empty((w.Fs, w.D), dtype=torch.float32, device=dev) for _ in range(w.N)]
    bwd = {"workload": f"{w.name}: T={w.T} D={w.D} F={w.F} N={w.N} bf16"}
    for mode in ("faithful", "fused"):
        ws = torch.empty(tp.tpmlp_block_workspace_bytes(w.T, sh, mode, 1), dtype=torch.uint8, device=dev)
        ms = _time_ms(lambda: tp.tpmlp_block_backward(x, dout, sh, mode, 1e-5, dx, dA, dB, ws), dev, stream, reps)
        alg = 8.0 * w.T * w.D * w.F / (ms * 1e-3) / 1e12
        bwd[mode] = {"ms": round(ms, 3), "TFLOP/s": round(alg, 1), "TFLOP/s_incl_recompute": round(alg * 10 / 8, 1)}
        del ws
    tp.tpmlp_check_status(stream)
    sh.free()
    out["backward"] = bwd
    return out


def bench_sp(args, local_rank, peaks):
    """Sequence-parallel form: the forward with X in N rank slices and Y
    reduce-scattered to them (large workload) against the plain forward, the
    two simulated collectives alone, and the backward (fwd+bwd workload)."""
    import torch

    import tensor_transformer_mlp_column_gb300 as tp
    from tpmlp_inputs import WORKLOADS, make_inputs

    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    reps = max(3, min(args.steps // 10, 10))
    w = WORKLOADS["large"]
    inp = make_inputs(w, seed=0)
    X = inp["X"].to(dev)
    sh = tp.tpmlp_shard(inp["A"].to(dev), inp["B"].to(dev), w.N)
    del inp
    n, Ts = w.N, w.T // w.N
    Xs = [c.clone() for c in torch.chunk(X, n, dim=0)]
    Ys = [torch.empty((Ts, w.D), dtype=torch.float32, device=dev) for _ in range(n)]
    Y = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
    fwd = {"workload": f"{w.name}: T={w.T} D={w.D} F={w.F} N={w.N} bf16, {Ts} tokens per rank"}
    Xg = torch.empty_like(X)
    # The gather moves 268 MB in about 40 us, less than the call's host-side
    # cost on this machine's cores: back-to-back eager calls would time the
    # host, so the kernel's rate comes from a CUDA graph of 20 calls (the
    # eager figure is kept beside it).
    ms = _time_ms(lambda: tp.tpmlp_all_gather(Xs, Xg), dev, stream, 20)
    gms = _time_graph_ms(lambda: tp.tpmlp_all_gather(Xs, Xg), dev, 20)
    gbs = 2.0 * w.T * w.D * 2 / (gms * 1e-3) / 1e9
    fwd["all_gather"] = {"ms": round(gms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                         "eager_ms": round(ms, 4), "timing": "CUDA graph of 20 calls"}
    Yp = torch.randn((n, w.T, w.D), dtype=torch.float32, device=dev)
    ms = _time_ms(lambda: tp.tpmlp_reduce_scatter(Yp, Ys), dev, stream, 20)
    gbs = (n + 1.0) * w.T * w.D * 4 / (ms * 1e-3) / 1e9
    fwd["reduce_scatter"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    del Yp
    for mode in ("faithful", "fused"):
        ws = torch.empty(tp.tpmlp_sp_workspace_bytes(w.T, sh, mode, 0), dtype=torch.uint8, device=dev)
        ms_sp = _time_ms(lambda: tp.tpmlp_forward_sp(Xs, sh, mode, Ys, ws), dev, stream, reps)
        ms_u = _time_ms(lambda: tp.tpmlp_forward(X, sh, mode, Y, ws), dev, stream, reps)
        fwd[mode] = {"ms": round(ms_sp, 4), "TFLOP/s": round(w.fwd_flops() / (ms_sp * 1e-3) / 1e12, 1),
                     "unsplit_forward_ms": round(ms_u, 4), "overhead_ms": round(ms_sp - ms_u, 4)}
        del ws
    tp.tpmlp_check_status(stream)
    sh.free()
    del X, Xs, Ys, Y, Xg
    out = {"forward": fwd}
    if args.no_backward:
        return out
    w = WORKLOADS["fwd_bwd"]
    inp = make_inputs(w, seed=0)
    n, Ts = w.N, w.T // w.N
    Xs = [c.clone() for c in torch.chunk(inp["X"].to(dev), n, dim=0)]
    dYs = [c.clone() for c in torch.chunk(inp["dY"].to(dev), n, dim=0)]
    sh = tp.tpmlp_shard(inp["A"].to(dev), inp["B"].to(dev), w.N)
    del inp
    dXs = [torch.empty((Ts, w.D), dtype=torch.float32, device=dev) for _ in range(n)]
    dA = [torch.empty((w.D, w.Fs), dtype=torch.float32, device=dev) for _ in range(n)]
    dB = [torch.empty((w.Fs, w.D), dtype=torch.float32, device=dev) for _ in range(n)]
    bwd = {"workload": f"{w.name}: T={w.T} D={w.D} F={w.F} N={w.N} bf16, {Ts} tokens per rank"}
    for mode in ("faithful", "fused"):
        ws = torch.empty(tp.tpmlp_sp_workspace_bytes(w.T, sh, mode, 1), dtype=torch.uint8, device=dev)
        ms = _time_ms(lambda: tp.tpmlp_backward_sp(Xs, dYs, sh, mode, dXs, dA, dB, ws), dev, stream, reps)
        alg = 8.0 * w.T * w.D * w.F / (ms * 1e-3) / 1e12
        bwd[mode] = {"ms": round(ms, 3), "TFLOP/s": round(alg, 1), "TFLOP/s_incl_recompute": round(alg * 10 / 8, 1)}
        del ws
    tp.tpmlp_check_status(stream)
    sh.free()
    out["backward"] = bwd
    return out


def bench_attention(args, local_rank, peaks):
    """Head-split attention over the sequence sweep (batch 8, seq 128/256/512,
    D=1024, 16 heads of 64, N=4): the whole forward in both modes and the
    local heads alone (QKV projection, V^T, attention), with the attention
    core's FLOP (4 batch seq^2 D) growing quadratically in seq."""
    import torch

    import tensor_transformer_mlp_column_gb300 as tp
    from tpmlp_inputs import ATTN_WORKLOADS, make_attn_inputs

    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name in ("attn_seq128", "attn_seq256", "attn_seq512"):
        w = ATTN_WORKLOADS[name]
        inp = make_attn_inputs(w, seed=0)
        d = {k: v.to(dev) for k, v in inp.items()}
        sh = tp.tpmlp_attn_shard(d["Wq"], d["Wk"], d["Wv"], d["Wo"], w.heads, w.N)
        Y = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
        O = torch.empty((w.N, w.T, w.D // w.N), dtype=torch.bfloat16, device=dev)
        res = {"batch": w.batch, "seq": w.seq, "D": w.D, "heads": w.heads, "N": w.N}
        ws = torch.empty(tp.tpmlp_attn_workspace_bytes(w.batch, w.seq, sh, None), dtype=torch.uint8, device=dev)
        ms = _time_ms(lambda: tp.tpmlp_attn_heads(d["X"], w.batch, sh, O, ws), dev, stream, 50, 5)
        res["heads_ms"] = round(ms, 4)
        for mode in ("faithful", "fused"):
            ws = torch.empty(tp.tpmlp_attn_workspace_bytes(w.batch, w.seq, sh, mode), dtype=torch.uint8, device=dev)
            ms = _time_ms(lambda: tp.tpmlp_attn_forward(d["X"], w.batch, sh, mode, Y, ws), dev, stream, 50, 5)
            gms = _time_graph_ms(lambda: tp.tpmlp_attn_forward(d["X"], w.batch, sh, mode, Y, ws), dev, 50)
            tf = w.fwd_flops() / (ms * 1e-3) / 1e12
            res[mode] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                         "frac_bf16": round(tf / peaks["bf16_tflops"], 4),
                         "graph_ms": round(gms, 4), "graph_TFLOP/s": round(w.fwd_flops() / (gms * 1e-3) / 1e12, 1)}
        tp.tpmlp_check_status(stream)
        sh.free()
        out[name] = res
    # Longer sequences at the same 4096 tokens (batch x seq = 4096): the
    # attention core's FLOP grow linearly in seq here, the projections not at all.
    for name in ("attn_long1024", "attn_long2048", "attn_long4096"):
        w = ATTN_WORKLOADS[name]
        inp = make_attn_inputs(w, seed=0)
        d = {k: v.to(dev) for k, v in inp.items()}
        sh = tp.tpmlp_attn_shard(d["Wq"], d["Wk"], d["Wv"], d["Wo"], w.heads, w.N)
        Y = torch.empty((w.T, w.D), dtype=torch.float32, device=dev)
        ws = torch.empty(tp.tpmlp_attn_workspace_bytes(w.batch, w.seq, sh, "fused"), dtype=torch.uint8, device=dev)
        ms = _time_ms(lambda: tp.tpmlp_attn_forward(d["X"], w.batch, sh, "fused", Y, ws), dev, stream, 20, 3)
        tf = w.fwd_flops() / (ms * 1e-3) / 1e12
        out[name] = {"batch": w.batch, "seq": w.seq, "fused": {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                     "frac_bf16": round(tf / peaks["bf16_tflops"], 4)}}
        tp.tpmlp_check_status(stream)
        sh.free()
    # heads time against seq: least squares on (1, seq, seq^2)
    import numpy as np

    seqs = np.array([128.0, 256.0, 512.0])
    ys = np.array([out[f"attn_seq{int(s)}"]["heads_ms"] for s in seqs])
    coef = np.linalg.solve(np.stack([np.ones(3), seqs, seqs ** 2], axis=1), ys)
    out["heads_ms_fit"] = {"c0": round(float(coef[0]), 5), "c1_per_seq": float(coef[1]), "c2_per_seq2": float(coef[2])}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tpmlp", "reference"], default="tpmlp")
    ap.add_argument("--workload", default="large")
    ap.add_argument("--T", type=int, default=0, help="override the token count (smaller profiling cases)")
    ap.add_argument("--N", type=int, default=0, help="override the shard count (experiments)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward measurement (fwd+bwd workload)")
    ap.add_argument("--only", choices=["backward", "gelu", "block", "sp", "attention", "small"], default=None,
                    help="run one secondary measurement alone and print it (smaller profiling commands)")
    ap.add_argument("--small", choices=["gpt2_small", "seq128", "seq256", "seq512"], default=None,
                    help="with --only small: that workload alone")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.only:
        import torch

        torch.cuda.set_device(0)
        peaks = load_peaks()
        fn = {"backward": lambda: bench_backward(args, 0, peaks), "gelu": lambda: bench_gelu(0, peaks),
              "block": lambda: bench_block(args, 0, peaks), "sp": lambda: bench_sp(args, 0, peaks),
              "attention": lambda: bench_attention(args, 0, peaks), "small": lambda: bench_small_workloads(0, args.small)}
        print(json.dumps({"only": args.only, args.only: fn[args.only]()}))
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from tpmlp_inputs import WORKLOADS

    w = WORKLOADS[args.workload]
    if args.T:
        w = w.with_(T=args.T)
    if args.N:
        w = w.with_(N=args.N)
    step_flops = 2 * w.fwd_flops()
    config = {"workload": f"{w.name}: T={w.T} D={w.D} F={w.F} N={w.N} bf16 operands, fp32 accumulate; "
                          "step = faithful forward + fused forward",
              "T": w.T, "D": w.D, "F": w.F, "N": w.N,
              "l2": "inputs larger than L2 (X + A + B = 402 MB, H = 537 MB per pass); no flush",
              "parallelism": "replicas" if args.gpus > 1 else "single GPU"}

    if args.impl == "reference":
        if rank != 0:
            return
        cores = len(os.sched_getaffinity(0))
        per_step = max(1.0, min(8.0, 150.0 / (args.warmup + args.steps)))
        r = run_oracle(per_step, args.warmup + args.steps, cores)
        rows = r["rows"]
        times = r["seconds"][args.warmup:]
        sample_flops = 4.0 * rows * w.D * w.F
        v = sample_flops * len(times) / sum(times) / 1e12
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded normal inputs of the large workload's shapes)", "config": config,
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                 "sample": f"{rows} token rows of the large workload per step (one float64 forward)"},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl", rank=rank, world_size=world,
                                             device_id=torch.device("cuda", local_rank))
    res = bench_tpmlp(args, rank, world, local_rank)
    ms_step = res["total_ms"] / args.steps
    e2e_ms = res["e2e_ms"]
    if world > 1:
        ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms], torch.device("cuda", local_rank))
    if rank != 0:
        torch.distributed.destroy_process_group() if world > 1 else None
        return

    peaks = load_peaks()
    avg = res["avg"]
    T, D, F, N = w.T, w.D, w.F, w.N
    gemm_flops = 2.0 * T * D * F
    flops_of = {"gemm1_gelu(faithful)": gemm_flops, "gemm2_partials": gemm_flops,
                "gemm1_gelu(fused)": gemm_flops, "gemm2_fused_sum": gemm_flops}
    reduce_bytes = (N + 1) * T * D * 4.0
    kernel_report = {}
    for k, ms in avg.items():
        if k == "allreduce":
            gbs = reduce_bytes / (ms * 1e-3) / 1e9
            kernel_report[k] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        else:
            tf = flops_of[k] / (ms * 1e-3) / 1e12
            kernel_report[k] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                                "frac_bf16": round(tf / peaks["bf16_tflops"], 4)}
    step_ms_sum = sum(avg.values())
    dominant = max((k for k in avg if k != "allreduce"), key=lambda k: avg[k])
    default_workload = args.workload == "large" and not args.T and not args.N
    # The timed region lasts res["total_ms"]: well under the seconds-long loop
    # that settles the sustained (power-capped) rate, so the kernels are held
    # against the burst peak; a region of several seconds takes the sustained one.
    long_region = res["total_ms"] >= 2000.0
    pk = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    pk_kind = (f"sustained bf16 (timed region {res['total_ms'] / 1e3:.2f} s)" if long_region else
               f"burst bf16 (timed region {res['total_ms'] / 1e3:.2f} s, under the seconds-long sustained loop)")
    ach = flops_of[dominant] / (avg[dominant] * 1e-3) / 1e12
    red_gbs = reduce_bytes / (avg["allreduce"] * 1e-3) / 1e9
    roof = {"kernel": dominant, "bound": "tensor", "achieved": round(ach, 1), "peak": pk, "unit": "TFLOP/s",
            "frac": round(ach / pk, 4), "traffic": traffic_of(dominant) if default_workload else None,
            "algorithmic_flops": flops_of[dominant],
            # operands read once and results written once
            "algorithmic_bytes": (2.0 * (T * D + D * F + T * F) if dominant.startswith("gemm1") else
                                  2.0 * (T * F + F * D) + 4.0 * T * D * (N if dominant == "gemm2_partials" else 1)),
            "peak_source": f"{peaks['source']}: {pk_kind}",
            # the second target: the faithful simulated all-reduce against HBM
            "reduce": {"kernel": "allreduce", "bound": "hbm", "achieved": round(red_gbs, 1),
                       "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(red_gbs / peaks["hbm_gbs"], 4),
                       "traffic": traffic_of("allreduce") if default_workload else None,
                       "algorithmic_bytes": reduce_bytes,
                       "peak_source": f"{peaks['source']}: copy bandwidth"},
            "modes": {}}
    value = job_throughput(world, step_flops, ms_step)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal inputs, A,B ~ N(0, 0.02), X ~ N(0, 1))", "config": config,
        "frac_bf16_peak": round(value / world / pk, 4),
        "reduce": {"GB/s": round(red_gbs, 1), "peak": peaks["hbm_gbs"],
                   "frac_hbm": round(red_gbs / peaks["hbm_gbs"], 4), "bytes": reduce_bytes},
        "modes": {
            "faithful": {"ms": round(avg["gemm1_gelu(faithful)"] + avg["gemm2_partials"] + avg["allreduce"], 4)},
            "fused": {"ms": round(avg["gemm1_gelu(fused)"] + avg["gemm2_fused_sum"], 4)},
        },
        "kernels": kernel_report, "kernel_ms_sum": round(step_ms_sum, 4),
        "roofline": roof,
        "clocks": res["clocks"],
        "e2e": {"value": round(job_throughput(world, step_flops, e2e_ms), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"]},
        "gpu_launches": res["launches"],
        "peaks": peaks,
    }
    for m in ("faithful", "fused"):
        ms = line["modes"][m]["ms"]
        tf = w.fwd_flops() / (ms * 1e-3) / 1e12
        line["modes"][m]["TFLOP/s"] = round(tf, 1)
        line["modes"][m]["frac_bf16"] = round(tf / pk, 4)
        roof["modes"][m] = dict(line["modes"][m])
    if not args.no_backward and world == 1 and not args.T and not args.N:
        line["backward"] = bench_backward(args, local_rank, peaks)
        line["other_workloads"] = bench_small_workloads(local_rank)
        line["gelu"] = bench_gelu(local_rank, peaks)
        line["block"] = bench_block(args, local_rank, peaks)
        line["sequence_parallel"] = bench_sp(args, local_rank, peaks)
        line["attention"] = bench_attention(args, local_rank, peaks)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
