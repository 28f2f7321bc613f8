#!/usr/bin/env python3
"""Benchmark of the host-streamed tiled linear operator on GB300.

One step = one forward + one backward of Y = X.W over the whole workload:
N weight tiles streamed host->device into the depth-d ring, forward GEMM per
tile, every tile fetched again for backward, dW_i written back device->host,
dX accumulated in fp32.  The headline workload is the largest one that fits
one GPU: the 64K-hidden FFN (X bf16 [2048, 65536], W bf16 [65536, 262144] =
32 GiB in pinned host memory, N = 16 tiles of 16384 columns, d = 2; dW another
32 GiB).  Inputs are synthetic (seeded normal draws).

Printed: one JSON line (rank 0).  `value` is whole-job fwd+bwd TFLOP/s
(6*T*K*M FLOPs per step) with X and dY resident in HBM; `e2e` is the same
metric when every step also copies X and dY from pinned host memory and reads
Y and dX back.  `exposed_copy_pct` = 100 * max(0, t_step - t_compute_resident)
/ t_copy_only, where t_compute_resident is the same GEMM sequence on tiles
already in HBM and t_copy_only the same copy schedule with no GEMMs.
`per_config` measures the pages' other layers in the same process: the
GPT-scale FFN, the 1T-width FFN at d = 1, 2, 3, and the arithmetic-intensity
sweep's token counts with automatic depth.  FLOPs, link bytes and the time
bounds come from offload_streamed_gb300.roofline.

--impl reference times the CPU oracle (the plain triple-loop definition) on a
bounded sample of the same workload on this machine's host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tiled-linear fwd+bwd TFLOP/s, host-streamed weights; % copy time exposed"
UNIT = "TFLOP/s"

CONFIGS = {
    "tiny": dict(T=256, K=1024, M=4096, N=4, d=1,
                 workload="tiny: X bf16 [256,1024] ~N(0,1), W bf16 [1024,4096] ~N(0,1/1024) pinned host, "
                          "N=4 tiles of 1024 cols, dY ~N(0,1), d=1"),
    "gpt": dict(T=8192, K=8192, M=32768, N=8, d=2,
                workload="GPT-scale FFN up-proj: X bf16 [8192,8192] ~N(0,1), W bf16 [8192,32768] ~N(0,1/8192) "
                         "pinned host (tile-major), N=8 tiles of 4096 cols, dY ~N(0,1), d=2"),
    "1t": dict(T=4096, K=25600, M=102400, N=16, d=2,
               workload="1T-width FFN: X bf16 [4096,25600] ~N(0,1), W bf16 [25600,102400] (5.2 GB) ~N(0,1/25600) "
                        "pinned host (tile-major), N=16 tiles of 6400 cols, dY ~N(0,1)"),
    "sweep": dict(T=8192, K=16384, M=65536, N=16, d=2,
                  workload="ait sweep: X bf16 [T,16384] ~N(0,1), W bf16 [16384,65536] (2 GiB) ~N(0,1/16384) "
                           "pinned host (tile-major), N=16 tiles of 4096 cols, dY ~N(0,1)"),
    "64k": dict(T=2048, K=65536, M=262144, N=16, d=2,
                workload="64K-hidden FFN: X bf16 [2048,65536] ~N(0,1), W bf16 [65536,262144] (32 GiB + 32 GiB dW) "
                         "~N(0,1/65536) pinned host (tile-major), N=16 tiles of 16384 cols, dY ~N(0,1), d=2"),
}
HEADLINE = "64k"  # the largest configuration that fits one GPU

# The pages' other layers, measured in the same run (config, d, T): the
# GPT-scale layer at its d; the 1T-width layer at d = 1, 2, 3; the ait sweep's
# token counts with automatic depth (d = -1), and its largest at fixed depths.
PER_CONFIG = [("gpt", 2, None), ("1t", 1, None), ("1t", 2, None), ("1t", 3, None),
              ("sweep", -1, 2048), ("sweep", -1, 4096), ("sweep", -1, 8192), ("sweep", -1, 65536),
              ("sweep", 4, 65536), ("sweep", 8, 65536), ("sweep", 15, 65536)]
PER_CONFIG_STEPS, PER_CONFIG_WARMUP = 6, 2
# each per-config block (streamed steps, resident GEMMs) times at least this
# long, after a warm-up of at least this long, so that both blocks settle at
# the clock the power budget gives that work
PER_CONFIG_SECONDS, PER_CONFIG_WARM_SECONDS = 0.3, 0.15

TIMING_EVERY = 4


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ----------------------------------------------------------------------------
class Dist:
    def __init__(self, backend: str):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.barrier()
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
            os.remove(self.path)
        except Exception:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the CPU oracle as a timed baseline
# ----------------------------------------------------------------------------
ORACLE_COLS = 1024  # W columns of the oracle's sample (part of tile 0)


def oracle_sample_inputs(x, dy, w_tile0, cols: int = ORACLE_COLS):
    """Host bf16 bits of the oracle's sample: X [T, K], the first `cols`
    columns of dY and of W (which tile 0 holds)."""
    import numpy as np

    from offload_streamed_gb300 import inputs as I
    xb = np.ascontiguousarray(I.bits(x.cpu()))
    c = min(cols, w_tile0.shape[1])
    dyb = np.ascontiguousarray(I.bits(dy[:, :c].contiguous().cpu()))
    wb = np.ascontiguousarray(I.bits(w_tile0[:, :c].contiguous().cpu()))
    return xb, dyb, wb


def oracle_sample_run(xb, dyb, wb, T_s: int):
    """Forward + backward of the same operator restricted to the first T_s
    tokens and the sample's columns, by the CPU oracle: Y and dW of those
    columns and their share of dX.  Returns (seconds, flops, threads)."""
    import numpy as np

    from oracle import oracle as O
    X = np.ascontiguousarray(xb[:T_s])
    dY = np.ascontiguousarray(dyb[:T_s])
    K, C = wb.shape
    t0 = time.perf_counter()
    O.forward(X, wb)
    O.backward(X, wb, dY)
    dt = time.perf_counter() - t0
    return dt, 6.0 * T_s * K * C, O.max_threads()


def oracle_baseline(xb, dyb, wb, target_s: float = 12.0):
    """Pick a token count so that the timed oracle run takes ~target_s: a run
    costs a fixed part plus a part per token, fitted from two short runs (16
    and 64 tokens, enough to keep every core busy as the final run does)."""
    t1, t2 = 16, 64
    d1 = oracle_sample_run(xb, dyb, wb, t1)[0]
    d2 = oracle_sample_run(xb, dyb, wb, t2)[0]
    per_token = max((d2 - d1) / (t2 - t1), 1e-6)
    fixed = max(d1 - per_token * t1, 0.0)
    T_s = max(2, min(xb.shape[0], int((target_s - fixed) / per_token)))
    dt, fl, thr = oracle_sample_run(xb, dyb, wb, T_s)
    C = wb.shape[1]
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"fwd+bwd of the first {T_s} tokens against the first {C} columns of W (Y and dW of "
                      f"those columns, their share of dX; 6*{T_s}*K*{C} FLOPs, {dt:.1f} s, plain C fp32 triple "
                      f"loops, OpenMP)",
            "seconds": dt, "tokens": T_s, "columns": C}


def oracle_extras(cfg, xb_full, dyh, w_tm_bits, rate_tflops: float, seed: int) -> dict:
    """Further timings of the oracle as it stands, on the host cores:
    (i) the tiny configuration in full (fwd + bwd) on one core and on all;
    (ii) the sampled check of this workload (4096 seeded entries of each of Y,
    dX and dW, plus the tile-edge entries), as the full-size parity tests run
    it, reading W in its tile-major host storage; (iii) the full problem's
    time extrapolated from the measured rate, an estimate, not a
    measurement."""
    from oracle import oracle as O
    from offload_streamed_gb300 import inputs as I
    out = {}
    tiny = CONFIGS["tiny"]
    Tt, Kt, Mt = tiny["T"], tiny["K"], tiny["M"]
    X = I.bits(I.make_x(Tt, Kt, seed))
    dY = I.bits(I.make_dy(Tt, Mt, seed))
    W = I.bits(I.make_w_tile(Kt, Mt, 0, seed))
    cores = O.max_threads()
    for label, n in (("one_core_s", 1), ("all_cores_s", cores)):
        O.set_threads(n)
        t0 = time.perf_counter()
        O.forward(X, W)
        O.backward(X, W, dY)
        out[label] = round(time.perf_counter() - t0, 4)
    O.set_threads(cores)
    out = {"tiny_full_fwd_bwd": dict(out, flops=6.0 * Tt * Kt * Mt, cores=cores)}
    T, K, M, N = cfg["T"], cfg["K"], cfg["M"], cfg["N"]
    dyb = I.bits(dyh)
    t0 = time.perf_counter()
    for tid, (nr, nc, fn, a, b) in enumerate([(T, M, O.sample_y, xb_full, w_tm_bits),
                                               (T, K, O.sample_dx, dyb, w_tm_bits),
                                               (K, M, O.sample_dw, xb_full, dyb)]):
        r, c = I.sample_indices(nr, nc, 4096, seed, tid)
        fn(a, b, r, c)
    out["sampled_check_s"] = round(time.perf_counter() - t0, 3)
    out["full_problem_s_est"] = round(6.0 * T * K * M / (rate_tflops * 1e12), 1)
    out["full_problem_note"] = "estimate: 6TKM at the measured sample rate, not run"
    return out


def measure_link(w, dw, nbytes: int, reps: int = 3):
    """Pinned host<->device copy bandwidth (GB/s): H2D alone, D2H alone, and
    each direction while both run."""
    import torch
    n = min(nbytes, w.nbytes, dw.nbytes)
    src = w.tensor.view(torch.uint8)[:n]
    dst_h = dw.tensor.view(torch.uint8)[:n]
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")
    dev2 = torch.empty(n, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        best = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            best.append(time.perf_counter() - t0)
        return min(best)

    def h2d():
        with torch.cuda.stream(s1):
            dev.copy_(src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            dst_h.copy_(dev2, non_blocking=True)

    def both():
        h2d()
        d2h()

    th, td, tb = timed(h2d), timed(d2h), timed(both)
    del dev, dev2
    return {"h2d_gbs": n / th / 1e9, "d2h_gbs": n / td / 1e9, "bidir_each_gbs": n / tb / 1e9,
            "bytes": n}


def time_copy_schedule(cfg, w, dw, reps: int = 3):
    """t_copy_only: the step's copy schedule alone -- forward's N tile fetches,
    then backward's N fetches with N gradient write-backs on a second
    stream."""
    import torch
    K, M, N = cfg["K"], cfg["M"], cfg["N"]
    tb = K * (M // N) * 2
    wt = w.tensor.view(torch.uint8)
    dwt = dw.tensor.view(torch.uint8)
    slots = torch.empty(2, tb, dtype=torch.uint8, device="cuda")
    s_h, s_d = torch.cuda.Stream(), torch.cuda.Stream()
    ts = []
    for _ in range(reps):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_h)
        s_d.wait_event(e0)
        with torch.cuda.stream(s_h):
            for i in range(N):
                slots[i % 2].copy_(wt[i * tb:(i + 1) * tb], non_blocking=True)
        fwd_done = torch.cuda.Event()
        fwd_done.record(s_h)
        s_d.wait_event(fwd_done)
        for i in reversed(range(N)):
            with torch.cuda.stream(s_h):
                slots[i % 2].copy_(wt[i * tb:(i + 1) * tb], non_blocking=True)
            with torch.cuda.stream(s_d):
                dwt[i * tb:(i + 1) * tb].copy_(slots[(i + 1) % 2], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(s_d)
        s_h.wait_event(ev)
        e1.record(s_h)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    del slots
    return min(ts)


def dx_group(d: int, N: int, Mi: int) -> int:
    """Tiles per dX launch at depth d: the engine's rule (tiled_linear.h,
    backward), max(2, ceil(8192 / Mi)) bounded by d, N and 4."""
    d = min(d, N - 1)
    if d < 2 or N < 2 or Mi % 64:
        return 1
    return min(max(2, -(-8192 // Mi)), d, N, 4)


def w_device_rowmajor(w, K: int, M: int, N: int):
    """W [K, M] row-major on the device from its tile-major host buffer, one
    tile at a time (no second full-size copy on either side)."""
    import torch
    Mi = M // N
    w_dev = torch.empty(K, M, dtype=torch.bfloat16, device="cuda")
    wt = w.tensor.view(N, K, Mi)
    for i in range(N):
        w_dev[:, i * Mi:(i + 1) * Mi].copy_(wt[i], non_blocking=True)
    torch.cuda.synchronize()
    return w_dev


def time_resident_compute(tl, cfg, x, dy, w_dev, steps: int, depth: int, warmup: int = 2):
    """t_compute_resident: the step's GEMM sequence (the same kernels, same
    order, dX over the same tile groups as at `depth`) on W already in HBM
    (row-major [K, M], so a group of tiles is one column block), through the
    resident-GEMM ABI; `warmup` untimed steps first."""
    import torch
    T, K, M, N = x.shape[0], cfg["K"], cfg["M"], cfg["N"]
    Mi = M // N
    gsz = dx_group(depth, N, Mi)
    y = torch.empty(T, M, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(T, K, dtype=torch.float32, device="cuda")
    stage = torch.empty(2, K, Mi, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    st = s.cuda_stream

    def step():
        for i in range(N):
            tl.tiled_linear_gemm_forward(T, K, Mi, x.data_ptr(), K, w_dev[:, i * Mi:].data_ptr(), M,
                                         y[:, i * Mi:].data_ptr(), M, err.data_ptr(), st)
        nx, pend = 0, 0
        for j in range(N):
            i = N - 1 - j
            tl.tiled_linear_gemm_dw(T, K, Mi, x.data_ptr(), K, dy[:, i * Mi:].data_ptr(), M,
                                    stage[j % 2].data_ptr(), Mi, err.data_ptr(), st)
            if pend + 1 < gsz and j + 1 < N:
                pend += 1
                continue  # reduced together with the next tiles
            w = (pend + 1) * Mi
            tl.tiled_linear_gemm_dx(T, K, w, dy[:, i * Mi:].data_ptr(), M, w_dev[:, i * Mi:].data_ptr(), M,
                                    dx.data_ptr(), K, nx > 0, err.data_ptr(), st)
            nx, pend = nx + 1, 0

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        step()
    e1.record(s)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    return e0.elapsed_time(e1) / steps


def run_e2e(op, cfg, x, dy, steps: int, warmup: int):
    """Same step through the public API with X, dY in pinned host memory
    copied in every step and Y, dX read back every step.  Activations are
    double-buffered across steps: step k's X and dY are copied in on one
    stream while step k-1 computes, and its Y and dX are read back on another
    while step k+1 computes.  Every copy of every timed step is inside the
    timed region (its end waits for the last read-back)."""
    import torch

    from offload_streamed_gb300 import tiled_linear as tl
    T, K, M = cfg["T"], cfg["K"], cfg["M"]
    xh = tl.PinnedBuffer(T * K)
    dyh = tl.PinnedBuffer(T * M)
    yh = [tl.PinnedBuffer(T * M) for _ in range(2)]
    dxh = [tl.PinnedBuffer(T * K, dtype=torch.float32) for _ in range(2)]
    xh.tensor.view(T, K).copy_(x)
    dyh.tensor.view(T, M).copy_(dy)
    xd = [torch.empty(T, K, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dyd = [torch.empty(T, M, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    yd = [torch.empty(T, M, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dxd = [torch.empty(T, K, dtype=torch.float32, device="cuda") for _ in range(2)]
    s = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()   # activations in / results out
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("x_in", "dy_in", "fwd", "bwd", "y_out", "dx_out")}
    for b in range(2):  # every buffer starts free
        for k in ("bwd", "y_out", "dx_out"):
            ev[k][b].record(s)
    k_step = [0]

    def step():
        b = k_step[0] % 2
        k_step[0] += 1
        with torch.cuda.stream(cin):        # set b's last users (two steps back) are done
            cin.wait_event(ev["bwd"][b])
            xd[b].copy_(xh.tensor.view(T, K), non_blocking=True)
            ev["x_in"][b].record(cin)
            dyd[b].copy_(dyh.tensor.view(T, M), non_blocking=True)
            ev["dy_in"][b].record(cin)
        with torch.cuda.stream(s):
            s.wait_event(ev["x_in"][b])
            s.wait_event(ev["y_out"][b])
            op.forward(xd[b], yd[b], stream=s)
            ev["fwd"][b].record(s)
        with torch.cuda.stream(cout):
            cout.wait_event(ev["fwd"][b])
            yh[b].tensor.view(T, M).copy_(yd[b], non_blocking=True)
            ev["y_out"][b].record(cout)
        with torch.cuda.stream(s):
            s.wait_event(ev["dy_in"][b])
            s.wait_event(ev["dx_out"][b])
            op.backward(xd[b], dyd[b], dxd[b], stream=s)
            ev["bwd"][b].record(s)
        with torch.cuda.stream(cout):
            cout.wait_event(ev["bwd"][b])
            dxh[b].tensor.view(T, K).copy_(dxd[b], non_blocking=True)
            ev["dx_out"][b].record(cout)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        step()
    for b in range(2):
        s.wait_event(ev["y_out"][b])
        s.wait_event(ev["dx_out"][b])
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h2d = T * K * 2 + T * M * 2
    d2h = T * M * 2 + T * K * 4
    for buf in [xh, dyh] + yh + dxh:
        buf.close()
    return ms, h2d, d2h


# DRAM traffic per launch of each GEMM kernel, from an ncu capture of
# `bench.py --config C --profile-gemms 2` (profiles/dram_traffic_<C>_tile.txt).
# The file records a hash of the kernel sources it was taken with; once they
# change the figure no longer describes the kernel and the bench reports null.
KERNEL_SOURCES = ["tl_gemm.cu", "tl_gemm.h", "tl_kernel_common.cuh", "tl_ptx.cuh"]


def traffic_file(config: str) -> str:
    return os.path.join(ROOT, "profiles", f"dram_traffic_{config}_tile.txt")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "offload_streamed_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def load_traffic(config: str) -> dict:
    """{kernel key: DRAM bytes per launch} if the profile of `config` matches
    the current kernel sources, else {}."""
    try:
        with open(traffic_file(config)) as fh:
            kv = dict(l.split(":", 1) for l in fh.read().splitlines() if ":" in l and not l.startswith("#"))
    except OSError:
        return {}
    kv = {k.strip(): v.strip() for k, v in kv.items()}
    if kv.get("source_sha256") != kernel_source_hash() or kv.get("config") != config:
        return {}
    return {k: int(v) for k, v in kv.items() if k.endswith("_bytes_per_launch")}


def profile_gemms(cfg, reps: int, kinds) -> None:
    """The resident GEMMs of one tile (dX of one tile group, as a step runs
    it) of the workload, `reps` times each, in the order fwd, dW, dX, for the
    kinds asked: a small fixed launch sequence for ncu captures of each kernel
    (inputs above L2; each kind allocates only its own operands)."""
    import torch

    import __graft_entry__ as g
    from offload_streamed_gb300 import inputs as I
    from offload_streamed_gb300 import tiled_linear as tl

    g.build()
    T, K, M, N = cfg["T"], cfg["K"], cfg["M"], cfg["N"]
    Mi = M // N
    nx = dx_group(cfg["d"], N, Mi) * Mi
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    x = I.make_x(T, K, 0, device="cuda")
    for kind in ("fwd", "dw", "dx"):
        if kind not in kinds:
            continue
        if kind == "fwd":
            w1 = I.make_w_tile(K, Mi, 0, 0, device="cuda")  # one tile, as a ring slot holds it
            y = torch.empty(T, Mi, dtype=torch.bfloat16, device="cuda")
            for _ in range(reps):
                tl.tiled_linear_gemm_forward(T, K, Mi, x.data_ptr(), K, w1.data_ptr(), Mi, y.data_ptr(), Mi,
                                             err.data_ptr(), st)
            torch.cuda.synchronize()
            del w1, y
        elif kind == "dw":
            dy = I.make_dy(T, Mi, 0, device="cuda")
            dw = torch.empty(K, Mi, dtype=torch.bfloat16, device="cuda")
            for _ in range(reps):
                tl.tiled_linear_gemm_dw(T, K, Mi, x.data_ptr(), K, dy.data_ptr(), Mi, dw.data_ptr(), Mi,
                                        err.data_ptr(), st)
            torch.cuda.synchronize()
            del dy, dw
        else:
            dy = I.make_dy(T, nx, 0, device="cuda")
            w = I.make_w_tile(K, nx, 0, 0, device="cuda")  # a tile group, row-major [K, nx]
            dx = torch.zeros(T, K, dtype=torch.float32, device="cuda")
            for _ in range(reps):
                tl.tiled_linear_gemm_dx(T, K, nx, dy.data_ptr(), nx, w.data_ptr(), nx, dx.data_ptr(), K, 1,
                                        err.data_ptr(), st)
            torch.cuda.synchronize()
            del dy, w, dx
        torch.cuda.empty_cache()
    if int(err[0].item()) != 0:
        raise SystemExit(f"profile_gemms: kernel timeout word {int(err[0].item())}")
    log(f"[bench] profile-gemms: {reps} x {sorted(kinds)} at T={T} K={K} Mi={Mi} (dX over {nx} columns)")


def profile_library_gemm(cfg, reps: int) -> None:
    """The library's bf16 GEMM (torch.matmul, cuBLAS) on the forward's tile
    shape, Y_i[T, Mi] = X[T, K] . W_i[K, Mi], `reps` times: the comparison
    point for the counters of our forward kernel (same inputs, same sizes)."""
    import torch

    from offload_streamed_gb300 import inputs as I
    T, K, M, N = cfg["T"], cfg["K"], cfg["M"], cfg["N"]
    Mi = M // N
    x = I.make_x(T, K, 0, device="cuda")
    w1 = I.make_w_tile(K, Mi, 0, 0, device="cuda")
    y = torch.empty(T, Mi, dtype=torch.bfloat16, device="cuda")
    for _ in range(reps):
        torch.matmul(x, w1, out=y)
    torch.cuda.synchronize()
    log(f"[bench] profile-library-gemm: {reps} x torch.matmul at T={T} K={K} Mi={Mi}")


def run_host_adam(tl, op, x, y, dy, dx, steps: int, dist: Dist, flops_step: float) -> dict:
    """Forward + backward + the Adam step on the host CPU (fp32 master and
    moments, all host threads), the update of each tile overlapping the GPU's
    backward of the later ones.  Restores the host W afterwards."""
    import torch
    w_save = op._w.tensor.clone()
    opt = tl.HostAdam(op, lr=1e-4, threads=0)
    s = torch.cuda.current_stream()
    for _ in range(2):
        op.forward(x, y, stream=s)
        op.backward(x, dy, dx, stream=s)
        opt.step()
    opt.wait()
    torch.cuda.synchronize()
    busy0 = opt.stats()["busy_seconds"]
    t0 = time.perf_counter()
    for _ in range(steps):
        op.forward(x, y, stream=s)
        op.backward(x, dy, dx, stream=s)
        opt.step()
    opt.wait()
    torch.cuda.synchronize()
    ms = dist.max((time.perf_counter() - t0) * 1e3 / steps)
    busy = (opt.stats()["busy_seconds"] - busy0) / steps
    n = op._w.numel
    opt.close()
    op._w.tensor.copy_(w_save)
    return {"value": round(dist.world * flops_step / (ms / 1e3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 3), "steps": steps, "optimizer_busy_ms_per_step": round(busy * 1e3, 3),
            "params": n, "host_optimizer_gbs": round(28.0 * n / busy / 1e9, 1) if busy > 0 else None,
            "host_threads": os.cpu_count(),
            "what": "forward + backward + Adam on the host CPU (fp32 master, m, v; 28 B per parameter read "
                    "and written), each tile's update overlapping the GPU; host wall-clock per step"}


def _union(iv):
    """Merged [start, end) intervals."""
    out = []
    for a, b in sorted(iv):
        if out and a <= out[-1][1]:
            out[-1][1] = max(out[-1][1], b)
        else:
            out.append([a, b])
    return out


def _overlap(x, y):
    i = j = 0
    tot = 0.0
    while i < len(x) and j < len(y):
        a, b = max(x[i][0], y[j][0]), min(x[i][1], y[j][1])
        tot += max(0.0, b - a)
        if x[i][1] < y[j][1]:
            i += 1
        else:
            j += 1
    return tot


def timeline_summary(trace: list) -> dict:
    """Busy shares of one call's timeline (tiled_linear_get_trace): GEMMs,
    the host->device and device->host copies, and both links at once under
    a GEMM, as percentages of the call's span.  The span starts at the call's
    start (time 0): copies fetched earlier, under the previous call's GEMMs,
    are clipped to it."""
    if not trace:
        return {}
    t1 = max(e["end_ms"] for e in trace)
    span = max(t1, 1e-9)
    sel = lambda f: _union([(max(e["start_ms"], 0.0), e["end_ms"]) for e in trace
                            if f(e["kind"]) and e["end_ms"] > 0.0])
    gem = sel(lambda k: k.endswith("gemm") or k == "pass")
    h2d = sel(lambda k: k == "h2d")
    d2h = sel(lambda k: k == "d2h")
    early = sum(1 for e in trace if e["kind"] == "h2d" and e["start_ms"] < 0.0)
    busy = lambda u: sum(b - a for a, b in u)
    both = _union([(max(a, c), min(b, d)) for a, b in h2d for c, d in d2h if min(b, d) > max(a, c)])
    pct = lambda v: round(100.0 * v / span, 1)
    return {"span_ms": round(span, 4), "gemm_busy_pct": pct(busy(gem)), "h2d_busy_pct": pct(busy(h2d)),
            "d2h_busy_pct": pct(busy(d2h)), "both_links_under_gemm_pct": pct(_overlap(both, gem)),
            "copy_outside_gemm_pct": pct(busy(_union(h2d + d2h)) - _overlap(_union(h2d + d2h), gem)),
            "copies_started_before_the_call": early}


def disk_bandwidth(path: str, nbytes: int, threads: int = 4, chunk: int = 16 << 20) -> tuple:
    """Direct-I/O write then read bandwidth (GB/s) of a scratch file of
    `nbytes` at `path`, in `chunk` requests spread over `threads` threads
    (the file tier's own request size and thread count)."""
    import mmap
    import threading
    nbytes -= nbytes % chunk
    bufs = [mmap.mmap(-1, chunk) for _ in range(threads)]  # page-aligned, as direct I/O needs
    for b in bufs:
        b.write(os.urandom(4096) * (chunk // 4096))

    def run(fd, write):
        nxt = [0]
        lock = threading.Lock()

        def work(b):
            while True:
                with lock:
                    off = nxt[0]
                    nxt[0] += chunk
                if off >= nbytes:
                    return
                if write:
                    os.pwrite(fd, b, off)
                else:
                    os.preadv(fd, [b], off)
        th = [threading.Thread(target=work, args=(b,)) for b in bufs]
        t0 = time.perf_counter()
        for t in th:
            t.start()
        for t in th:
            t.join()
        return nbytes / (time.perf_counter() - t0) / 1e9

    fd = os.open(path, os.O_RDWR | os.O_CREAT | os.O_TRUNC | os.O_DIRECT, 0o644)
    try:
        w = run(fd, True)
        os.fsync(fd)
        r = run(fd, False)
    finally:
        os.close(fd)
        os.unlink(path)
    return w, r


def run_file_tier(tl, cfg, w, x, y, dy, dx, steps: int, dist: Dist, flops_step: float, peaks: dict,
                  tier_dir: str) -> dict:
    """The same step with W and dW in files (tiled_linear_create_file): every
    tile read from the W file with direct I/O into pinned host slots, every
    dW tile written to the dW file, one storage tier below host memory."""
    import tempfile

    import torch
    K, M, N, d = cfg["K"], cfg["M"], cfg["N"], cfg["d"]
    work = tempfile.mkdtemp(prefix="tl_tier_", dir=tier_dir)
    wp, dwp = os.path.join(work, "w.bin"), os.path.join(work, "dw.bin")
    try:
        w.tensor.view(torch.int16).numpy().tofile(wp)  # tile-major, as the tier reads it
        bw_write, bw_read = disk_bandwidth(os.path.join(work, "probe.bin"), 2 * K * M)
        op = tl.TiledLinearFile(K, M, N, d, wp, dwp, host_slots=4, io_threads=4)
        s = torch.cuda.current_stream()
        op.forward(x, y, stream=s)
        op.backward(x, dy, dx, stream=s)
        op.sync()
        f0 = op.file_stats()
        dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            op.forward(x, y, stream=s)
            op.backward(x, dy, dx, stream=s)
        torch.cuda.synchronize()
        op.sync()  # the step's dW is in its file
        sec = dist.max((time.perf_counter() - t0) / steps)
        f1 = op.file_stats()
        op.close()
    except (tl.TiledLinearError, OSError) as e:  # e.g. a filesystem without direct I/O
        if dist.world > 1:  # the other ranks would wait at this extension's barrier
            raise
        return {"unavailable": f"{type(e).__name__}: {e}"}
    finally:
        for f in (wp, dwp, os.path.join(work, "probe.bin")):
            if os.path.exists(f):
                os.unlink(f)
        os.rmdir(work)
    from offload_streamed_gb300 import roofline as RL
    rd = f1["read_bytes"] - f0["read_bytes"]
    wr = f1["write_bytes"] - f0["write_bytes"]
    R = peaks["bf16_tflops"] * 1e12
    t_in, t_out = RL.step_h2d_bytes(K, M) / (bw_read * 1e9), RL.step_d2h_bytes(K, M) / (bw_write * 1e9)
    t_roof = max(flops_step / R, t_in, t_out)
    t_serial = max(flops_step / R, t_in + t_out)
    return {"value": round(dist.world * flops_step / sec / 1e12, 2), "unit": UNIT, "ms_per_step": round(sec * 1e3, 2),
            "steps": steps, "read_bytes_per_step": rd // steps, "write_bytes_per_step": wr // steps,
            "disk_read_gbs": round(bw_read, 2), "disk_write_gbs": round(bw_write, 2),
            "tier_read_gbs": round(rd / steps / sec / 1e9, 2), "tier_write_gbs": round(wr / steps / sec / 1e9, 2),
            "fetch_wait_ms_per_step": round((f1["fetch_wait_seconds"] - f0["fetch_wait_seconds"]) / steps * 1e3, 2),
            "step_roofline": {
                "form": "one disk serves the reads and the writes in turn: t_roof = max(6TKM/R, 4KM/B_disk_read + "
                        "2KM/B_disk_write); frac_if_overlapped uses max(6TKM/R, 4KM/B_read, 2KM/B_write)",
                "roofline_tflops": round(flops_step / t_serial / 1e12, 2), "frac": round(t_serial / sec, 4),
                "t_roof_ms": round(t_serial * 1e3, 2), "frac_if_overlapped": round(t_roof / sec, 4)},
            "host_slots": f1["host_slots"], "io_threads": f1["io_threads"], "dir": tier_dir,
            "what": "W and dW in files on the box's disk, read and written with direct I/O through pinned host "
                    "slots (tiled_linear_create_file); host wall-clock per step until dW is in its file"}


def run_ffn_chain(tl, cfg, x, y_up, dx, seed: int, steps: int, dist: Dist) -> dict:
    """The workload's layer followed by its down-projection (M -> K, N tiles of
    K/N columns, W2 [M, K] pinned, tile-major), run as one chain: one ring and
    one prefetcher across both operators.  A step is a chain forward plus a
    chain backward (12 T K M FLOPs); X, Y_up and dX are the main workload's
    device buffers."""
    import torch

    from offload_streamed_gb300 import inputs as I
    T, K, M, N, d = cfg["T"], cfg["K"], cfg["M"], cfg["N"], cfg["d"]
    w1, dw1 = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
    w2, dw2 = tl.PinnedBuffer(M * K), tl.PinnedBuffer(M * K)
    I.fill_w_host(w1.tensor, K, M, N, True, seed, device="cuda")
    I.fill_w_host(w2.tensor, M, K, N, True, seed + 1, device="cuda")
    ch = tl.TiledLinearChain([K, M, K], [N, N], d, [w1, w2], [dw1, dw2])
    y_down = torch.empty(T, K, dtype=torch.bfloat16, device="cuda")
    dy = I.make_dy(T, K, seed + 1, device="cuda")
    ys = [y_up, y_down]
    s = torch.cuda.current_stream()
    for _ in range(3):
        ch.forward(x, ys, stream=s)
        ch.backward(x, ys, dy, dx, stream=s)
    torch.cuda.synchronize()
    ch.reset_stats()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        ch.forward(x, ys, stream=s)
        ch.backward(x, ys, dy, dx, stream=s)
    e1.record(s)
    torch.cuda.synchronize()
    ms = dist.max(e0.elapsed_time(e1) / steps)
    st = ch.stats()
    ch.close()
    for b in (w1, dw1, w2, dw2):
        b.close()
    from offload_streamed_gb300 import roofline as RL
    flops = RL.step_flops(T, K, M) + RL.step_flops(T, M, K)  # up- then down-projection
    return {"value": round(dist.world * flops / (ms / 1e3) / 1e12, 2), "unit": UNIT, "ms_per_step": round(ms, 4),
            "steps": steps, "tiles": st["n_tiles"], "launches_per_step": st["fwd_launches"] + st["bwd_launches"],
            "h2d_bytes_per_step": st["fwd_h2d_bytes"] + st["bwd_h2d_bytes"],
            "d2h_bytes_per_step": st["bwd_d2h_bytes"],
            "compute_stream_idle_pct": round(100.0 * (1.0 - (st["sum_fwd_gemm_ms"] + st["sum_bwd_dw_gemm_ms"]
                                                              + st["sum_bwd_dx_gemm_ms"]) /
                                                        max(st["sum_fwd_total_ms"] + st["sum_bwd_total_ms"], 1e-9)),
                                             2),
            "workload": f"FFN chain: up [{K}->{M}] then down [{M}->{K}], N={N} tiles each, d={d}, T={T}, "
                        "one ring and prefetcher over both; bf16 activations between the operators"}


# ----------------------------------------------------------------------------
def _extension(fn, dist: Dist) -> dict:
    """Run one extension measurement; a failure there (a pinned allocation
    the host refuses, a filesystem without direct I/O) is reported in its own
    object and never costs the method's measurement.  A CUDA failure is not
    caught: it can leave the context unusable, and then nothing after it is
    trustworthy.  With several ranks nothing is caught either: a rank that
    went on would leave the others waiting in the extension's collectives."""
    from offload_streamed_gb300 import tiled_linear as tl
    if dist.world > 1:
        return fn()
    try:
        return fn()
    except (tl.TiledLinearError, OSError, MemoryError) as e:
        if isinstance(e, tl.TiledLinearError) and e.status in (tl.TL_ERR_CUDA, tl.TL_ERR_TIMEOUT):
            raise
        return {"unavailable": f"{type(e).__name__}: {e}"}


# ----------------------------------------------------------------------------
# workloads, timed steps and one measured configuration
# ----------------------------------------------------------------------------
def config_dict(cfg, world: int) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": cfg["workload"], "T": cfg["T"], "K": cfg["K"], "M": cfg["M"], "N": cfg["N"], "d": cfg["d"],
            "host_layout": "tile-major [N][K][M/N]",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 between steps: W streamed from host every pass"}


class Workload:
    """Pinned host W and dW (tile-major) and device X and dY of one layer; X
    and dY are drawn for `T_alloc` tokens (a measurement at fewer tokens uses
    their first rows)."""

    def __init__(self, cfg, seed: int, T_alloc: int | None = None):
        from offload_streamed_gb300 import inputs as I
        from offload_streamed_gb300 import tiled_linear as tl
        self.K, self.M, self.N = cfg["K"], cfg["M"], cfg["N"]
        T = T_alloc or cfg["T"]
        self.w = tl.PinnedBuffer(self.K * self.M)
        self.dw = tl.PinnedBuffer(self.K * self.M)
        I.fill_w_host(self.w.tensor, self.K, self.M, self.N, True, seed, device="cuda")
        self.x = I.make_x(T, self.K, seed, device="cuda")
        self.dy = I.make_dy(T, self.M, seed, device="cuda")

    def close(self):
        import torch
        self.w.close()
        self.dw.close()
        self.x = self.dy = None
        torch.cuda.empty_cache()


def timed_steps(op, x, dy, y, dx, steps: int, warmup: int, before=None, after=None):
    """`warmup` untimed steps, then `steps` steps timed with CUDA events on the
    current stream, one event per step boundary; the engine records
    per-launch events on every TIMING_EVERY-th call.  `before` / `after` run
    just outside the timed region (barriers, clock sampling).  Returns (mean
    ms per step, sorted per-step ms, engine stats of the timed calls)."""
    import torch
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        op.forward(x, y, stream=s)
        op.backward(x, dy, dx, stream=s)
    torch.cuda.synchronize()
    op.set_timing(TIMING_EVERY)
    op.reset_stats()
    if before:
        before()
    torch.cuda.synchronize()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    marks[0].record(s)
    for k in range(steps):
        op.forward(x, y, stream=s)
        op.backward(x, dy, dx, stream=s)
        marks[k + 1].record(s)
    torch.cuda.synchronize()
    if after:
        after()
    ms = marks[0].elapsed_time(marks[-1]) / steps
    per_step = sorted(marks[k].elapsed_time(marks[k + 1]) for k in range(steps))
    st = op.stats()
    op.set_timing(1)
    return ms, per_step, st


KERNEL_NAMES = {"fwd_gemm": "fwd_gemm (Y_i = X.W_i)", "dw_gemm": "dw_gemm (dW_i = X^T.dY_i)",
                "dx_gemm": "dx_gemm (dX += dY_i.W_i^T over a tile group)"}


def kernel_rates(st, T: int, K: int, M: int, N: int) -> dict:
    """Per GEMM kind over the timed calls: mean launch time (the engine's CUDA
    events on the compute stream), FLOPs and algorithmic HBM bytes per launch
    (the dX figures are the means over a backward's tile-group launches, the
    first of which stores and the rest add), launches per step."""
    from offload_streamed_gb300 import roofline as RL
    Mi = M // N
    fc, bc = max(st["fwd_timed_calls"], 1), max(st["bwd_timed_calls"], 1)
    n_dx = max(st["bwd_launches"] - N, 1)
    wx = M / n_dx  # mean reduction width of a dX launch
    dx_bytes = sum(RL.gemm_bytes("dx", T, K, wx, accumulate=j > 0) for j in range(n_dx)) / n_dx
    out = {"fwd_gemm": (st["sum_fwd_gemm_ms"] / (fc * N), RL.gemm_flops(T, K, Mi), N, RL.gemm_bytes("fwd", T, K, Mi)),
           "dw_gemm": (st["sum_bwd_dw_gemm_ms"] / (bc * N), RL.gemm_flops(T, K, Mi), N, RL.gemm_bytes("dw", T, K, Mi)),
           "dx_gemm": (st["sum_bwd_dx_gemm_ms"] / (bc * n_dx), RL.gemm_flops(T, K, wx), n_dx, dx_bytes)}
    return {k: {"avg_launch_ms": ms, "flops_per_launch": fl, "launches_per_step": n, "bytes_per_launch": b,
                "tflops": fl / (ms / 1e3) / 1e12 if ms > 0 else None}
            for k, (ms, fl, n, b) in out.items()}


def step_bounds(T: int, K: int, M: int, R: float, link: dict) -> dict:
    """The step's roofline: tightest (forward and backward may overlap across
    calls) and per phase (summed separately, the backward's two directions
    at their concurrent rates)."""
    from offload_streamed_gb300 import roofline as RL
    bh, bd, bb = link["h2d_gbs"] * 1e9, link["d2h_gbs"] * 1e9, link["bidir_each_gbs"] * 1e9
    t, bound = RL.step_bound(T, K, M, R, bh, bd)
    tf, tb = RL.phase_bound(T, K, M, R, bh, bb, bb)
    flops = RL.step_flops(T, K, M)
    return {"t_roof_ms": t * 1e3, "roofline_tflops": flops / t / 1e12, "bound_by": bound,
            "t_phase_ms": (tf + tb) * 1e3, "phase_tflops": flops / (tf + tb) / 1e12,
            "t_phase_fwd_ms": tf * 1e3, "t_phase_bwd_ms": tb * 1e3,
            "ait_h2d_flop_per_byte": RL.ait_h2d(T), "crossover_T": RL.crossover_tokens(R, bh)}


def mean_link(a: dict, b: dict) -> dict:
    return {k: 0.5 * (a[k] + b[k]) if isinstance(a[k], float) else a[k] for k in a}


def block_sizes(step_ms: float, steps: int, warmup: int) -> tuple[int, int]:
    """Timed steps and warm-up steps of one per-config block, from one
    step's time: at least `steps` and `warmup`, and at least
    PER_CONFIG_SECONDS of timed steps after PER_CONFIG_WARM_SECONDS of
    warm-up (a step read as under 1 ms counts as 1 ms)."""
    est = max(step_ms, 1.0)
    return (max(steps, math.ceil(PER_CONFIG_SECONDS * 1e3 / est)),
            max(warmup, math.ceil(PER_CONFIG_WARM_SECONDS * 1e3 / est)))


def measure_config(tl, wl, cfg, d: int, T: int, steps: int, warmup: int, R: float, w_dev,
                   R_sustained: float | None = None) -> dict:
    """One layer at depth d (-1: automatic) and T tokens: TFLOP/s over the
    mean step, the step roofline (tightest and per phase), exposed copy
    against the resident GEMMs and the copy schedule alone, the depth and
    staging slots the handle used, and each GEMM kind's rate.  The host link
    is shared with the machine's other jobs and its speed drifts, so the
    link and the copy schedule are measured right before and after the
    point's streamed steps, and the point's roofline uses their mean.
    `steps` and `warmup` are minimums: each block runs at least
    PER_CONFIG_SECONDS after at least PER_CONFIG_WARM_SECONDS of warm-up.
    With R_sustained, the step roofline is also given against the sustained
    bf16 peak (the blocks run long enough to reach the power cap)."""
    import torch

    from offload_streamed_gb300 import roofline as RL
    K, M, N = cfg["K"], cfg["M"], cfg["N"]
    x, dy = wl.x[:T], wl.dy[:T]
    y = torch.empty(T, M, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(T, K, dtype=torch.float32, device="cuda")
    op = tl.TiledLinear(K, M, N, d, wl.w, wl.dw, tile_major=True)
    resident = w_dev is not None
    link0 = measure_link(wl.w, wl.dw, 1 << 29, reps=2)
    t_copy0 = time_copy_schedule(cfg, wl.w, wl.dw, reps=2)
    # the automatic depth is chosen after the first forward and used from the
    # second; one streamed step then sizes the blocks
    op.forward(x, y)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    op.forward(x, y, stream=s)
    op.backward(x, dy, dx, stream=s)
    e1.record(s)
    torch.cuda.synchronize()
    steps, warmup = block_sizes(e0.elapsed_time(e1), steps, warmup)
    depth = op.stats()["depth"]
    # The resident GEMMs run right before and right after the streamed
    # steps, with the same warm-up and at least as many timed steps, and
    # the two are averaged: each block settles at the clock the power budget
    # gives its own work, and the clock's drift over seconds cancels
    if resident:
        t_res0 = time_resident_compute(tl, cfg, x, dy, w_dev, steps, depth, warmup)
    ms, per_step, st = timed_steps(op, x, dy, y, dx, steps, warmup)
    if resident:
        t_res1 = time_resident_compute(tl, cfg, x, dy, w_dev, steps, st["depth"], warmup)
    assert op.close() == tl.TL_OK
    del y, dx
    t_copy1 = time_copy_schedule(cfg, wl.w, wl.dw, reps=2)
    link1 = measure_link(wl.w, wl.dw, 1 << 29, reps=2)
    link = mean_link(link0, link1)
    t_copy_only = 0.5 * (t_copy0 + t_copy1)
    flops = RL.step_flops(T, K, M)
    b = step_bounds(T, K, M, R, link)
    med = per_step[len(per_step) // 2]
    kr = kernel_rates(st, T, K, M, N)
    fc, bc = max(st["fwd_timed_calls"], 1), max(st["bwd_timed_calls"], 1)
    h2d_ms = st["sum_fwd_h2d_ms"] + st["sum_bwd_h2d_ms"]
    out = {"config": cfg["name"], "T": T, "K": K, "M": M, "N": N, "d": d, "depth": st["depth"],
           "staging_slots": st["staging_slots"], "steps": steps, "warmup": warmup,
           "tflops": round(flops / (ms / 1e3) / 1e12, 1), "ms_per_step": round(ms, 3),
           "step_ms_median": round(med, 3), "step_ms_max": round(per_step[-1], 3),
           # the same at the median step: a stall of the shared host link
           # (tens of ms, now and then) moves the mean of a short block
           "tflops_median_step": round(flops / (med / 1e3) / 1e12, 1),
           "step_roofline": {"tflops": round(b["roofline_tflops"], 1), "frac": round(b["t_roof_ms"] / ms, 4),
                             "bound_by": b["bound_by"]},
           "phase_roofline": {"tflops": round(b["phase_tflops"], 1), "frac": round(b["t_phase_ms"] / ms, 4)},
           "kernels_tflops": {k: (round(v["tflops"], 1) if v["tflops"] else None) for k, v in kr.items()},
           "link_gbs_before_after": {"h2d": [round(link0["h2d_gbs"], 1), round(link1["h2d_gbs"], 1)],
                                     "d2h": [round(link0["d2h_gbs"], 1), round(link1["d2h_gbs"], 1)],
                                     "bidir_each": [round(link0["bidir_each_gbs"], 1),
                                                    round(link1["bidir_each_gbs"], 1)]},
           "link_gbs_during_steps": {
               "h2d_per_copy": round((st["fwd_h2d_bytes"] + st["bwd_h2d_bytes"]) * fc / (h2d_ms / 1e3) / 1e9, 1)
               if h2d_ms > 0 else None,
               "d2h_per_copy": round(st["bwd_d2h_bytes"] * bc / (st["sum_bwd_d2h_ms"] / 1e3) / 1e9, 1)
               if st["sum_bwd_d2h_ms"] > 0 else None}}
    if R_sustained:
        bs = step_bounds(T, K, M, R_sustained, link)
        out["step_roofline"]["sustained"] = {"R_tflops": round(R_sustained / 1e12, 1),
                                             "tflops": round(bs["roofline_tflops"], 1),
                                             "frac": round(bs["t_roof_ms"] / ms, 4), "bound_by": bs["bound_by"]}
    out["t_copy_only_ms"] = round(t_copy_only, 3)
    # how long the compute stream sat idle inside the timed calls (waiting
    # for copies), as a share of the copy schedule: the part of the exposed
    # copy that is waiting, not GEMMs slowed by the copies running beside them
    gemm_ms = st["sum_fwd_gemm_ms"] + st["sum_bwd_dw_gemm_ms"] + st["sum_bwd_dx_gemm_ms"]
    wait_ms = max(0.0, st["sum_fwd_total_ms"] + st["sum_bwd_total_ms"] - gemm_ms) / fc
    out["compute_wait_ms_per_step"] = round(wait_ms, 3)
    out["compute_wait_pct_of_copy"] = round(100.0 * wait_ms / t_copy_only, 2)
    if resident:
        t_res = 0.5 * (t_res0 + t_res1)
        out["t_compute_resident_ms"] = round(t_res, 3)
        out["t_compute_resident_before_after_ms"] = [round(t_res0, 3), round(t_res1, 3)]
        out["exposed_copy_pct"] = round(100.0 * max(0.0, ms - t_res) / t_copy_only, 2)
        out["exposed_copy_pct_median_step"] = round(100.0 * max(0.0, med - t_res) / t_copy_only, 2)
    return out


def run_per_config(tl, args, R: float, dist: Dist, R_sustained: float | None = None) -> dict:
    """The pages' other layers (PER_CONFIG), each workload built once and
    measured at its depths and token counts."""
    import torch
    out, groups = [], {}
    for name, d, T in PER_CONFIG:
        groups.setdefault(name, []).append((d, T))
    for name, pts in groups.items():
        cfg = dict(CONFIGS[name], name=name)
        T_alloc = max(T or cfg["T"] for _, T in pts)
        log(f"[bench] per-config {name}: T up to {T_alloc}, points {pts}")
        wl = Workload(cfg, args.seed, T_alloc)
        w_dev = w_device_rowmajor(wl.w, cfg["K"], cfg["M"], cfg["N"])
        for d, T in pts:
            out.append(measure_config(tl, wl, cfg, d, T or cfg["T"], PER_CONFIG_STEPS, PER_CONFIG_WARMUP, R, w_dev,
                                      R_sustained))
            log(f"[bench] {out[-1]}")
        del w_dev
        wl.close()
    torch.cuda.synchronize()
    return {"min_steps": PER_CONFIG_STEPS, "min_warmup": PER_CONFIG_WARMUP,
            "min_block_s": PER_CONFIG_SECONDS, "min_warmup_s": PER_CONFIG_WARM_SECONDS,
            "what": "each layer measured in this process like the headline (mean step over the timed steps, "
                    "each point's `steps` and `warmup` sized to at least min_block_s and min_warmup_s); "
                    "d = -1 is the automatic depth, `depth` the one it chose and `staging_slots` the dW slots it "
                    "carved; exposed_copy_pct against the same GEMMs on W resident in HBM (timed right before and "
                    "right after the streamed steps, each block as long and as warmed up as the streamed one) "
                    "and the copy schedule alone; step_roofline is max(6TKM/R, 4KM/B_h2d, "
                    "2KM/B_d2h) with R the burst bf16 peak (`sustained`: the same with the sustained one, which "
                    "these blocks run long enough to meet), phase_roofline sums forward and backward bounds "
                    "with the backward's links at "
                    "their concurrent rates, both with the link measured right before and after the point "
                    "(the host link is shared with the machine's other jobs)",
            "points": out}


def run_ours(args, cfg, dist: Dist):
    import torch

    import __graft_entry__ as g
    from offload_streamed_gb300 import roofline as RL
    from offload_streamed_gb300 import tiled_linear as tl

    torch.cuda.set_device(dist.local_rank)
    if dist.rank == 0:  # one rank builds; the others find the library fresh after the barrier
        g.build()
    dist.barrier()
    if dist.rank != 0:
        g.build()
    peaks = load_peaks()
    R = peaks["bf16_tflops"] * 1e12
    T, K, M, N, d = cfg["T"], cfg["K"], cfg["M"], cfg["N"], cfg["d"]
    flops_step = RL.step_flops(T, K, M)
    want_cpu = (not args.no_cpu_baseline) and dist.rank == 0 and dist.world == 1

    log(f"[bench] rank {dist.rank}: building workload {args.config} (T={T} K={K} M={M} N={N} d={d})")
    wl = Workload(cfg, args.seed)
    x, dy = wl.x, wl.dy
    op = tl.TiledLinear(K, M, N, d, wl.w, wl.dw, tile_major=True)
    y = torch.empty(T, M, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(T, K, dtype=torch.float32, device="cuda")

    # --- timed region -------------------------------------------------------
    try:
        gpu_id = str(torch.cuda.get_device_properties(dist.local_rank).uuid)
        gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    clocks = {}

    def before():
        dist.barrier()
        sampler.start()
        time.sleep(0.25)

    def after():
        dist.barrier()
        clocks["v"] = sampler.stop()

    link_before = measure_link(wl.w, wl.dw, 1 << 30) if not args.skip_aux else None
    ms_local, per_step, st = timed_steps(op, x, dy, y, dx, args.steps, args.warmup, before, after)
    ms = dist.max(ms_local)
    launches = args.steps * (st["fwd_launches"] + st["bwd_launches"])

    # --- the last timed call's launch and copy timeline ------------------------
    trace_f, trace_b = op.trace(False), op.trace(True)
    if args.trace_out and dist.rank == 0:
        with open(args.trace_out, "w") as f:
            json.dump({"workload": cfg["workload"], "forward": trace_f, "backward": trace_b}, f)

    # --- the dominant kernel against its roofline ------------------------------
    kr = kernel_rates(st, T, K, M, N)
    dom = max(kr, key=lambda k: kr[k]["avg_launch_ms"] * kr[k]["launches_per_step"])
    kd = kr[dom]
    achieved = kd["flops_per_launch"] / (kd["avg_launch_ms"] / 1e3) / 1e12
    traffic = load_traffic(args.config).get(dom + "_bytes_per_launch")
    roofline = {"bound": "tensor", "kernel": KERNEL_NAMES[dom], "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_kind": f"bf16 dense burst, {peaks['source']} (the kernel runs inside a sub-second call; "
                             "the clocks object gives the SM clock of the timed region)",
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "sustained_peak": peaks["bf16_tflops_sustained"],
                "flops_per_launch": kd["flops_per_launch"], "avg_launch_ms": round(kd["avg_launch_ms"], 4),
                "launches_per_step": kd["launches_per_step"],
                "algorithmic_bytes_per_launch": int(kd["bytes_per_launch"]), "traffic": traffic,
                "traffic_source": f"profiles/dram_traffic_{args.config}_tile.txt (ncu dram__bytes_read.sum + "
                                  "dram__bytes_write.sum; null when the kernel sources changed since)",
                "all_kernels_tflops": {KERNEL_NAMES[k]: round(v["tflops"], 1) for k, v in kr.items() if v["tflops"]},
                "timing": f"CUDA events around every launch of every {TIMING_EVERY}th step "
                          f"({st['fwd_timed_calls']} of {st['fwd_calls']} steps), on the compute stream"}

    out = {"metric": METRIC, "value": round(dist.world * flops_step / (ms / 1e3) / 1e12, 2), "unit": UNIT,
           "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": config_dict(cfg, dist.world), "gpu_launches": launches}
    gemm_ms = st["sum_fwd_gemm_ms"] + st["sum_bwd_dw_gemm_ms"] + st["sum_bwd_dx_gemm_ms"]
    h2d_ms = st["sum_fwd_h2d_ms"] + st["sum_bwd_h2d_ms"]
    fc, bc = max(st["fwd_timed_calls"], 1), max(st["bwd_timed_calls"], 1)
    out["timed_region"] = {
        "launch_mode": "one launch per tile and GEMM (dX per tile group)",
        "depth": st["depth"], "staging_slots": st["staging_slots"],
        "step_ms_median": round(per_step[len(per_step) // 2], 4),
        "step_ms_p90": round(per_step[min(len(per_step) - 1, int(0.9 * len(per_step)))], 4),
        "step_ms_max": round(per_step[-1], 4),
        "gemm_ms_per_step": round(gemm_ms / fc, 4),
        "compute_stream_idle_pct": round(100.0 * max(0.0, 1.0 - gemm_ms / max(
            st["sum_fwd_total_ms"] + st["sum_bwd_total_ms"], 1e-9)), 2),
        "fwd_h2d_gbs_per_copy": round(st["fwd_h2d_bytes"] * fc / (st["sum_fwd_h2d_ms"] / 1e3) / 1e9, 1)
        if st["sum_fwd_h2d_ms"] > 0 else None,
        "h2d_gbs_per_copy": round((st["fwd_h2d_bytes"] + st["bwd_h2d_bytes"]) * fc / (h2d_ms / 1e3) / 1e9, 1)
        if h2d_ms > 0 else None,
        "d2h_gbs_per_copy": round(st["bwd_d2h_bytes"] * bc / (st["sum_bwd_d2h_ms"] / 1e3) / 1e9, 1)
        if st["sum_bwd_d2h_ms"] > 0 else None}
    out["roofline"] = roofline
    out["timeline"] = {"forward": timeline_summary(trace_f), "backward": timeline_summary(trace_b),
                       "source": "CUDA events around every launch and copy of the last timed call "
                                 "(tiled_linear_get_trace)"}
    out["engine_stats_last_step"] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in st.items()
                                     if not k.startswith("sum_")}
    out["clocks"] = clocks.get("v")

    # --- link, copy-only and resident-compute references; end to end -----------
    if not args.skip_aux:
        link_after = measure_link(wl.w, wl.dw, 1 << 30)
        link = mean_link(link_before, link_after)
        t_copy = time_copy_schedule(cfg, wl.w, wl.dw)
        w_dev = w_device_rowmajor(wl.w, K, M, N)
        t_res = time_resident_compute(tl, cfg, x, dy, w_dev, max(3, min(args.steps, 10)), st["depth"])
        del w_dev
        # the headline's resident GEMMs run after its timed steps; at this
        # layer the step is bound by the host link, and the copy schedule
        # (t_copy_only) is as long as the step, so clock drift moves the
        # exposed share by well under a point
        torch.cuda.empty_cache()
        out["copy_overlap"] = {
            "exposed_copy_pct": round(100.0 * max(0.0, ms_local - t_res) / t_copy, 2),
            "exposed_copy_pct_median_step": round(100.0 * max(0.0, per_step[len(per_step) // 2] - t_res) / t_copy, 2),
            "t_step_ms": round(ms_local, 4), "t_compute_resident_ms": round(t_res, 4),
            "t_copy_only_ms": round(t_copy, 4),
            "what": "100 * max(0, t_step - t_compute_resident) / t_copy_only; t_compute_resident = the same GEMM "
                    "launches on W resident in HBM, t_copy_only = the same copy schedule with no GEMMs"}
        out["exposed_copy_pct"] = out["copy_overlap"]["exposed_copy_pct"]
        b = step_bounds(T, K, M, R, link)
        out["step_roofline"] = {
            "form": "t_roof = max(6TKM/R, 4KM/B_h2d, 2KM/B_d2h); roofline TFLOP/s = 6TKM/t_roof",
            "R_tflops": peaks["bf16_tflops"], "B_h2d_gbs": round(link["h2d_gbs"], 1),
            "B_d2h_gbs": round(link["d2h_gbs"], 1), "B_bidir_each_gbs": round(link["bidir_each_gbs"], 1),
            "t_roof_ms": round(b["t_roof_ms"], 4), "roofline_tflops": round(b["roofline_tflops"], 1),
            "frac": round(b["t_roof_ms"] / ms_local, 4), "bound_by": b["bound_by"],
            "ait_h2d_flop_per_byte": b["ait_h2d_flop_per_byte"], "crossover_T": round(b["crossover_T"]),
            "per_phase": {"form": "t = max(2TKM/R, 2KM/B_h2d) + max(4TKM/R, 2KM/B_h2d_bidir, 2KM/B_d2h_bidir)",
                          "t_ms": round(b["t_phase_ms"], 4), "t_fwd_ms": round(b["t_phase_fwd_ms"], 4),
                          "t_bwd_ms": round(b["t_phase_bwd_ms"], 4), "roofline_tflops": round(b["phase_tflops"], 1),
                          "frac": round(b["t_phase_ms"] / ms_local, 4)}}
        out["link"] = {k: round(v, 1) if isinstance(v, float) else v for k, v in link.items()}
        out["link"]["what"] = "pinned 1 GiB copies (h2d alone, d2h alone, each way while both run), the mean of " \
                              "one measurement right before and one right after the timed steps"
        out["link"]["before_after_h2d_gbs"] = [round(link_before["h2d_gbs"], 1), round(link_after["h2d_gbs"], 1)]
        e_ms, h2d, d2h = run_e2e(op, cfg, x, dy, max(3, min(args.steps, 20)), 2)
        e_ms = dist.max(e_ms)
        t_e2e = RL.e2e_bound(T, K, M, R, h2d, d2h, link["h2d_gbs"] * 1e9, link["d2h_gbs"] * 1e9,
                             link["bidir_each_gbs"] * 1e9)
        out["e2e"] = {"value": round(dist.world * flops_step / (e_ms / 1e3) / 1e12, 2), "unit": UNIT,
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 4),
                      "roofline": {"form": "t = max(6TKM/R, link time of (4KM + in) bytes in and (2KM + out) "
                                           "bytes out, both directions together at B_bidir for the smaller "
                                           "amount, the rest alone)",
                                   "t_ms": round(t_e2e * 1e3, 4), "tflops": round(flops_step / t_e2e / 1e12, 1),
                                   "frac": round(t_e2e * 1e3 / e_ms, 4)},
                      # the weight tiles the step streams besides (W in twice, dW out once)
                      "weight_h2d_bytes_per_step": int(RL.step_h2d_bytes(K, M)),
                      "weight_d2h_bytes_per_step": int(RL.step_d2h_bytes(K, M)),
                      "what": "X, dY copied from pinned host memory and Y, dX read back every step "
                              "(weights streamed as always), activations double-buffered across steps"}
    op.close()
    del y, dx

    # --- CPU oracle baseline on a bounded sample of this workload --------------
    if want_cpu:
        from offload_streamed_gb300 import inputs as I
        Mi = M // N
        w_tm = I.bits(wl.w.tensor).reshape(N, K, Mi)
        xb, dyb, wb = oracle_sample_inputs(x, dy, wl.w.tensor.view(N, K, Mi)[0])
        out["cpu_baseline"] = oracle_baseline(xb, dyb, wb, target_s=args.cpu_seconds)
        out["cpu_baseline"].update(oracle_extras(cfg, xb, dy.cpu(), w_tm, out["cpu_baseline"]["value"], args.seed))
        del w_tm
    wl.close()

    # --- the pages' other layers ----------------------------------------------
    if not args.skip_aux and not args.no_per_config:
        out["per_config"] = run_per_config(tl, args, R, dist, peaks["bf16_tflops_sustained"] * 1e12)

    # --- extensions on the GPT-scale layer, apart from the method's metric -------
    if not args.skip_aux:
        gcfg = dict(CONFIGS["gpt"], name="gpt")
        gw = Workload(gcfg, args.seed)
        gT, gK, gM, gN = gcfg["T"], gcfg["K"], gcfg["M"], gcfg["N"]
        gflops = RL.step_flops(gT, gK, gM)
        gop = tl.TiledLinear(gK, gM, gN, gcfg["d"], gw.w, gw.dw, tile_major=True)
        gy = torch.empty(gT, gM, dtype=torch.bfloat16, device="cuda")
        gdx = torch.empty(gT, gK, dtype=torch.float32, device="cuda")
        out["tile_reuse"] = run_tile_reuse(gop, gw.x, gw.dy, gy, gdx, gflops, max(3, min(args.steps, 30)), dist)
        out["host_adam"] = _extension(lambda: run_host_adam(tl, gop, gw.x, gy, gw.dy, gdx,
                                                            max(3, min(args.steps, 10)), dist, gflops), dist)
        out["ffn_chain"] = _extension(lambda: run_ffn_chain(tl, gcfg, gw.x, gy, gdx, args.seed,
                                                            max(3, min(args.steps, 20)), dist), dist)
        out["file_tier"] = _extension(lambda: run_file_tier(tl, gcfg, gw.w, gw.x, gy, gw.dy, gdx, 3, dist, gflops,
                                                            peaks, args.tier_dir), dist)
        for k in ("tile_reuse", "host_adam", "ffn_chain", "file_tier"):
            if isinstance(out.get(k), dict):
                out[k]["layer"] = gcfg["workload"]
        gop.close()
        gw.close()
    return out


def run_tile_reuse(op, x, dy, y, dx, flops_step: float, steps: int, dist: Dist) -> dict:
    """The backward takes the min(d+1, N) tiles the forward left in the ring
    instead of fetching them again (tiled_linear_set_tile_reuse)."""
    import torch
    s = torch.cuda.current_stream()
    op.set_tile_reuse(True)
    for _ in range(3):
        op.forward(x, y, stream=s)
        op.backward(x, dy, dx, stream=s)
    torch.cuda.synchronize()
    op.reset_stats()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(s)
    for _ in range(steps):
        op.forward(x, y, stream=s)
        op.backward(x, dy, dx, stream=s)
    r1.record(s)
    torch.cuda.synchronize()
    r_ms = dist.max(r0.elapsed_time(r1) / steps)
    rs = op.stats()
    op.set_tile_reuse(False)
    return {"value": round(dist.world * flops_step / (r_ms / 1e3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(r_ms, 4), "steps": steps, "bwd_reused_tiles": rs["bwd_reused_tiles"],
            "h2d_bytes_per_step": rs["fwd_h2d_bytes"] + rs["bwd_h2d_bytes"],
            "what": "backward reuses the tiles still resident from forward (not the pages' method, which "
                    "refetches every tile; W unchanged between the two calls)"}


def run_sweep(args, dist: Dist):
    """The arithmetic-intensity sweep: one streamed layer (K = 16384,
    M = 65536, N = 16) timed at T = 512 ... 65536 tokens and depth d = 1 ... 4
    and automatic.  Per point: TFLOP/s over the mean step, the step roofline
    max(6TKM/R, 4KM/B_h2d, 2KM/B_d2h) with the link measured here, and the
    exposed copy against the same GEMMs on resident W and the same copies
    alone.  The link hides behind compute once ait = 1.5 T FLOP/B passes
    R / B_h2d (tm_zero_infinity, "The honest cost")."""
    try:
        depths = [int(v) for v in args.sweep_d.split(",")] if args.sweep_d else SWEEP_D
        tokens = [int(v) for v in args.sweep_t.split(",")] if args.sweep_t else SWEEP_T
    except ValueError:
        depths = tokens = []
    if not depths or not tokens or any(d < -1 for d in depths) or any(not 1 <= T <= max(SWEEP_T) for T in tokens):
        raise SystemExit(f"--sweep-d / --sweep-t: integer depths >= -1 and token counts in 1..{max(SWEEP_T)}")
    import torch

    import __graft_entry__ as g
    from offload_streamed_gb300 import tiled_linear as tl

    torch.cuda.set_device(dist.local_rank)
    g.build()
    peaks = load_peaks()
    R = peaks["bf16_tflops"] * 1e12
    cfg = dict(CONFIGS["sweep"], name="sweep")
    T_max = max(tokens)
    log(f"[sweep] building workload (T up to {T_max}, K={cfg['K']}, M={cfg['M']}, N={cfg['N']})")
    wl = Workload(cfg, args.seed, T_max)
    w_dev = w_device_rowmajor(wl.w, cfg["K"], cfg["M"], cfg["N"])
    sampler = ClockSampler(None)
    sampler.start()
    points = []
    for d in depths:
        for T in tokens:
            points.append(measure_config(tl, wl, cfg, d, T, args.steps, args.warmup, R, w_dev,
                                         peaks["bf16_tflops_sustained"] * 1e12))
            log(f"[sweep] {points[-1]}")
    clocks = sampler.stop()
    del w_dev
    wl.close()
    return {"sweep": "ait", "metric": METRIC, "unit": UNIT, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg["workload"], "K": cfg["K"], "M": cfg["M"], "N": cfg["N"], "T": tokens,
                       "d": depths, "host_layout": "tile-major [N][K][M/N]"},
            "R_tflops": peaks["bf16_tflops"], "points": points,
            "clocks": clocks}


SWEEP_T = [512 << j for j in range(8)]  # 512 ... 65536
SWEEP_D = [1, 2, 3, 4, -1]


def run_reference(args, cfg, dist: Dist):
    """The oracle, as it stands, timed on the host cores: each step is the
    forward + backward of `ref_tokens` tokens of the workload against
    ORACLE_COLS columns of W.  The sample's inputs are drawn on the CPU from
    the workload's seeded streams at the sample's own shapes (the values
    differ from the GPU's draws; the oracle's time does not depend on them)."""
    from oracle import oracle as O
    from offload_streamed_gb300 import inputs as I
    O.build()
    K, M, N = cfg["K"], cfg["M"], cfg["N"]
    C = min(ORACLE_COLS, M // N)
    t = min(args.ref_tokens, cfg["T"])
    xb = I.bits(I.make_x(t, K, args.seed))
    dyb = I.bits(I.make_dy(t, C, args.seed))
    wb = I.bits(I.make_w_tile(K, C, 0, args.seed))
    for _ in range(args.warmup):
        oracle_sample_run(xb, dyb, wb, t)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dt, fl, thr = oracle_sample_run(xb, dyb, wb, t)
    total = time.perf_counter() - t0
    ms = total / args.steps * 1e3
    val = fl / (ms / 1e3) / 1e12
    sample = (f"fwd+bwd of {t} tokens against {C} columns of W per step (Y and dW of those columns, their share "
              f"of dX; 6*{t}*K*{C} FLOPs; inputs drawn on the CPU from the workload's seeded streams)")
    return {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 (fp32 accumulation over bf16 inputs)",
            "data": "synthetic", "config": config_dict(cfg, dist.world),
            "cpu_baseline": {"value": round(val, 6), "unit": UNIT, "cores": thr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(val, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(CONFIGS), default=HEADLINE)
    ap.add_argument("--d", type=int, default=None, help="override the prefetch depth (-1: automatic)")
    ap.add_argument("--T", type=int, default=None, help="override the token count")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--skip-aux", action="store_true",
                    help="only the headline timed steps: no link / copy-only / resident / e2e measurements, "
                         "per-config layers or extensions")
    ap.add_argument("--no-per-config", action="store_true", help="skip the other layers (per_config)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--trace-out", default=None,
                    help="write the last timed forward and backward call's launch / copy timeline (JSON)")
    ap.add_argument("--tier-dir", default=os.environ.get("TMPDIR", "/tmp"),
                    help="directory for the file tier's W and dW files (the file_tier measurement)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-tokens", type=int, default=48)
    ap.add_argument("--sweep", action="store_true",
                    help="time the arithmetic-intensity sweep (K=16384, M=65536, N=16; T = 512..65536, "
                         "d = 1..4 and automatic) and print one JSON line with every point")
    ap.add_argument("--sweep-d", type=str, default=None, metavar="D,...",
                    help="with --sweep: only these depths (-1 = automatic), e.g. 3,4,-1")
    ap.add_argument("--sweep-t", type=str, default=None, metavar="T,...",
                    help="with --sweep: only these token counts (each in 1..65536)")
    ap.add_argument("--profile-gemms", type=int, default=0, metavar="R",
                    help="only run the resident GEMMs of one tile R times (for ncu), print nothing")
    ap.add_argument("--profile-kinds", default="fwd,dw,dx", help="kernels --profile-gemms runs")
    ap.add_argument("--profile-library-gemm", type=int, default=0, metavar="R",
                    help="only run the library's bf16 GEMM (cuBLAS) on the forward's tile shape R times "
                         "(for ncu), print nothing")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        log("[bench] note: fewer than 3 warm-up steps")
    cfg = dict(CONFIGS[args.config], name=args.config)
    if args.d is not None:
        cfg["d"] = args.d
        cfg["workload"] += f" (d set to {args.d})"
    if args.T is not None:
        cfg["T"] = args.T
        cfg["workload"] += f" (T set to {args.T})"
    if args.profile_gemms > 0:
        profile_gemms(cfg, args.profile_gemms, set(args.profile_kinds.split(",")))
        return
    if args.profile_library_gemm > 0:
        profile_library_gemm(cfg, args.profile_library_gemm)
        return
    if args.sweep:
        out = run_sweep(args, Dist("nccl"))
        print(json.dumps(out), flush=True)
        return
    if args.impl == "reference":
        # rank 0 alone times the CPU oracle; other ranks have nothing to do
        if int(os.environ.get("RANK", "0")) != 0:
            return
        os.environ["WORLD_SIZE"] = "1"
        print(json.dumps(run_reference(args, cfg, Dist("gloo"))), flush=True)
        return
    dist = Dist("nccl")
    out = run_ours(args, cfg, dist)
    if dist.rank == 0:
        print(json.dumps(out), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
