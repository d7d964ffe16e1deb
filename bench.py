#!/usr/bin/env python
"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..6] [--all] [--bwd]

One step = one tk_attn_fwd launch over the whole workload (every (b,h) head,
every query row), inputs resident in HBM.  Default workload: B16 H32 N1024
D128 non-causal, Q,K ~ N(0,3^2), V ~ U(-1,1) (the non-causal D=128 shape the
>=60%-of-peak target is stated for).  Its inputs (3 x 128 MiB) and output
exceed the 126 MiB L2, so no explicit flush is needed between steps.

Prints ONE JSON line on rank 0 (``--all``: one line per workload).  Metric:
attention forward TFLOP/s, algorithmic flops 4*B*H*N^2*D (halved under the
causal mask).  Extra objects: ``roofline`` (tensor-bound, against the measured
dense bf16 peak), ``cpu_baseline`` (the fp64 CPU oracle timed on a bounded
sample on this host), ``e2e`` (the same metric through the public API with
pinned host buffers, copies inside the timed region), ``clocks`` (sampled
with nvidia-smi during the timed region) and ``gpu_launches``.

``--bwd``: the same line for the backward pass (tk_attn_bwd; flops
10*B*H*N^2*D, halved under the causal mask), with the fp64 backward oracle as
the CPU baseline.

``--based``: causal Based linear attention (tk_based_fwd, B16 H16 N4096, feature
dim 16, value dim 64), reported as GB/s of algorithmic HBM traffic against the
measured HBM bandwidth (the linear form's arithmetic intensity is below the
ridge).

``--hedgehog``: the same for causal Hedgehog linear attention (tk_hedgehog_fwd,
B8 H16 N4096, query/key dim 64, 64 + 64 softmax features, value dim 64).

``--gemm``: the same line for the GEMM on the same pipeline (tk_gemm,
C = A B^T, M = N = K = 8192 unless ``--gemm-shape M,N,K``; flops 2*M*N*K), with
the fp64 oracle GEMM on sampled rows as the CPU baseline and cuBLAS (through
torch.matmul) timed beside it for context.

``--impl reference``: the comparison arm is the fp64 CPU oracle (there is no
runnable reference implementation), timed on this host's cores on a bounded
sample of the same workload per step.

The forward line also carries ``parity`` (the timed launch's O and LSE
against the fp64 oracle on sampled heads and rows, with the target's bars)
and, for the default workload, ``configs``: kernel time, TFLOP/s, fraction of
peak and parity of the other four workloads, measured in the same process.

Multi-GPU (one rank per GPU; ``--gpus N`` alone re-runs the script under
torchrun): the B*H heads of the one workload are split into contiguous
slices, one per rank, and each rank runs tk_attn_fwd on its slice as a
[1, heads, N, D] problem.  No data-path collective: the step time is the max
over ranks and ``value`` is the whole workload's flops over that time
(strong scaling).  ``--gather`` also times an NCCL all-gather of O and LSE,
reported apart.  The backward, GEMM and linear-attention modes run the full
problem on every rank (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s on 1 GB300 (fraction of dense BF16 peak) vs CPU oracle"
FALLBACK_BF16_TFLOPS = 1900.0  # one earlier GB300 measurement, used only without MEASURED_PEAKS.json
FALLBACK_BF16_SUSTAINED_TFLOPS = 1700.0  # the same measurement held for seconds under the power limit
L2_BYTES = 126 * 1024 * 1024
KERNEL_SOURCES = ["tiled_attention_tk_gb300/csrc/attn_fwd.cu", "tiled_attention_tk_gb300/csrc/tk_ptx.cuh",
                  "tiled_attention_tk_gb300/csrc/tk_sync.cuh"]
DEFAULT_WORKLOAD = 4


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def max_over_ranks(value: float, dist_mod, device=None) -> float:
    """Max of a per-rank float over all ranks (identity on one rank)."""
    if dist_mod is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def peaks(sustained: bool = False):
    """(bf16 TF/s, label) from MEASURED_PEAKS.json (the burst figure, or the
    sustained one for a kernel that runs under the power limit through a
    seconds-long timed region), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            v = d.get("bf16_tflops_sustained" if sustained else "bf16_tflops")
            if isinstance(v, dict):
                v = v.get("value")
            if v:
                return float(v), "of measured sustained" if sustained else "of measured"
        except (OSError, ValueError, TypeError):
            pass
    return (FALLBACK_BF16_SUSTAINED_TFLOPS, "of fallback sustained") if sustained else \
        (FALLBACK_BF16_TFLOPS, "of fallback")


FWD256_SOURCES = ["tiled_attention_tk_gb300/csrc/attn_fwd256.cu", "tiled_attention_tk_gb300/csrc/tk_ptx.cuh",
                  "tiled_attention_tk_gb300/csrc/tk_sync.cuh"]


def traffic_for(workload_name: str, D: int = 128):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the forward kernel that runs head dim D; else
    None."""
    if D == 256:
        return sources_traffic_for(workload_name, FWD256_SOURCES)
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload_name)
        if e and e.get("kernel_source_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError, TypeError):
        pass
    return None


class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the
    driver): SM clock, its maximum and the clock-event reason bits."""

    CLOCK_SM = 1
    # clock-event reason bits, as nvml.h numbers them
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    GPU_IDLE = 0x1

    def __init__(self, uuid: str):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML device for " + uuid)
        try:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        m = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.dev, self.CLOCK_SM, ctypes.byref(m))
        self.max_mhz = float(m.value)

    def sample(self):
        clk, bits = self.c.c_uint(), self.c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, self.CLOCK_SM, self.c.byref(clk)) != 0:
            return None
        if self.reasons_fn(self.dev, self.c.byref(bits)) != 0:
            return None
        return float(clk.value), int(bits.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and clock-event reasons while the timed region runs.

    A host thread queries NVML every ~2 ms between start (the constructor) and
    stop(), so even a timed region of a few milliseconds gets samples; the
    samples also go to the CSV file named by TK_BENCH_CLOCKS_CSV, when set
    (with `<i>` replaced by the GPU index).  Where NVML cannot be loaded it
    falls back to `nvidia-smi --loop-ms`, whose start-up takes longer than
    short timed regions."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 100):
        self.proc = None
        self.nvml = None
        want = os.environ.get("TK_BENCH_CLOCKS_CSV")
        self.keep = bool(want)
        if want:
            self.path = want.replace("<i>", str(gpu_index))
        else:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="tk_clocks_", suffix=".csv")
            os.close(fd)
        gpu_id = str(gpu_index)
        try:  # the UUID names the right GPU whatever CUDA_VISIBLE_DEVICES says
            import torch
            u = str(torch.cuda.get_device_properties(gpu_index).uuid)
            gpu_id = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
        except OSError:
            pass
        try:
            self.nvml = _Nvml(gpu_id)
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            import threading
            self.samples = []
            self.stop_flag = threading.Event()

            def loop():
                while not self.stop_flag.is_set():
                    r = self.nvml.sample()
                    if r is not None:
                        self.samples.append((time.perf_counter(), r[0], r[1]))
                    self.stop_flag.wait(0.002)
            self.first = self.nvml.sample()
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"--loop-ms={interval_ms}"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _stop_nvml(self):
        self.stop_flag.set()
        self.thread.join(timeout=5)
        last = self.nvml.sample()
        self.nvml.close()
        pts = list(self.samples)
        try:
            if self.keep:
                with open(self.path, "w") as f:
                    f.write("t_s,sm_mhz,max_sm_mhz,reason_bits\n")
                    for t, mhz, bits in pts:
                        f.write(f"{t:.6f},{mhz:.0f},{self.nvml.max_mhz:.0f},{bits:#x}\n")
            else:
                os.remove(self.path)
        except OSError:
            pass
        if not pts:
            pts = [(0.0, r[0], r[1]) for r in (self.first, last) if r is not None]
        if not pts:
            return {"sm_mhz": None, "sm_max_mhz": self.nvml.max_mhz, "reasons": ["no samples"], "samples": 0,
                    "source": "nvml"}
        busy = [p for p in pts if not p[2] & _Nvml.GPU_IDLE] or pts
        mhz = sorted(p[1] for p in busy)
        reasons = sorted({name for p in pts for bit, name in _Nvml.REASONS.items() if p[2] & bit})
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": self.nvml.max_mhz, "reasons": reasons,
                "samples": len(pts), "samples_busy": len(busy) if busy is not pts else 0, "source": "nvml"}

    def stop(self):
        if self.nvml is not None:
            return self._stop_nvml()
        if self.proc is None:
            if not self.keep:
                try:
                    os.remove(self.path)
                except OSError:
                    pass
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(n)
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "source": "nvidia-smi"}
        sms.sort()
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms), "source": "nvidia-smi"}


def l2_description(in_bytes: int) -> str:
    """How the timed region treats L2 for inputs of `in_bytes` (the same text
    in both arms' config)."""
    if in_bytes > L2_BYTES:
        return f"inputs {in_bytes / 2**20:.0f} MiB > {L2_BYTES >> 20} MiB L2, no flush"
    return (f"inputs {in_bytes / 2**20:.0f} MiB fit in L2: a {2 * L2_BYTES >> 20} MiB write flushes L2 "
            "before every timed launch (outside its events)")


def l2_flusher(in_bytes: int, dev):
    """(buffer, description): where the timed launch's inputs fit in L2, a
    buffer of twice L2 that is written before every timed launch, outside its
    event pair, so that no launch starts on operands left in L2 by the last."""
    import torch
    if in_bytes > L2_BYTES:
        return None, l2_description(in_bytes)
    buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    return buf, l2_description(in_bytes)


# ---------------------------------------------------------------- CPU oracle timing

def row_flops(w, r: int) -> float:
    """Algorithmic flops of query row r: 4*D per key it sees."""
    keys = min(r + 1 + w.Nkv - w.N, w.Nkv) if w.causal else w.Nkv
    return 4.0 * keys * w.D


def time_oracle_sample(w, q, k, v, budget_s: float, min_rows: int = 64):
    """Times the fp64 oracle on whole heads of the workload, one after another,
    until ``budget_s`` of work has been done (at least ``min_rows`` rows).
    Returns (TFLOP/s, cores, description)."""
    import oracle
    oracle.build()
    done_flops, rows_done, t_total, heads = 0.0, 0, 0.0, 0
    start = time.perf_counter()
    bh_total = w.B * w.H
    while True:
        b, h = divmod(heads % bh_total, w.H)
        # whole head, but at most enough rows to stay near the budget
        remaining = max(budget_s - (time.perf_counter() - start), 0.0)
        rows = list(range(w.N))
        if rows_done and t_total > 0:
            rate = rows_done / t_total
            rows = rows[: max(min_rows, min(w.N, int(rate * remaining)))]
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(q[b, h], k[b, h], v[b, h], rows, w.causal, w.scale)
        dt = time.perf_counter() - t0
        t_total += dt
        done_flops += sum(row_flops(w, r) for r in rows)
        rows_done += len(rows)
        heads += 1
        if time.perf_counter() - start >= budget_s or heads >= bh_total:
            break
    cores = oracle.last_threads()
    desc = (f"{rows_done} query rows of {heads} head(s) of {w.name} "
            f"({done_flops / 1e9:.2f} GFLOP fp64, {t_total:.1f} s)")
    return done_flops / t_total / 1e12, cores, desc


# ---------------------------------------------------------------- our arm

def shard(bh_total: int, world: int, rank: int):
    """(first, count): the contiguous slice of the B*H heads that rank
    `rank` of `world` computes.  The first bh_total % world ranks take one
    head more; every head belongs to exactly one rank."""
    base, extra = divmod(bh_total, world)
    first = rank * base + min(rank, extra)
    return first, base + (1 if rank < extra else 0)


def parity_rows(w, limit: int = 320):
    """Query rows compared with the oracle in one head: all of them for
    short sequences, else the first and last 64, both sides of every fourth
    128-row tile boundary and a seeded draw, `limit` rows at most."""
    if w.N <= limit:
        return list(range(w.N))
    import random
    rows = set(range(64)) | set(range(w.N - 64, w.N))
    for t in range(128, w.N, 512):
        rows.update((t - 1, t))
    rnd = random.Random(1000 * w.index + w.N)
    while len(rows) < limit:
        rows.add(rnd.randrange(w.N))
    return sorted(rows)


def parity_check(w, q, k, v, o, lse, heads, first: int = 0):
    """O and LSE of the given global heads (b*H + h, inside this rank's slice
    that starts at head `first`) against the fp64 oracle on sampled rows.
    Returns the error figures with the pass/fail of the target's bars."""
    import numpy as np
    import oracle
    oracle.build()
    rows = parity_rows(w)
    o_max = o_sum = lse_max = 0.0
    count = 0
    for gh in heads:
        b, h = divmod(gh, w.H)
        O_ref, L_ref = oracle.attn_fwd_rows(q[b, h], k[b, h], v[b, h], rows, w.causal, w.scale)
        o_gpu = o[gh - first][rows].double().cpu().numpy()
        l_gpu = lse[gh - first][rows].double().cpu().numpy()
        e = np.abs(o_gpu - O_ref)
        o_max = max(o_max, float(e.max()))
        o_sum += float(e.sum())
        count += e.size
        lse_max = max(lse_max, float(np.abs(l_gpu - L_ref).max()))
    o_mean = o_sum / max(count, 1)
    return {"heads": len(heads), "rows_per_head": len(rows), "o_max": float(f"{o_max:.3e}"),
            "o_mean": float(f"{o_mean:.3e}"), "lse_max": float(f"{lse_max:.3e}"),
            "ok": bool(o_max <= 2e-2 and o_mean <= 2e-3 and lse_max <= 1e-3)}


def parity_heads(first: int, count: int, n: int = 4, seed: int = 11):
    """Up to n global heads of the slice [first, first+count): its first and
    last head and a seeded draw of the rest."""
    if count <= 0:
        return []
    if count <= n:
        return list(range(first, first + count))
    import random
    chosen = {first, first + count - 1}
    rnd = random.Random(seed + first)
    while len(chosen) < n:
        chosen.add(first + rnd.randrange(count))
    return sorted(chosen)


class ForwardRun:
    """One workload on this rank: its slice of the heads resident on the
    device, and the launch of tk_attn_fwd_ws over that slice as one
    [1, count, N, D] problem (with its workspace when the shape's last round
    of work units is split by key tiles)."""

    def __init__(self, w, dev, ws: int, rank: int):
        import torch
        from tiled_attention_tk_gb300.inputs import workload_inputs
        self.w = w
        self.first, self.count = shard(w.B * w.H, ws, rank)
        q, k, v = workload_inputs(w)
        self.q, self.k, self.v = q, k, v
        sl = slice(self.first, self.first + self.count)
        self.qd = q.reshape(w.B * w.H, w.N, w.D)[sl].to(dev)
        self.kd = k.reshape(w.B * w.H, w.Nkv, w.D)[sl].to(dev)
        self.vd = v.reshape(w.B * w.H, w.Nkv, w.D)[sl].to(dev)
        self.o = torch.empty_like(self.qd)
        self.lse = torch.empty((self.count, w.N), dtype=torch.float32, device=dev)
        self.in_bytes = self.count * (w.N + 2 * w.Nkv) * w.D * 2
        import tiled_attention_tk_gb300 as tk
        with torch.cuda.device(dev):
            self.ws_bytes = tk.fwd_workspace_bytes(1, self.count, w.N, w.Nkv, w.D, w.causal) if self.count else 0
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev) if self.ws_bytes else None

    def launch(self, stream_handle: int):
        import tiled_attention_tk_gb300 as tk
        w = self.w
        if self.count == 0:
            return
        ptrs = (self.qd.data_ptr(), self.kd.data_ptr(), self.vd.data_ptr(), self.o.data_ptr(), self.lse.data_ptr())
        tk.fwd_ws_raw(*ptrs, self.ws.data_ptr() if self.ws is not None else None, self.ws_bytes, 1, self.count,
                      w.N, w.Nkv, w.D, w.causal, w.scale, stream_handle)


def time_launches(run, steps: int, warmup: int, dev, stream, flush, dist_mod):
    """Warm-up, then `steps` timed launches, each in its own event pair, with
    the whole region in one more pair.  Returns (total ms of the region, mean
    ms per launch, {median, min, max} ms per launch); with an L2 flush between
    launches the region's time is the sum of the launches' own times."""
    import torch
    import tiled_attention_tk_gb300 as tk
    sh = int(stream.cuda_stream)
    for _ in range(warmup):
        run.launch(sh)
    torch.cuda.synchronize(dev)
    st, detail = tk.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) after warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start_ev, end_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist_mod:
        dist_mod.barrier()
    torch.cuda.synchronize(dev)
    start_ev.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        run.launch(sh)
        ev[i][1].record(stream)
    end_ev.record(stream)
    torch.cuda.synchronize(dev)
    if dist_mod:
        dist_mod.barrier()
    st, detail = tk.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) after timing")
    per_launch = sorted(a.elapsed_time(b) for a, b in ev)
    kernel_ms = sum(per_launch) / steps
    total_ms = kernel_ms * steps if flush is not None else start_ev.elapsed_time(end_ev)
    mid = steps // 2
    median = per_launch[mid] if steps % 2 else 0.5 * (per_launch[mid - 1] + per_launch[mid])
    stats = {"median": round(median, 5), "min": round(per_launch[0], 5), "max": round(per_launch[-1], 5)}
    return total_ms, kernel_ms, stats


# Workloads measured beside the default line (kernel time, TFLOP/s, fraction
# of peak, parity on sampled heads) within the same process.
SIDE_WORKLOADS = (1, 2, 3, 5)


def measure_side_configs(args, dev, stream, dist_mod, ws, rank, peak):
    import torch
    from tiled_attention_tk_gb300.inputs import WORKLOADS
    out = {}
    for idx in SIDE_WORKLOADS:
        w = WORKLOADS[idx]
        run = ForwardRun(w, dev, ws, rank)
        flush, _ = l2_flusher(max(run.in_bytes, 1), dev)
        steps = 200 if w.flops < 1e10 else 20
        _, kernel_ms, _ = time_launches(run, steps, 3, dev, stream, flush, dist_mod)
        kernel_ms = max_over_ranks(kernel_ms, dist_mod, dev)
        tf = w.flops / (kernel_ms * 1e-3) / 1e12
        entry = {"kernel_ms": round(kernel_ms, 5), "tflops": round(tf, 2), "frac": round(tf / peak, 4),
                 "l2_flush": flush is not None}
        if rank == 0 and not args.no_parity:
            entry["parity"] = parity_check(w, run.q, run.k, run.v, run.o, run.lse,
                                           parity_heads(run.first, run.count, 2), run.first)
        out[w.name] = entry
        del run, flush
        torch.cuda.empty_cache()
    return out


def run_ours(args, w):
    import torch
    import tiled_attention_tk_gb300 as tk

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_mod = init_dist(ws, "nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    run = ForwardRun(w, dev, ws, rank)
    flush, l2_desc = l2_flusher(max(run.in_bytes, 1), dev)
    sampler = ClockSampler(local)
    total_ms, kernel_ms, launch_stats = time_launches(run, args.steps, args.warmup, dev, stream, flush, dist_mod)
    clocks = sampler.stop()
    total_ms = max_over_ranks(total_ms, dist_mod, dev)
    ms_per_step = total_ms / args.steps
    # strong scaling: the ranks share one workload, so the whole workload's
    # flops count once against the slowest rank's time
    value = w.flops / (ms_per_step * 1e-3) / 1e12

    parity = None
    if rank == 0 and not args.no_parity:
        parity = parity_check(w, run.q, run.k, run.v, run.o, run.lse, parity_heads(run.first, run.count),
                              run.first)

    # ---- optional all-gather of every rank's O and LSE to all ranks (NCCL),
    # timed on its own: the forward itself needs no exchange
    gather = None
    if dist_mod is not None and args.gather:
        base, extra = divmod(w.B * w.H, ws)
        cnt = base + (1 if extra else 0)  # the largest slice; smaller ones are padded
        o_pad = torch.zeros((cnt, w.N, w.D), dtype=torch.bfloat16, device=dev)
        l_pad = torch.zeros((cnt, w.N), dtype=torch.float32, device=dev)
        o_pad[:run.count].copy_(run.o)
        l_pad[:run.count].copy_(run.lse)
        o_all = [torch.empty_like(o_pad) for _ in range(ws)]
        l_all = [torch.empty_like(l_pad) for _ in range(ws)]
        dist_mod.all_gather(o_all, o_pad)
        dist_mod.all_gather(l_all, l_pad)
        torch.cuda.synchronize(dev)
        dist_mod.barrier()
        t0 = time.perf_counter()
        for _ in range(5):
            dist_mod.all_gather(o_all, o_pad)
            dist_mod.all_gather(l_all, l_pad)
        torch.cuda.synchronize(dev)
        g_ms = max_over_ranks((time.perf_counter() - t0) / 5 * 1e3, dist_mod, dev)
        gather = {"ms_per_step": round(g_ms, 4), "bytes_per_rank": (o_pad.numel() * 2 + l_pad.numel() * 4),
                  "collective": "all_gather (NCCL) of O and LSE"}

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        sl = slice(run.first, run.first + run.count)
        qh = run.q.reshape(w.B * w.H, w.N, w.D)[sl].reshape(1, run.count, w.N, w.D).pin_memory()
        kh = run.k.reshape(w.B * w.H, w.Nkv, w.D)[sl].reshape(1, run.count, w.Nkv, w.D).pin_memory()
        vh = run.v.reshape(w.B * w.H, w.Nkv, w.D)[sl].reshape(1, run.count, w.Nkv, w.D).pin_memory()
        e2e_steps = max(3, min(20, args.steps // 50))
        if run.count:
            tk.fwd(qh, kh, vh, causal=w.causal, scale=w.scale)  # warm
        if dist_mod:
            dist_mod.barrier()
        t0 = time.perf_counter()
        oh = lh = None
        for _ in range(e2e_steps):
            if run.count:
                oh, lh = tk.fwd(qh, kh, vh, causal=w.causal, scale=w.scale)
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e_s = max_over_ranks(e2e_s, dist_mod, dev)
        h2d = (qh.numel() + kh.numel() + vh.numel()) * qh.element_size()
        d2h = (oh.numel() * oh.element_size() + lh.numel() * lh.element_size()) if oh is not None else 0
        e2e = {"value": round(w.flops / e2e_s / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_s * 1e3, 3), "steps": e2e_steps,
               "path": "tk.fwd on pinned host tensors: heads in chunks over two streams, copies in and out "
                       "overlapping the kernels"}

    peak, peak_label = peaks()
    side = None
    if args.side_configs and not args.all and not args.shape:
        side = measure_side_configs(args, dev, stream, dist_mod, ws, rank, peak)

    if rank != 0:
        if dist_mod:
            dist_mod.barrier()
        return None
    achieved = w.flops * (run.count / (w.B * w.H)) / (kernel_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded torch.Generator, fp32 draws rounded to bf16)",
        "config": dict(w.describe(), l2=l2_description(w.B * w.H * (w.N + 2 * w.Nkv) * w.D * 2),
                       tail_split=bool(run.ws_bytes)),
        "sharding": {"ranks": ws, "heads": w.B * w.H,
                     "rule": "rank r computes a contiguous slice of the B*H heads (the first B*H % ranks "
                             "ranks one head more); no data-path collective",
                     "rank0_heads": [run.first, run.first + run.count]},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": peak_label, "traffic": traffic_for(w.name, w.D) if ws == 1 else None,
                     "kernel": f"attn_fwd_kernel<{w.D}>" if w.D != 256 else f"attn_fwd256_kernel<256, {str(bool(w.causal)).lower()}>",
                     "kernel_ms": round(kernel_ms, 5)},
        "launch_ms": launch_stats,  # this rank's per-launch CUDA-event times
        "parity": parity,
        "e2e": e2e,
        "gpu_launches": args.steps if run.count else 0,
        "clocks": clocks,
    }
    if side is not None:
        line["configs"] = side
    if gather is not None:
        line["gather"] = gather
    if not args.no_cpu_baseline:
        tf, cores, desc = time_oracle_sample(w, run.q, run.k, run.v, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores,
                                "kind": "oracle", "sample": desc}
    if dist_mod:
        dist_mod.barrier()
    return line


# ---------------------------------------------------------------- backward

BWD_METRIC = "attention bwd TFLOP/s on 1 GB300 (fraction of dense BF16 peak) vs CPU oracle"


def time_oracle_bwd_sample(w, q, k, v, do, budget_s: float):
    """The fp64 backward oracle on whole heads until ``budget_s`` is spent.
    Returns (TFLOP/s, cores, description); flops counted as 10*N^2*D per head
    (halved under the causal mask), the same count as the GPU line."""
    import oracle
    oracle.build()
    per_head = 10.0 * w.N * w.N * w.D / (2.0 if w.causal else 1.0)
    done, t_total, heads = 0.0, 0.0, 0
    while heads < w.B * w.H:
        b, h = divmod(heads, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        t0 = time.perf_counter()
        oracle.attn_bwd(q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous(), do[sl].contiguous(),
                        w.causal, w.scale)
        t_total += time.perf_counter() - t0
        done += per_head
        heads += 1
        if t_total >= budget_s:
            break
    return (done / t_total / 1e12, oracle.last_threads(),
            f"{heads} head(s) of {w.name} ({done / 1e9:.1f} GFLOP fp64, {t_total:.1f} s)")


def run_bwd(args, w):
    """One step = tk_attn_bwd over the whole workload (three launches: row
    values, main kernel, dQ rounding), inputs and forward outputs resident."""
    import torch
    import tiled_attention_tk_gb300 as tk
    from tiled_attention_tk_gb300.inputs import make_qkv, workload_inputs

    _, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v = workload_inputs(w)
    do = make_qkv(w.B, w.H, w.N, w.D, 1000 * w.index + 500, "normal")[0]
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, do))
    o, lse = tk.fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    ws = torch.empty(tk.bwd_workspace_bytes(w.B, w.H, w.N, w.D), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return tk.bwd(qd, kd, vd, o, lse, gd, causal=w.causal, scale=w.scale, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, detail = tk.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) after warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    flush, l2_desc = l2_flusher(w.B * w.H * (3 * w.N + 2 * w.Nkv) * w.D * 2, dev)
    sampler = ClockSampler(local)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    st, detail = tk.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) after timing")
    flops = 2.5 * w.flops
    peak, peak_label = peaks()
    achieved = flops / (step_ms * 1e-3) / 1e12
    line = {
        "metric": BWD_METRIC, "value": round(achieved, 2), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded torch.Generator, fp32 draws rounded to bf16)",
        "config": dict(w.describe(), flops="10*B*H*N^2*D (halved causal): S, dP, dV, dK, dQ", l2=l2_desc),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_label, "traffic": None,
                     "kernel": f"attn_bwd_kernel<{w.D}> + prep + dQ rounding (whole step)"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        tf, cores, desc = time_oracle_bwd_sample(w, q, k, v, do, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    return line


# ---------------------------------------------------------------- GEMM

GEMM_METRIC = "GEMM bf16 TFLOP/s on 1 GB300 (C = A B^T, fp32 accumulate; fraction of dense BF16 peak) vs CPU oracle"
GEMM_SOURCES = ["tiled_attention_tk_gb300/csrc/gemm.cu", "tiled_attention_tk_gb300/csrc/tk_ptx.cuh",
                "tiled_attention_tk_gb300/csrc/tk_ptx_pair.cuh", "tiled_attention_tk_gb300/csrc/tk_sync.cuh"]


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def gemm_inputs(M: int, N: int, K: int):
    """Seeded bf16 A [M,K] and B [N,K] on the host (N(0,1) draws rounded to bf16)."""
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(7000)
    a = torch.randn((M, K), generator=g, dtype=torch.float32).to(torch.bfloat16)
    g.manual_seed(7001)
    b = torch.randn((N, K), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return a, b


def time_oracle_gemm_sample(a, b, budget_s: float):
    """The fp64 oracle GEMM on rows of C until ``budget_s`` is spent."""
    import oracle
    oracle.build()
    M, K = a.shape
    N = b.shape[0]
    rows_done, t_total, start = 0, 0.0, time.perf_counter()
    chunk = 8
    while time.perf_counter() - start < budget_s and rows_done < M:
        rows = list(range(rows_done, min(M, rows_done + chunk)))
        t0 = time.perf_counter()
        oracle.gemm(a, b, True, rows=rows)
        t_total += time.perf_counter() - t0
        rows_done += len(rows)
        chunk = min(chunk * 2, 256)
    flops = 2.0 * rows_done * N * K
    return flops / t_total / 1e12, oracle.last_threads(), (
        f"{rows_done} of {M} rows of C ({flops / 1e9:.1f} GFLOP fp64, {t_total:.1f} s)")


def run_gemm(args):
    import torch
    import tiled_attention_tk_gb300 as tk
    M, N, K = (int(x) for x in args.gemm_shape.split(","))
    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_mod = init_dist(ws_n, "nccl")
    dev = torch.device("cuda", local)
    a, b = gemm_inputs(M, N, K)
    ad, bd = a.to(dev), b.to(dev)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    need = tk.gemm_workspace_bytes(M, N, K, True)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        tk.gemm(ad, bd, b_kmajor=True, stream_k=True, out=c, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, detail = tk.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) after warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start_ev, end_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush, l2_desc = l2_flusher((M + N) * K * 2, dev)
    sampler = ClockSampler(local)
    if dist_mod:
        dist_mod.barrier()
    torch.cuda.synchronize(dev)
    start_ev.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    end_ev.record(stream)
    torch.cuda.synchronize(dev)
    if dist_mod:
        dist_mod.barrier()
    clocks = sampler.stop()
    kernel_ms = sum(x.elapsed_time(y) for x, y in ev) / args.steps
    total_ms = max_over_ranks(start_ev.elapsed_time(end_ev) if flush is None else kernel_ms * args.steps,
                              dist_mod, dev)
    st, detail = tk.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) after timing")
    flops = 2.0 * M * N * K
    ms_per_step = total_ms / args.steps
    value = flops * ws_n / (ms_per_step * 1e-3) / 1e12

    # cuBLAS on the same operands, for context (not the target, not a bench value)
    bt = bd.t()
    for _ in range(3):
        torch.matmul(ad, bt, out=c)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        torch.matmul(ad, bt, out=c)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    cublas = flops / (e0.elapsed_time(e1) / args.steps * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        ah, bh = a.pin_memory(), b.pin_memory()
        ch = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
        steps = max(3, min(10, args.steps // 10))

        def e2e_step():
            with torch.cuda.stream(stream):
                ad.copy_(ah, non_blocking=True)
                bd.copy_(bh, non_blocking=True)
                tk.gemm(ad, bd, b_kmajor=True, stream_k=True, out=c, workspace=ws, stream=stream)
                ch.copy_(c, non_blocking=True)
            stream.synchronize()
        e2e_step()
        t0 = time.perf_counter()
        for _ in range(steps):
            e2e_step()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / steps, dist_mod, dev)
        e2e = {"value": round(flops * ws_n / e2e_s / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": (a.numel() + b.numel()) * 2, "d2h_bytes_per_step": M * N * 2,
               "ms_per_step": round(e2e_s * 1e3, 3), "steps": steps}
    if rank != 0:
        return None
    # A GEMM of this size runs the GPU into its power limit (sw_power_cap, SM
    # clock well below maximum) over a timed region of about a second and a
    # half: the sustained measured peak is its denominator; the burst one is
    # reported beside it.
    peak, peak_label = peaks(sustained=True)
    burst, _ = peaks()
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    name = f"gemm-M{M}N{N}K{K}"
    pairs = tk.gemm_uses_pairs(M, N, K, True)
    line = {
        "metric": GEMM_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded torch.Generator, N(0,1) fp32 draws rounded to bf16)",
        "config": {"workload": name, "M": M, "N": N, "K": K, "b_layout": "[N,K] (C = A B^T)",
                   "stream_k": "on where the schedule uses it",
                   "cta_pairs": pairs,
                   "workspace_bytes": need,
                   "l2": l2_desc},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_label,
                     "peak_burst": burst, "frac_of_burst": round(achieved / burst, 4),
                     "traffic": gemm_traffic_for(name),
                     "kernel": "gemm_pair_kernel<true>" if pairs else "gemm_kernel<true>",
                     "kernel_ms": round(kernel_ms, 5)},
        "cublas_context_tflops": round(cublas, 2),
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        tf, cores, desc = time_oracle_gemm_sample(a, b, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    return line


def gemm_traffic_for(name: str):
    return sources_traffic_for(name, GEMM_SOURCES)


def sources_traffic_for(name: str, sources):
    """DRAM bytes per launch recorded in profiles/traffic.json for workload
    `name`, if taken on the current source of the kernel's files; else None."""
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            e = json.load(f).get(name)
        if e and e.get("kernel_source_hash") == h.hexdigest()[:16]:
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError, TypeError, AttributeError):
        pass
    return None


def run_reference_gemm(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None
    M, N, K = (int(x) for x in args.gemm_shape.split(","))
    a, b = gemm_inputs(M, N, K)
    tf, cores, desc = time_oracle_gemm_sample(a, b, budget_s=args.reference_budget)
    return {"impl": "reference", "metric": GEMM_METRIC, "value": round(tf, 6), "unit": "TFLOP/s",
            "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"gemm-M{M}N{N}K{K}", "M": M, "N": N, "K": K},
            "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": desc, "value": round(tf, 6)},
            "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- Based linear attention

BASED_METRIC = ("Based linear attention GB/s of algorithmic HBM traffic on 1 GB300 "
                "(fraction of measured HBM bandwidth) vs CPU oracle")
BASED_SOURCES = ["tiled_attention_tk_gb300/csrc/based.cu", "tiled_attention_tk_gb300/csrc/tk_ptx.cuh",
                 "tiled_attention_tk_gb300/csrc/tk_sync.cuh"]


def hbm_peak():
    """(HBM GB/s, label) from MEASURED_PEAKS.json, else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = json.load(f).get("hbm_gbs")
        if isinstance(v, dict):
            v = v.get("value")
        if v:
            return float(v), "of measured"
    except (OSError, ValueError, TypeError):
        pass
    return 6800.0, "of fallback"


def based_inputs(B, H, N):
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(8000)
    q = torch.randn((B, H, N, 16), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, N, 16), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, N, 64), generator=g).to(torch.bfloat16)
    return q, k, v


HEDGEHOG_METRIC = ("Hedgehog linear attention GB/s of algorithmic HBM traffic on 1 GB300 "
                   "(fraction of measured HBM bandwidth) vs CPU oracle")
HEDGEHOG_SOURCES = ["tiled_attention_tk_gb300/csrc/hedgehog.cu", "tiled_attention_tk_gb300/csrc/tk_ptx.cuh",
                    "tiled_attention_tk_gb300/csrc/tk_sync.cuh"]


def hedgehog_inputs(B, H, N):
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(8100)
    q = torch.randn((B, H, N, 64), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, N, 64), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, N, 64), generator=g).to(torch.bfloat16)
    wq = (torch.randn((H, 64, 64), generator=g) * 0.2).to(torch.bfloat16)
    wk = (torch.randn((H, 64, 64), generator=g) * 0.2).to(torch.bfloat16)
    return q, k, v, wq, wk


def run_based(args, kind: str = "based"):
    """One step = tk_based_fwd over B16 H16 N4096 (tk_hedgehog_fwd over B8 H16
    N4096; both read 192 MiB of inputs, more than L2) unless
    --based-shape B,H,N.  Value: algorithmic bytes (Q, K, V read once, O and
    DEN written once) per second; the chunked linear form's flops are reported
    beside it."""
    import torch
    import tiled_attention_tk_gb300 as tk
    shape = args.based_shape or ("8,16,4096" if kind == "hedgehog" else "16,16,4096")
    B, H, N = (int(x) for x in shape.split(","))
    _, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hh = kind == "hedgehog"
    if hh:
        q, k, v, wq, wk = hedgehog_inputs(B, H, N)
        wqd, wkd = wq.to(dev), wk.to(dev)
    else:
        q, k, v = based_inputs(B, H, N)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty((B, H, N, 64), dtype=torch.bfloat16, device=dev)
    den = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if hh:
            tk.hedgehog(qd, kd, vd, wqd, wkd, out=o, den=den, stream=stream)
        else:
            tk.based(qd, kd, vd, scale=0.25, out=o, den=den, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    dqk = 64 if hh else 16
    flush, l2_desc = l2_flusher(B * H * N * (2 * dqk + 64) * 2, dev)
    sampler = ClockSampler(local)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = sum(x.elapsed_time(y) for x, y in ev) / args.steps
    st, detail = tk.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) after timing")
    tokens = B * H * N
    alg_bytes = tokens * (dqk * 2 + dqk * 2 + 64 * 2 + 64 * 2 + 4) + (2 * H * 64 * 64 * 2 if hh else 0)
    # chunked linear form per token: in-chunk phi(Q) phi(K)^T (Hedgehog, after
    # the two 64 x 64 projections) or Q K^T (Based) and P [V|1] over the
    # causal half of 128 rows; carried phi(Q) S and the state update
    # [V|1]^T phi(K) (features x 65)
    nf = 128 if hh else 153
    flops = tokens * ((2 * 2 * 64 * 64 if hh else 0) + 2 * (nf if hh else 16) * 64 + 2 * 65 * 64 +
                      2 * (2 * nf * 65))
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    peak, label = hbm_peak()
    if rank != 0:
        return None
    line = {
        "metric": HEDGEHOG_METRIC if hh else BASED_METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded torch.Generator, N(0,1) fp32 draws rounded to bf16)",
        "config": {"workload": f"{kind}-B{B}H{H}N{N}", "B": B, "H": H, "N": N, "Dqk": dqk, "Dv": 64,
                   **({"F": 64, "W": "N(0,0.2^2) per head"} if hh else {"scale": 0.25}),
                   "causal": True, "alg_bytes": alg_bytes,
                   "l2": l2_desc},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_source": label,
                     "traffic": sources_traffic_for(f"{kind}-B{B}H{H}N{N}",
                                                    HEDGEHOG_SOURCES if hh else BASED_SOURCES),
                     "kernel": f"{kind}_kernel", "kernel_ms": round(ms, 5)},
        "linear_form_tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "tokens_per_s": round(tokens / (ms * 1e-3), 1),
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        t_total, rows_done, heads = 0.0, 0, 0
        start = time.perf_counter()
        while time.perf_counter() - start < args.cpu_budget and heads < B * H:
            b, h = divmod(heads, H)
            rows = list(range(N - 256, N))  # the longest rows of the head
            t0 = time.perf_counter()
            if hh:
                oracle.hedgehog(q[b, h], k[b, h], v[b, h], wq[h], wk[h], rows=rows)
            else:
                oracle.based(q[b, h], k[b, h], v[b, h], 0.25, rows=rows)
            t_total += time.perf_counter() - t0
            rows_done += len(rows)
            heads += 1
        # the quadratic form reads every earlier key once per row: bytes of the
        # rows' own inputs/outputs, scaled to the workload by rows
        cpu_gbs = rows_done * (alg_bytes / tokens) / t_total / 1e9
        line["cpu_baseline"] = {"value": round(cpu_gbs, 6), "unit": "GB/s", "cores": oracle.last_threads(),
                                "kind": "oracle",
                                "sample": f"the last 256 rows of {heads} head(s), quadratic form in fp64 "
                                          f"({t_total:.1f} s)"}
    return line


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    from tiled_attention_tk_gb300.inputs import workload_inputs
    oracle.build()
    q, k, v = workload_inputs(w)
    # Rows per step: sized from a measured rate so K steps take ~budget seconds.
    probe_rows = list(range(min(w.N, 64)))
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(q[0, 0], k[0, 0], v[0, 0], probe_rows, w.causal, w.scale)
    rate = len(probe_rows) / max(time.perf_counter() - t0, 1e-6)
    rows_per_step = int(max(8, min(w.N, rate * args.reference_budget / max(1, args.steps + args.warmup))))

    def step(i):
        bh = i % (w.B * w.H)
        b, h = divmod(bh, w.H)
        start = (i * rows_per_step) % w.N
        rows = [(start + r) % w.N for r in range(rows_per_step)]
        oracle.attn_fwd_rows(q[b, h], k[b, h], v[b, h], rows, w.causal, w.scale)
        return sum(row_flops(w, r) for r in rows)

    for i in range(args.warmup):
        step(i)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    cores = oracle.last_threads()
    sample = (f"{rows_per_step} query rows of one (b,h) head of {w.name} per step "
              f"(a 1/{w.B * w.H * w.N / rows_per_step:.0f} share of the workload), fp64")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded torch.Generator, fp32 draws rounded to bf16)",
        "config": dict(w.describe(), l2=l2_description(w.B * w.H * (w.N + 2 * w.Nkv) * w.D * 2)),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def relaunch_cmd(n: int, argv, port: int):
    """The torchrun command that runs this script as n ranks on one node."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]


def relaunch_ranks(n: int, argv) -> int:
    """Runs the benchmark as n ranks (rank 0 prints the line) and returns
    their exit status."""
    return subprocess.call(relaunch_cmd(n, argv, free_port()))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    from tiled_attention_tk_gb300.inputs import WORKLOADS, Workload
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--all", action="store_true", help="one line per workload")
    ap.add_argument("--shape", type=str, default=None,
                    help="B,H,N,D,causal[,Nkv]: a custom N(0,1) workload instead of a named one")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--bwd", action="store_true", help="time the backward pass instead of the forward")
    ap.add_argument("--gemm", action="store_true", help="time the GEMM on the same pipeline instead")
    ap.add_argument("--gemm-shape", type=str, default="8192,8192,8192", help="M,N,K for --gemm")
    ap.add_argument("--based", action="store_true", help="time the Based linear attention instead")
    ap.add_argument("--hedgehog", action="store_true", help="time the Hedgehog linear attention instead")
    ap.add_argument("--based-shape", type=str, default=None,
                    help="B,H,N for --based (default 16,16,4096) / --hedgehog (default 8,16,4096)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--reference-budget", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the check of the timed launch's O/LSE against the oracle on sampled heads")
    ap.add_argument("--no-side-configs", dest="side_configs", action="store_false",
                    help="skip the other workloads measured beside the default line")
    ap.add_argument("--gather", action="store_true",
                    help="under several ranks, also time an all-gather of every rank's O and LSE")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, _ = dist_env()
    if ws != args.gpus and ws != 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={ws}")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: start the ranks under torchrun, same arguments
        sys.exit(relaunch_ranks(args.gpus, sys.argv[1:] if argv is None else list(argv)))

    if args.shape:
        f = [int(x) for x in args.shape.split(",")]
        if len(f) not in (5, 6):
            ap.error("--shape wants B,H,N,D,causal[,Nkv]")
        todo = [Workload(0, f[0], f[1], f[2], f[3], bool(f[4]), "normal", f[5] if len(f) == 6 else None)]
    else:
        todo = [WORKLOADS[i] for i in (sorted(WORKLOADS) if args.all else [args.workload])]
    if args.based or args.hedgehog:
        line = run_based(args, "hedgehog" if args.hedgehog else "based")
        if line is not None and rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.gemm:
        line = run_reference_gemm(args) if args.impl == "reference" else run_gemm(args)
        if line is not None and rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.bwd:
        todo = [w for w in todo if w.Nkv == w.N]  # the backward takes Nq = Nkv only
    for w in todo:
        if args.impl == "reference":
            line = run_reference(args, w)
        elif args.bwd:
            line = run_bwd(args, w)
        else:
            line = run_ours(args, w)
        if line is not None and rank == 0:
            print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
