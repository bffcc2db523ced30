#!/usr/bin/env python
"""Benchmark of the GDN speculative-verify round on GB300; prints ONE JSON line.

Workload (one step): the shared verify round of one GDN layer with 27B-like
heads (Hk=16 key heads, Hv=48 value heads, d_k=d_v=128): 16 streams x 16-row
chain windows (256 rows), every row's fp32 state and conv tail recorded
(gdn_window), then each stream's random accepted length 0..16 committed
(gdn_commit).  Inputs are seeded synthetic tensors resident in HBM; L2 is
flushed (a 256 MiB write) between timed steps, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one rank per GPU, each rank on its own round
(weak scaling, no collective on the data path); rank 0 prints the line with
the max-over-ranks time.  --impl reference times the CPU oracle (the plain
sequential definition) on the host cores instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_deltanet_speculative_gb300 import synth  # noqa: E402

METRIC = "GDN verify rows/s (16 streams×16 rows); state HBM GB/s vs GB300 peak"
GEOM = synth.LIKE_27B
N_STREAMS, WINDOW = 16, 16
SEED = 2
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("verify round, one GDN layer: 16 streams x 16-row chain windows (256 rows), 27B-like heads "
            "(Hk=16, Hv=48, d_k=d_v=128), every row's fp32 state and conv tail recorded, then a random "
            "accepted length 0..16 per stream committed")


# ---- algorithmic bytes (each byte the round must move at least once) ------

def window_bytes(g: synth.Geometry, n_streams: int, n_rows: int) -> int:
    tile = g.d_v * g.d_k * 4
    state_in = n_streams * g.n_v_heads * tile                 # committed slot tiles, read once
    rec_state = n_rows * g.n_v_heads * tile                   # every row's state, written once
    tail_in = n_streams * 3 * g.channels * 2                  # committed conv tails
    rec_tail = n_rows * 3 * g.channels * 2                    # every row's conv tail
    acts = n_rows * (g.channels + g.n_v_heads * g.d_v + 2 * g.n_v_heads) * 2   # mixed, z, a, b
    y = n_rows * g.n_v_heads * g.d_v * 2
    weights = g.channels * 4 * 2 + g.n_v_heads * 8 + g.d_v * 2
    return state_in + rec_state + tail_in + rec_tail + acts + y + weights


def commit_bytes(g: synth.Geometry, n_committed: int) -> int:
    return n_committed * 2 * (g.n_v_heads * g.d_v * g.d_k * 4 + 3 * g.channels * 2)


def source_digest() -> str:
    """sha256 of the window kernel's sources (ties ncu counters to a kernel version)."""
    csrc = os.path.join(ROOT, "gated_deltanet_speculative_gb300", "csrc")
    h = hashlib.sha256()
    for fn in ("gdn_common.cuh", "gdn_rows.cuh", "gdn_launch.h", "gdn_rows_d128.cu"):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_profile: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", kernel_profile)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_digest") != source_digest():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---- clocks during the timed region --------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={device_id}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t0 <= ts <= t1]
        window = "timed"
        if len(inside) < 3:
            inside = [p for _, p in rows]
            window = "warmup+timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(inside[0][2]),
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


def nvsmi_id(local_rank: int) -> str:
    """nvidia-smi's name for this CUDA device (its UUID when torch has it)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[local_rank] if vis else str(local_rank)


# ---- our arm ---------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import gated_deltanet_speculative_gb300 as gdn

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    g = GEOM
    R = N_STREAMS * WINDOW
    seed = SEED + 1000 * rank
    w = synth.layer_weights(g, seed)
    cache = synth.slot_cache(g, N_STREAMS, seed)
    rows = synth.row_inputs(g, R, seed)
    rp = synth.row_ptr([WINDOW] * N_STREAMS)
    rng = np.random.default_rng([seed, 7])
    acc = synth.accepted_lengths(N_STREAMS, WINDOW, rng)
    keep = np.where(acc > 0, rp[:-1] + acc - 1, -1).astype(np.int32)
    slots = np.arange(N_STREAMS, dtype=np.int32)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)

    d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    dw = {"conv_w": bf(w["conv_w"]).to(dev), "A_log": torch.from_numpy(w["A_log"]).to(dev),
          "dt_bias": torch.from_numpy(w["dt_bias"]).to(dev), "norm_w": bf(w["norm_w"]).to(dev)}
    dc = {"state": torch.from_numpy(cache["state"]).to(dev), "tail": bf(cache["tail"]).to(dev)}
    host_in = {k: bf(rows[k]).pin_memory() for k in ("mixed", "z", "a", "b")}
    dr = {k: v.to(dev) for k, v in host_in.items()}
    dr["y"] = torch.empty((R, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device=dev)
    host_keep = torch.from_numpy(keep).pin_memory()
    host_y = torch.empty_like(dr["y"], device="cpu").pin_memory()
    slot_t = torch.from_numpy(slots).to(dev)
    rp_t = torch.from_numpy(rp).to(dev)
    keep_t = host_keep.to(dev)
    rec_state = torch.empty((R, g.n_v_heads, g.d_v, g.d_k), dtype=torch.float32, device=dev)
    rec_tail = torch.empty((R, 3, g.channels), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        gdn.window(d, dw, dc, slot_t, rp_t, dr, rec_state, rec_tail, stream)
        gdn.commit(d, dc, slot_t, keep_t, rec_state, rec_tail, stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(nvsmi_id(local_rank)) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.fill_(i & 0xff)
        ev[i][0].record(stream)
        gdn.window(d, dw, dc, slot_t, rp_t, dr, rec_state, rec_tail, stream)
        ev[i][1].record(stream)
        gdn.commit(d, dc, slot_t, keep_t, rec_state, rec_tail, stream)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    win_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    com_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    step_ms = sum(a + b for a, b in zip(win_ms, com_ms)) / K

    # end to end through the public API: host inputs in, y back out, each step
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xff)
        ev2[i][0].record(stream)
        for k in ("mixed", "z", "a", "b"):
            dr[k].copy_(host_in[k], non_blocking=True)
        keep_t.copy_(host_keep, non_blocking=True)
        step()
        host_y.copy_(dr["y"], non_blocking=True)
        ev2[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    t2 = time.time()
    if sampler:
        sampler.stop()
    e2e_ms = sum(ev2[i][0].elapsed_time(ev2[i][1]) for i in range(K)) / K
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error word set during the timed steps")

    if world > 1:
        t = torch.tensor([step_ms, e2e_ms, statistics.mean(win_ms)], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        step_ms, e2e_ms, win_avg = t.tolist()
    else:
        win_avg = statistics.mean(win_ms)
    if rank != 0:
        return None

    n_committed = int((keep >= 0).sum())
    wbytes = window_bytes(g, N_STREAMS, R)
    peak, peak_src = hbm_peak()
    achieved = wbytes / (win_avg * 1e-3) / 1e9
    h2d = sum(host_in[k].numel() * 2 for k in host_in) + host_keep.numel() * 4
    d2h = host_y.numel() * 2
    line = {
        "metric": METRIC,
        "value": world * R / (step_ms * 1e-3),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64: bf16 activations N(0,1), fp32 states N(0,0.05))",
        "config": {"workload": WORKLOAD, "streams": N_STREAMS, "rows": R, "layers": 1,
                   "heads": {"Hk": g.n_k_heads, "Hv": g.n_v_heads, "d_k": g.d_k, "d_v": g.d_v},
                   "committed_streams": n_committed,
                   "l2": "flushed between timed steps (256 MiB device write, outside the events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "gdn_rows_kernel<128, window>", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} (hbm_gbs)" if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": wbytes,
                     "window_ms_per_launch": win_avg,
                     "traffic": ncu_traffic("gdn_window_verify_16x16.md")},
        "commit": {"ms_per_launch": statistics.mean(com_ms), "bytes_per_launch": commit_bytes(g, n_committed),
                   "gbs": commit_bytes(g, n_committed) / (statistics.mean(com_ms) * 1e-3) / 1e9},
        "e2e": {"value": world * R / (e2e_ms * 1e-3), "unit": "rows/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * K,
        "clocks": sampler.summary(t0, t1) if sampler else None,
        "wall_s": {"timed": t1 - t0, "e2e": t2 - t1},
    }
    return line


# ---- the CPU oracle, timed on the host cores --------------------------------

def oracle_rounds(budget_s: float, min_rounds: int = 1, max_streams=None):
    """Time the oracle on full streams of the same workload until budget_s."""
    import oracle

    g = GEOM
    w = synth.layer_weights(g, SEED)
    cache = synth.slot_cache(g, N_STREAMS, SEED)
    rows = synth.row_inputs(g, N_STREAMS * WINDOW, SEED)
    od = oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    threads = os.cpu_count() or 1
    done_rows, t_total, s = 0, 0.0, 0
    limit = max_streams or 10 ** 9
    while (t_total < budget_s or s < min_rounds) and s < limit:
        st = s % N_STREAMS
        lo, hi = st * WINDOW, (st + 1) * WINDOW
        t = time.perf_counter()
        oracle.gdn_rows(od, w, cache["state"][st], cache["tail"][st], rows["mixed"][lo:hi], rows["z"][lo:hi],
                        rows["a"][lo:hi], rows["b"][lo:hi], threads=threads)
        t_total += time.perf_counter() - t
        done_rows += WINDOW
        s += 1
    return done_rows, t_total, threads, s


def cpu_baseline():
    rows, secs, threads, streams = oracle_rounds(10.0)
    return {"value": rows / secs, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": f"{streams} stream windows of 16 rows (all 48 value heads, recorded), "
                      f"{secs:.1f} s of oracle time, heads split over {threads} threads"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle

    g = GEOM
    w = synth.layer_weights(g, SEED)
    cache = synth.slot_cache(g, N_STREAMS, SEED)
    rows = synth.row_inputs(g, WINDOW, SEED)
    od = oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    threads = os.cpu_count() or 1
    K, W = args.steps, max(args.warmup, 3)

    def one(heads):
        t = time.perf_counter()
        oracle.gdn_rows(od, w, cache["state"][0], cache["tail"][0], rows["mixed"], rows["z"], rows["a"], rows["b"],
                        heads=(0, heads), threads=min(threads, heads))
        return time.perf_counter() - t

    # size each step so the whole run stays within about two minutes
    t_one = min(one(1) for _ in range(2))
    heads = int(max(1, min(g.n_v_heads, 120.0 / ((K + W) * max(t_one, 1e-4)))))
    for _ in range(W):
        one(heads)
    times = [one(heads) for _ in range(K)]
    step_s = sum(times) / K
    rows_per_step = WINDOW * heads / g.n_v_heads
    value = rows_per_step / step_s
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "streams": N_STREAMS, "rows": N_STREAMS * WINDOW},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": min(threads, heads), "kind": "oracle",
                             "sample": f"each step: one 16-row window of {heads} of the 48 value heads "
                                       f"(a row counts as {heads}/48 of a layer row)"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_ours(args, rank, world, local_rank)
        if line is not None:
            if world == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline()
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
