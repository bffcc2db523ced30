#!/usr/bin/env python
"""Benchmark of the GDN speculative-verify round on GB300; prints ONE JSON line.

Workload (one step): the shared verify round of one GDN layer with 27B-like
heads (Hk=16 key heads, Hv=48 value heads, d_k=d_v=128): 16 streams x 16-row
chain windows (256 rows), every row's fp32 state and conv tail recorded into
a pool of cache entries (gdn_window_pooled), then each stream's random
accepted length 0..16 committed by index (gdn_commit_swap: the slot takes
the kept row's entry).  The same round with a record buffer and the copy
commit (gdn_window + gdn_commit) is reported beside it.  Inputs are seeded
synthetic tensors resident in HBM; L2 is flushed (a 256 MiB write) between
timed steps, outside the timed events.

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
            "(Hk=16, Hv=48, d_k=d_v=128), every row's fp32 state and conv tail recorded (into a pool of "
            "cache entries), then a random accepted length 0..16 per stream committed (by index)")


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
    for fn in ("gdn_common.cuh", "gdn_tc.cuh", "gdn_rows.cuh", "gdn_launch.h", "gdn_rows_d128.cu"):
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


def rank_seed(rank: int) -> int:
    """Each rank runs its own, independent round (weak scaling)."""
    return SEED + 1000 * rank


def reduce_max(values, world: int, device):
    """Max over ranks of a few timings (the only cross-rank step; timing only)."""
    if world <= 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


# ---- our arm ---------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import gated_deltanet_speculative_gb300 as gdn

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    g = GEOM
    R = N_STREAMS * WINDOW
    seed = rank_seed(rank)
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
    # A serving loop's step inputs (the rows' mixed, z, a, b and the keep
    # rows) back to back in one pinned buffer, so they cross in one copy.
    layout, pack_bytes = pack_layout({**{k: host_in[k] for k in ("mixed", "z", "a", "b")}, "keep": host_keep})
    host_pack = torch.empty(pack_bytes, dtype=torch.uint8).pin_memory()
    for k, v in unpack(host_pack, layout).items():
        v.copy_(host_in[k] if k != "keep" else host_keep)
    slot_t = torch.from_numpy(slots).to(dev)
    rp_t = torch.from_numpy(rp).to(dev)
    keep_t = host_keep.to(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # The round records every row in a pool of cache entries (gdn_window_pooled)
    # and commits by index (gdn_commit_swap).  The pool holds the 16 committed
    # states, the 256 records of a round and 16 spare entries; the entries
    # each round records into come from a first-in first-out free list that
    # the host keeps (the rows a round does not keep and the slots it
    # replaces are freed), computed ahead for every round the bench runs, in
    # the order the rounds run.
    n_pool = N_STREAMS + R + N_STREAMS
    pool_state = torch.empty((n_pool, g.n_v_heads, g.d_v, g.d_k), dtype=torch.float32, device=dev)
    pool_tail = torch.empty((n_pool, 3, g.channels), dtype=torch.bfloat16, device=dev)
    pool_state[:N_STREAMS].copy_(dc["state"])
    pool_tail[:N_STREAMS].copy_(dc["tail"])
    pool = {"state": pool_state, "tail": pool_tail}
    n_rounds = max(args.warmup, 3) + 4 * args.steps + 2
    recs = np.empty((n_rounds, R), np.int32)
    free, cur = list(range(N_STREAMS, n_pool)), list(range(N_STREAMS))
    for i in range(n_rounds):
        rec, free = free[:R], free[R:]
        kept = set()
        for s_ in range(N_STREAMS):
            if keep[s_] >= 0:
                free.append(cur[s_])
                cur[s_] = rec[keep[s_]]
                kept.add(cur[s_])
        free += [x for x in rec if x not in kept]
        recs[i] = rec
    host_recs = torch.from_numpy(recs).pin_memory()
    recs_t = host_recs.to(dev)
    rec_t = torch.empty(R, dtype=torch.int32, device=dev)   # the round's entries, as a serving loop sends them
    round_no = [0]

    def step(rec_slot=None, rows_=None, keep_=None):
        rs = recs_t[round_no[0]] if rec_slot is None else rec_slot
        gdn.window_pooled(d, dw, pool, slot_t, rp_t, dr if rows_ is None else rows_, rs, stream)
        gdn.commit_swap(d, pool, slot_t, rp_t, keep_t if keep_ is None else keep_, rs, None, stream)
        round_no[0] += 1

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
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(nvsmi_id(local_rank)) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.fill_(i & 0xff)
        rs = recs_t[round_no[0]]
        ev[i][0].record(stream)
        gdn.window_pooled(d, dw, pool, slot_t, rp_t, dr, rs, stream)
        gdn.commit_swap(d, pool, slot_t, rp_t, keep_t, rs, None, stream)
        ev[i][1].record(stream)
        round_no[0] += 1
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    step_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))

    # The same rounds with an event between the two launches, for the time
    # of each kernel alone (the window's is the roofline's denominator).  The
    # event also keeps the commit from being scheduled before the window ends,
    # so these two times add up to more than a step above.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xff)
        rs = recs_t[round_no[0]]
        evs[i][0].record(stream)
        gdn.window_pooled(d, dw, pool, slot_t, rp_t, dr, rs, stream)
        evs[i][1].record(stream)
        gdn.commit_swap(d, pool, slot_t, rp_t, keep_t, rs, None, stream)
        evs[i][2].record(stream)
        round_no[0] += 1
    torch.cuda.synchronize()
    win_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(K)]
    com_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(K)]

    # end to end through the public API: host inputs in, y back out, each step
    dev_pack = [torch.empty(pack_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    packed = [{**unpack(dp, layout), "y": y_} for dp, y_ in zip(dev_pack, (dr["y"], torch.empty_like(dr["y"])))]
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xff)
        ev2[i][0].record(stream)
        dev_pack[0].copy_(host_pack, non_blocking=True)
        rec_t.copy_(host_recs[round_no[0]], non_blocking=True)
        step(rec_slot=rec_t, rows_=packed[0], keep_=packed[0]["keep"])
        host_y.copy_(packed[0]["y"], non_blocking=True)
        ev2[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    if sampler:
        sampler.stop()
    e2e_serial_ms = sum(ev2[i][0].elapsed_time(ev2[i][1]) for i in range(K)) / K

    # end to end as a serving loop runs it: the same copies and calls, with
    # two device input sets, so step i+1's host->device copies (one copy
    # stream) and step i's y read-back (another) overlap the GPU work of the
    # steps around them.  The timed region spans all K steps, every copy
    # included; no L2 flush (each step writes 805 MB of records, far past L2).
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    recbufs = [rec_t, torch.empty_like(rec_t)]
    in_round = [0, 0]
    host_ys = [host_y, torch.empty_like(host_y).pin_memory()]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_y = [torch.cuda.Event() for _ in range(2)]

    def copy_in(b, rnd):
        with torch.cuda.stream(h2d_s):
            dev_pack[b].copy_(host_pack, non_blocking=True)
            recbufs[b].copy_(host_recs[rnd], non_blocking=True)
        ev_in[b].record(h2d_s)

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    h2d_s.wait_stream(stream)
    first = round_no[0]
    copy_in(0, first)
    for i in range(K):
        b = i & 1
        stream.wait_event(ev_in[b])
        gdn.window_pooled(d, dw, pool, slot_t, rp_t, packed[b], recbufs[b], stream)
        gdn.commit_swap(d, pool, slot_t, rp_t, packed[b]["keep"], recbufs[b], None, stream)
        ev_done[b].record(stream)
        round_no[0] += 1
        d2h_s.wait_event(ev_done[b])
        with torch.cuda.stream(d2h_s):
            host_ys[b].copy_(packed[b]["y"], non_blocking=True)
        ev_y[b].record(d2h_s)
        if i + 1 < K:
            nb = (i + 1) & 1   # last used by step i - 1: its calls and its y read-back must be done
            h2d_s.wait_event(ev_done[nb])
            h2d_s.wait_event(ev_y[nb])
            copy_in(nb, first + i + 1)
    stream.wait_event(ev_y[(K - 1) & 1])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    t2 = time.time()
    e2e_ms = t_start.elapsed_time(t_end) / K
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error word set during the timed steps")
    # the same round with its records in a buffer of their own and the copy
    # commit (gdn_window + gdn_commit), for comparison
    copy_round = None
    if rank == 0:
        del pool, pool_state, pool_tail
        rec_state = torch.empty((R, g.n_v_heads, g.d_v, g.d_k), dtype=torch.float32, device=dev)
        rec_tail = torch.empty((R, 3, g.channels), dtype=torch.bfloat16, device=dev)
        nk = min(K, 50)
        slot_c = torch.from_numpy(slots).to(dev)   # the pooled rounds moved slot_t into the pool
        evc = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nk + 3)]
        for i in range(nk + 3):
            flush.fill_(i & 0xff)
            evc[i][0].record(stream)
            gdn.window(d, dw, dc, slot_c, rp_t, dr, rec_state, rec_tail, stream)
            evc[i][1].record(stream)
            gdn.commit(d, dc, slot_c, rp_t, keep_t, rec_state, rec_tail, stream)
            evc[i][2].record(stream)
        torch.cuda.synchronize()
        cw_ms = statistics.mean(evc[i][0].elapsed_time(evc[i][1]) for i in range(3, nk + 3))
        cc_ms = statistics.mean(evc[i][1].elapsed_time(evc[i][2]) for i in range(3, nk + 3))
        n_committed_ = int((keep >= 0).sum())
        copy_round = {"ms_per_step": cw_ms + cc_ms, "rows_per_s": R / ((cw_ms + cc_ms) * 1e-3),
                      "window_ms": cw_ms, "commit_ms": cc_ms, "commit_bytes": commit_bytes(g, n_committed_),
                      "commit_gbs": commit_bytes(g, n_committed_) / (cc_ms * 1e-3) / 1e9,
                      "method": "gdn_window into a record buffer, then gdn_commit copying each kept row's "
                                "state and tail into its slot; CUDA events, L2 flushed between steps"}
        del rec_state, rec_tail
    extra = None
    if not args.no_extra and rank == 0:
        extra = run_extra(dev, stream, flush)
        if gdn.get_device_error() != 0:
            raise RuntimeError("device error word set during the secondary measurements")

    step_ms, e2e_ms, e2e_serial_ms, win_avg = reduce_max([step_ms, e2e_ms, e2e_serial_ms, statistics.mean(win_ms)],
                                                         world, dev)
    if rank != 0:
        return None

    n_committed = int((keep >= 0).sum())
    wbytes = window_bytes(g, N_STREAMS, R)
    peak, peak_src = hbm_peak()
    achieved = wbytes / (win_avg * 1e-3) / 1e9
    h2d = pack_bytes + R * 4   # the packed inputs (with alignment padding) + the round's pool entries
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
                     "traffic": ncu_traffic("gdn_window_verify_16x16.md"),
                     "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum of one launch, read from the "
                                       "committed ncu summary profiles/gdn_window_verify_16x16.md (not measured "
                                       "in this run); null when the kernel's sources changed since that capture"},
        "timing": "ms_per_step: CUDA events around each step's two launches (the commit launched as a "
                  "programmatic dependent of the window); the window's and the commit's own times come from "
                  "K more rounds with an event between the launches",
        "commit": {"kind": "index swap (gdn_commit_swap): slot[s] takes the kept row's pool entry",
                   "ms_per_launch": statistics.mean(com_ms), "streams_committed": n_committed},
        "copy_commit_round": copy_round,
        "e2e": {"value": world * R / (e2e_ms * 1e-3), "unit": "rows/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "method": "pinned host inputs (one packed buffer, plus the round's pool entries) copied in "
                          "and y read back every step through the public API; two device input sets, step "
                          "i+1's copies overlap step i's calls; one event pair around all steps, no L2 flush "
                          "(805 MB of records a step)",
                "serial": {"value": world * R / (e2e_serial_ms * 1e-3), "ms_per_step": e2e_serial_ms,
                           "method": "each step timed alone: copies in, calls, y back, in sequence"}},
        "gpu_launches": 2 * K,
        "clocks": sampler.summary(t0, t1) if sampler else None,
        "wall_s": {"timed": t1 - t0, "e2e": t2 - t1},
    }
    if extra is not None:
        line["extra"] = extra
    return line


def pack_layout(tensors: dict):
    """Byte offsets of the tensors placed back to back, each start 256-byte
    aligned: ({name: (offset, nbytes, dtype, shape)}, total bytes)."""
    layout, off = {}, 0
    for k, t in tensors.items():
        n = t.numel() * t.element_size()
        layout[k] = (off, n, t.dtype, tuple(t.shape))
        off = (off + n + 255) // 256 * 256
    return layout, off


def unpack(buf, layout) -> dict:
    """Views of a uint8 buffer laid out by pack_layout."""
    return {k: buf[o:o + n].view(dt).view(shape) for k, (o, n, dt, shape) in layout.items()}


# ---- secondary measurements: the other rows of the path ------------------

def _bf(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)


def _timed(fn, reps, stream, flush):
    """Mean ms per call: CUDA events around each call, L2 flushed between calls."""
    import torch
    fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        flush.fill_(3)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / reps


def prefill_flops(g: synth.Geometry, n_tokens: int, C: int = 64) -> float:
    """KK^T, QK^T, W, U~, WS^T, QS^T, PU, U^T K per chunk-head (the C x C solve excluded)."""
    d = g.d_k
    per_chunk_head = 2 * (5 * C * C * d + 3 * C * d * d)
    return n_tokens / C * g.n_v_heads * per_chunk_head


def prefill_bytes(g: synth.Geometry, n_tokens: int, n_seqs: int) -> int:
    row = (g.channels + 2 * g.n_v_heads * g.d_v + 2 * g.n_v_heads) * 2      # mixed, z, y, a, b
    return n_tokens * row + n_seqs * 2 * (g.n_v_heads * g.d_v * g.d_k * 4 + 3 * g.channels * 2)


def decode_bytes(g: synth.Geometry, n_streams: int) -> int:
    per = 2 * g.n_v_heads * g.d_v * g.d_k * 4 + 2 * 3 * g.channels * 2 + \
        (g.channels + 2 * g.n_v_heads * g.d_v + 2 * g.n_v_heads) * 2
    return n_streams * per


def run_extra(dev, stream, flush, reps=20, only=None):
    out = {}
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    bf16 = float(peaks.get("bf16_tflops", 1950.0))
    bf16_src = "measured bf16_tflops (burst)" if "bf16_tflops" in peaks else "fallback 1.95 PFLOP/s"

    if only in (None, "tree"):
        out["tree_round_16x16"] = _extra_tree(dev, stream, flush, reps, hbm)
        out["few_stream_windows_27b_like"] = _extra_few_streams(dev, stream, flush, reps, hbm)
    if only in (None, "replay"):
        out["logged_round_replay_commit_16x16"] = _extra_logged_round(dev, stream, flush, reps, hbm)
        out["logged_tree_replay_commit_16x16"] = _extra_logged_tree(dev, stream, flush, reps, hbm)
    if only in (None, "decode"):
        out["decode_24_layers_2b_like"] = _extra_decode(dev, stream, flush, reps, hbm)
    if only in (None, "prefill"):
        out["prefill_27b_like"] = _extra_prefill(dev, stream, flush, reps, hbm, bf16, bf16_src)
    return out


def logged_round_bytes(g: synth.Geometry, n_streams: int, n_rows: int, n_committed: int) -> int:
    """Window that logs instead of records, plus the replay commit."""
    tile = g.d_v * g.d_k * 4
    window = (n_streams * g.n_v_heads * tile + n_streams * 3 * g.channels * 2 + n_rows * 3 * g.channels * 2 +
              n_rows * (g.channels + g.n_v_heads * g.d_v + 2 * g.n_v_heads) * 2 + n_rows * g.n_v_heads * g.d_v * 2 +
              n_rows * (g.n_v_heads * (1 + g.d_v) + g.n_k_heads * g.d_k) * 4)
    replay = n_committed * (2 * g.n_v_heads * tile + 2 * 3 * g.channels * 2)   # logs re-read from L2 not counted
    return window + replay


def _extra_logged_round(dev, stream, flush, reps, hbm):
    """The verify round with logged rows (decay, write, key) and a replay
    commit in place of recorded states and a copy commit."""
    import torch
    import gated_deltanet_speculative_gb300 as gdn
    g = GEOM
    R = N_STREAMS * WINDOW
    w = synth.layer_weights(g, SEED)
    cache = synth.slot_cache(g, N_STREAMS, SEED)
    rows = synth.row_inputs(g, R, SEED)
    rp = synth.row_ptr([WINDOW] * N_STREAMS)
    rng = np.random.default_rng([SEED, 7])
    acc = synth.accepted_lengths(N_STREAMS, WINDOW, rng)
    keep = np.where(acc > 0, rp[:-1] + acc - 1, -1).astype(np.int32)
    d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    dw = {"conv_w": _bf(w["conv_w"]).to(dev), "A_log": torch.from_numpy(w["A_log"]).to(dev),
          "dt_bias": torch.from_numpy(w["dt_bias"]).to(dev), "norm_w": _bf(w["norm_w"]).to(dev)}
    dc = {"state": torch.from_numpy(cache["state"]).to(dev), "tail": _bf(cache["tail"]).to(dev)}
    dr = {k: _bf(rows[k]).to(dev) for k in ("mixed", "z", "a", "b")}
    dr["y"] = torch.empty((R, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device=dev)
    la = torch.empty((R, g.n_v_heads), dtype=torch.float32, device=dev)
    lu = torch.empty((R, g.n_v_heads, g.d_v), dtype=torch.float32, device=dev)
    lk = torch.empty((R, g.n_k_heads, g.d_k), dtype=torch.float32, device=dev)
    rt = torch.empty((R, 3, g.channels), dtype=torch.bfloat16, device=dev)
    slot_t = torch.arange(N_STREAMS, dtype=torch.int32, device=dev)
    rp_t = torch.from_numpy(rp).to(dev)
    keep_t = torch.from_numpy(keep).to(dev)

    def step():
        gdn.window_log(d, dw, dc, slot_t, rp_t, dr, la, lu, lk, rt, stream)
        gdn.commit_replay(d, dc, slot_t, rp_t, keep_t, la, lu, lk, rt, stream)

    ms = _timed(step, reps, stream, flush)
    ms_w = _timed(lambda: gdn.window_log(d, dw, dc, slot_t, rp_t, dr, la, lu, lk, rt, stream), reps, stream, flush)
    b = logged_round_bytes(g, N_STREAMS, R, int((keep >= 0).sum()))
    return {"ms_per_round": ms, "rows_per_s": R / (ms * 1e-3), "window_log_ms": ms_w,
            "algorithmic_gbs": b / (ms * 1e-3) / 1e9, "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm,
            "algorithmic_bytes": b}


def _tree_round_inputs(dev):
    """The tree round's inputs: 16 streams x 16-node random trees, one random
    leaf per stream kept."""
    import torch
    import gated_deltanet_speculative_gb300 as gdn
    g = GEOM
    R = N_STREAMS * WINDOW
    w = synth.layer_weights(g, 3)
    cache = synth.slot_cache(g, N_STREAMS, 3)
    rows = synth.row_inputs(g, R, 3)
    rng = np.random.default_rng([3, 9])
    parent = np.concatenate([synth.random_tree(WINDOW, rng) for _ in range(N_STREAMS)]).astype(np.int32)
    keep = np.array([s * WINDOW + synth.random_leaf(parent[s * WINDOW:(s + 1) * WINDOW], rng)
                     for s in range(N_STREAMS)], np.int32)
    d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    dw = {"conv_w": _bf(w["conv_w"]).to(dev), "A_log": torch.from_numpy(w["A_log"]).to(dev),
          "dt_bias": torch.from_numpy(w["dt_bias"]).to(dev), "norm_w": _bf(w["norm_w"]).to(dev)}
    dc = {"state": torch.from_numpy(cache["state"]).to(dev), "tail": _bf(cache["tail"]).to(dev)}
    dr = {k: _bf(rows[k]).to(dev) for k in ("mixed", "z", "a", "b")}
    dr["y"] = torch.empty((R, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device=dev)
    return {"d": d, "dw": dw, "dc": dc, "dr": dr, "keep": keep,
            "slot": torch.arange(N_STREAMS, dtype=torch.int32, device=dev),
            "rp": torch.from_numpy(synth.row_ptr([WINDOW] * N_STREAMS)).to(dev),
            "par": torch.from_numpy(parent).to(dev), "keep_t": torch.from_numpy(keep).to(dev)}


def _extra_logged_tree(dev, stream, flush, reps, hbm):
    """The tree round with logged nodes and a replay commit of one random
    leaf per stream, beside the recorded tree plus a copy commit."""
    import torch
    import gated_deltanet_speculative_gb300 as gdn
    g = GEOM
    R = N_STREAMS * WINDOW
    t = _tree_round_inputs(dev)
    d, dw, dc, dr = t["d"], t["dw"], t["dc"], t["dr"]
    la = torch.empty((R, g.n_v_heads), dtype=torch.float32, device=dev)
    lu = torch.empty((R, g.n_v_heads, g.d_v), dtype=torch.float32, device=dev)
    lk = torch.empty((R, g.n_k_heads, g.d_k), dtype=torch.float32, device=dev)
    rt = torch.empty((R, 3, g.channels), dtype=torch.bfloat16, device=dev)
    rs = torch.empty((R, g.n_v_heads, g.d_v, g.d_k), dtype=torch.float32, device=dev)

    def logged():
        gdn.tree_log(d, dw, dc, t["slot"], t["rp"], t["par"], dr, la, lu, lk, rt, stream)
        gdn.commit_replay_tree(d, dc, t["slot"], t["rp"], t["par"], t["keep_t"], la, lu, lk, rt, stream)

    def recorded():
        gdn.tree(d, dw, dc, t["slot"], t["rp"], t["par"], dr, rs, rt, stream)
        gdn.commit(d, dc, t["slot"], t["rp"], t["keep_t"], rs, rt, stream)

    ms = _timed(logged, reps, stream, flush)
    ms_w = _timed(lambda: gdn.tree_log(d, dw, dc, t["slot"], t["rp"], t["par"], dr, la, lu, lk, rt, stream), reps,
                  stream, flush)
    ms_rec = _timed(recorded, reps, stream, flush)
    del rs
    b = logged_round_bytes(g, N_STREAMS, R, N_STREAMS)
    return {"ms_per_round": ms, "rows_per_s": R / (ms * 1e-3), "tree_log_ms": ms_w,
            "algorithmic_gbs": b / (ms * 1e-3) / 1e9, "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm,
            "algorithmic_bytes": b,
            "recorded_tree_and_commit_ms": ms_rec, "recorded_rows_per_s": R / (ms_rec * 1e-3),
            "note": "parent states rebuilt from the slot (an L2 re-read plus a replay of the logged path) "
                    "are not counted"}


def _extra_few_streams(dev, stream, flush, reps, hbm):
    """Verify windows of 1, 2 and 4 streams x 16 rows, and a lone stream's
    16-node tree (27B-like heads, all rows recorded): latency-bound, the case
    a lone stream's round meets."""
    import torch
    import gated_deltanet_speculative_gb300 as gdn
    g = GEOM
    out = {}
    for S in (1, 2, 4):
        R = S * WINDOW
        w = synth.layer_weights(g, 5)
        cache = synth.slot_cache(g, S, 5)
        rows = synth.row_inputs(g, R, 5)
        d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
        dw = {"conv_w": _bf(w["conv_w"]).to(dev), "A_log": torch.from_numpy(w["A_log"]).to(dev),
              "dt_bias": torch.from_numpy(w["dt_bias"]).to(dev), "norm_w": _bf(w["norm_w"]).to(dev)}
        dc = {"state": torch.from_numpy(cache["state"]).to(dev), "tail": _bf(cache["tail"]).to(dev)}
        dr = {k: _bf(rows[k]).to(dev) for k in ("mixed", "z", "a", "b")}
        dr["y"] = torch.empty((R, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device=dev)
        rs = torch.empty((R, g.n_v_heads, g.d_v, g.d_k), dtype=torch.float32, device=dev)
        rt = torch.empty((R, 3, g.channels), dtype=torch.bfloat16, device=dev)
        slot_t = torch.arange(S, dtype=torch.int32, device=dev)
        rp_t = torch.from_numpy(synth.row_ptr([WINDOW] * S)).to(dev)
        ms = _timed(lambda: gdn.window(d, dw, dc, slot_t, rp_t, dr, rs, rt, stream), max(reps, 20), stream, flush)
        wb = window_bytes(g, S, R)
        out[str(S)] = {"us_per_window": ms * 1e3, "rows_per_s": R / (ms * 1e-3),
                       "frac_hbm": wb / (ms * 1e-3) / 1e9 / hbm}
        if S == 1:   # a lone stream's 16-node random tree, all nodes recorded
            par_t = torch.from_numpy(synth.random_tree(WINDOW, np.random.default_rng([5, 1]))).to(dev)
            ms_t = _timed(lambda: gdn.tree(d, dw, dc, slot_t, rp_t, par_t, dr, rs, rt, stream), max(reps, 20), stream,
                          flush)
            out["1"]["us_per_tree"] = ms_t * 1e3
    return out


def _extra_tree(dev, stream, flush, reps, hbm):
    """Tree round: 16 streams x 16-node random trees, all nodes recorded."""
    import torch
    import gated_deltanet_speculative_gb300 as gdn
    g = GEOM
    R = N_STREAMS * WINDOW
    w = synth.layer_weights(g, 3)
    cache = synth.slot_cache(g, N_STREAMS, 3)
    rows = synth.row_inputs(g, R, 3)
    rng = np.random.default_rng([3, 9])
    parent = np.concatenate([synth.random_tree(WINDOW, rng) for _ in range(N_STREAMS)]).astype(np.int32)
    d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    dw = {"conv_w": _bf(w["conv_w"]).to(dev), "A_log": torch.from_numpy(w["A_log"]).to(dev),
          "dt_bias": torch.from_numpy(w["dt_bias"]).to(dev), "norm_w": _bf(w["norm_w"]).to(dev)}
    dc = {"state": torch.from_numpy(cache["state"]).to(dev), "tail": _bf(cache["tail"]).to(dev)}
    dr = {k: _bf(rows[k]).to(dev) for k in ("mixed", "z", "a", "b")}
    dr["y"] = torch.empty((R, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device=dev)
    rs = torch.empty((R, g.n_v_heads, g.d_v, g.d_k), dtype=torch.float32, device=dev)
    rt = torch.empty((R, 3, g.channels), dtype=torch.bfloat16, device=dev)
    slot_t = torch.arange(N_STREAMS, dtype=torch.int32, device=dev)
    rp_t = torch.from_numpy(synth.row_ptr([WINDOW] * N_STREAMS)).to(dev)
    par_t = torch.from_numpy(parent).to(dev)
    ms = _timed(lambda: gdn.tree(d, dw, dc, slot_t, rp_t, par_t, dr, rs, rt, stream), reps, stream, flush)
    wb = window_bytes(g, N_STREAMS, R)
    return {"ms": ms, "rows_per_s": R / (ms * 1e-3), "algorithmic_gbs": wb / (ms * 1e-3) / 1e9,
            "frac_hbm": wb / (ms * 1e-3) / 1e9 / hbm,
            "note": "parent reloads of non-adjacent children are L2/HBM re-reads, not counted"}


def _extra_decode(dev, stream, flush, reps, hbm):
    """Decode: 24 independent 2B-like layers stepped in order, one row per stream."""
    import torch
    import gated_deltanet_speculative_gb300 as gdn
    g2 = synth.LIKE_2B
    d2 = gdn.Dims(g2.n_k_heads, g2.n_v_heads, g2.d_k, g2.d_v)
    dec = {}
    for S in (1, 4, 8, 16):
        layers = []
        for layer in range(24):
            w = synth.layer_weights(g2, 1 + 100 * layer)
            cache = synth.slot_cache(g2, S, 1 + 100 * layer)
            rows = synth.row_inputs(g2, S, 1 + 100 * layer)
            lw = {"conv_w": _bf(w["conv_w"]).to(dev), "A_log": torch.from_numpy(w["A_log"]).to(dev),
                  "dt_bias": torch.from_numpy(w["dt_bias"]).to(dev), "norm_w": _bf(w["norm_w"]).to(dev)}
            lc = {"state": torch.from_numpy(cache["state"]).to(dev), "tail": _bf(cache["tail"]).to(dev)}
            lr = {k: _bf(rows[k]).to(dev) for k in ("mixed", "z", "a", "b")}
            lr["y"] = torch.empty((S, g2.n_v_heads, g2.d_v), dtype=torch.bfloat16, device=dev)
            layers.append((lw, lc, lr))
        sl = torch.arange(S, dtype=torch.int32, device=dev)

        def step24():
            for lw, lc, lr in layers:
                gdn.step(d2, lw, lc, sl, lr, stream)

        ms = _timed(step24, reps, stream, flush)
        # the same calls prepared once (arguments checked and marshalled), then
        # enqueued eagerly: one ctypes call each
        prepared = [gdn.prepare(gdn.step, d2, lw, lc, sl, lr) for lw, lc, lr in layers]

        def step24_prepared():
            for call in prepared:
                call(stream)

        ms_p = _timed(step24_prepared, reps, stream, flush)
        # the same 24 launches captured once in a CUDA graph and replayed
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            step24_on = lambda: [gdn.step(d2, lw, lc, sl, lr, side) for lw, lc, lr in layers]
            step24_on()   # warm on the side stream before capture
            side.synchronize()
            with torch.cuda.graph(graph, stream=side):
                step24_on()
        torch.cuda.current_stream(dev).wait_stream(side)
        ms_g = _timed(graph.replay, reps, stream, flush)
        # the same replays back to back, no flush: the 24 layers' states stay in L2
        graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(50):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_nf = e0.elapsed_time(e1) / 50
        # the same 24 steps with GDN_STEP_EARLY_STATE: each step's kernel before
        # is the step of another layer, so its state, tail and weights may be
        # read while that kernel finishes
        graph_e = torch.cuda.CUDAGraph()
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            step24_early = lambda: [gdn.step_ex(d2, lw, lc, sl, lr, gdn.STEP_EARLY_STATE, side)
                                    for lw, lc, lr in layers]
            step24_early()
            side.synchronize()
            with torch.cuda.graph(graph_e, stream=side):
                step24_early()
        torch.cuda.current_stream(dev).wait_stream(side)
        ms_e = _timed(graph_e.replay, reps, stream, flush)
        b = 24 * decode_bytes(g2, S)
        dec[str(S)] = {"ms_per_24_layer_step": ms, "rows_per_s": S / (ms * 1e-3),
                       "algorithmic_gbs": b / (ms * 1e-3) / 1e9, "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm,
                       "graph": {"ms_per_24_layer_step": ms_g, "rows_per_s": S / (ms_g * 1e-3),
                                 "algorithmic_gbs": b / (ms_g * 1e-3) / 1e9,
                                 "frac_hbm": b / (ms_g * 1e-3) / 1e9 / hbm},
                       "eager_prepared": {"ms_per_24_layer_step": ms_p, "rows_per_s": S / (ms_p * 1e-3),
                                          "call": "gdn.prepare(gdn.step, ...) per layer, then 24 eager calls"},
                       "graph_early_state": {"ms_per_24_layer_step": ms_e, "rows_per_s": S / (ms_e * 1e-3),
                                             "algorithmic_gbs": b / (ms_e * 1e-3) / 1e9,
                                             "frac_hbm": b / (ms_e * 1e-3) / 1e9 / hbm,
                                             "call": "gdn_step_ex(..., GDN_STEP_EARLY_STATE): slot, state, tail "
                                                     "and weights read while the previous layer's step finishes"},
                       "graph_no_l2_flush": {"ms_per_24_layer_step": ms_nf, "rows_per_s": S / (ms_nf * 1e-3),
                                             "note": "50 replays back to back, one event pair; the layers' "
                                                     "states stay in L2, so no HBM fraction is given"}}
    return dec


def _extra_prefill(dev, stream, flush, reps, hbm, bf16, bf16_src):
    """Prefill: (i) one 4722-token prompt; (ii) 512/1024/2048/4096 in one pass."""
    import torch
    import gated_deltanet_speculative_gb300 as gdn
    g = GEOM
    d = gdn.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    pre = {}
    for name, lengths in (("i_4722", [4722]), ("ii_512_1024_2048_4096", [512, 1024, 2048, 4096])):
        T = sum(lengths)
        S = len(lengths)
        w = synth.layer_weights(g, 4)
        cache = synth.slot_cache(g, S, 4, zero=True)
        rows = synth.row_inputs(g, T, 4)
        dw = {"conv_w": _bf(w["conv_w"]).to(dev), "A_log": torch.from_numpy(w["A_log"]).to(dev),
              "dt_bias": torch.from_numpy(w["dt_bias"]).to(dev), "norm_w": _bf(w["norm_w"]).to(dev)}
        dc = {"state": torch.from_numpy(cache["state"]).to(dev), "tail": _bf(cache["tail"]).to(dev)}
        dr = {k: _bf(rows[k]).to(dev) for k in ("mixed", "z", "a", "b")}
        dr["y"] = torch.empty((T, g.n_v_heads, g.d_v), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(gdn.prefill_workspace_size(d, S, T), dtype=torch.uint8, device=dev)
        sl = torch.arange(S, dtype=torch.int32, device=dev)
        cu = torch.from_numpy(synth.row_ptr(lengths)).to(dev)
        state0 = dc["state"].clone()
        tail0 = dc["tail"].clone()

        def run():
            dc["state"].copy_(state0)   # every pass starts from the zero state (tiny copy)
            dc["tail"].copy_(tail0)
            gdn.prefill(d, dw, dc, sl, cu, dr, ws, stream=stream)

        ms = _timed(run, max(5, reps // 2), stream, flush)
        fl = prefill_flops(g, T)
        by = prefill_bytes(g, T, S)
        pre[name] = {"ms": ms, "tokens_per_s": T / (ms * 1e-3), "algorithmic_tflops": fl / (ms * 1e-3) / 1e12,
                     "frac_bf16_tensor_peak": fl / (ms * 1e-3) / 1e12 / bf16,
                     "bf16_peak_tflops": bf16,
                     "bf16_peak_source": bf16_src + ": each call is a sub-millisecond burst",
                     "algorithmic_gbs": by / (ms * 1e-3) / 1e9, "frac_hbm": by / (ms * 1e-3) / 1e9 / hbm,
                     "algorithmic_flop": fl, "algorithmic_bytes": by,
                     "note": "d=128, C=64: contractions on tcgen05 bf16 tensor cores as 3-pass hi/lo splits (3x the algorithmic MMA work); time includes a state reset copy"}
        del ws, dr, dc
    return pre


# ---- the CPU oracle, timed on the host cores --------------------------------

def oracle_rounds(budget_s: float, min_rounds: int = 1, max_streams=None, threads=None):
    """Time the oracle on full streams of the same workload until budget_s."""
    import oracle

    g = GEOM
    w = synth.layer_weights(g, SEED)
    cache = synth.slot_cache(g, N_STREAMS, SEED)
    rows = synth.row_inputs(g, N_STREAMS * WINDOW, SEED)
    od = oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    threads = threads or os.cpu_count() or 1
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


def oracle_other_workloads():
    """The oracle on the other rows' workloads, whole, on all host cores:
    the 24-layer 2B-like decode step at one stream, and the two prefill
    passes (the sequential recurrence, token by token)."""
    import oracle

    threads = os.cpu_count() or 1
    out = {}
    g2 = synth.LIKE_2B
    od2 = oracle.Dims(g2.n_k_heads, g2.n_v_heads, g2.d_k, g2.d_v)
    layers = [(synth.layer_weights(g2, 1 + 100 * l), synth.slot_cache(g2, 1, 1 + 100 * l),
               synth.row_inputs(g2, 1, 1 + 100 * l)) for l in range(24)]
    t = time.perf_counter()
    for w2, c2, r2 in layers:
        oracle.gdn_rows(od2, w2, c2["state"][0], c2["tail"][0], r2["mixed"], r2["z"], r2["a"], r2["b"],
                        record=False, final=True, threads=threads)
    dt = time.perf_counter() - t
    out["decode_24_layers_2b_like_1_stream"] = {"ms_per_24_layer_step": dt * 1e3, "rows_per_s": 1 / dt}
    g = GEOM
    od = oracle.Dims(g.n_k_heads, g.n_v_heads, g.d_k, g.d_v)
    for name, lengths in (("prefill_i_4722", [4722]), ("prefill_ii_512_1024_2048_4096", [512, 1024, 2048, 4096])):
        w = synth.layer_weights(g, 4)
        cache = synth.slot_cache(g, len(lengths), 4, zero=True)
        rows = synth.row_inputs(g, sum(lengths), 4)
        cu = synth.row_ptr(lengths)
        t = time.perf_counter()
        for s_ in range(len(lengths)):
            lo, hi = int(cu[s_]), int(cu[s_ + 1])
            oracle.gdn_rows(od, w, cache["state"][s_], cache["tail"][s_], rows["mixed"][lo:hi], rows["z"][lo:hi],
                            rows["a"][lo:hi], rows["b"][lo:hi], record=False, final=True, threads=threads)
        dt = time.perf_counter() - t
        out[name] = {"ms": dt * 1e3, "tokens_per_s": sum(lengths) / dt}
    out["cores"] = threads
    return out


def cpu_baseline():
    rows, secs, threads, streams = oracle_rounds(10.0)
    rows1, secs1, _, streams1 = oracle_rounds(3.0, threads=1)
    return {"value": rows / secs, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": f"{streams} stream windows of 16 rows (all 48 value heads, recorded), "
                      f"{secs:.1f} s of oracle time, heads split over {threads} threads",
            "single_thread": {"value": rows1 / secs1, "unit": "rows/s", "cores": 1,
                              "sample": f"{streams1} stream windows of 16 rows, {secs1:.1f} s, one thread "
                                        f"(the plain sequential definition)"},
            "other_workloads": oracle_other_workloads()}


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
    ap.add_argument("--no-extra", action="store_true", help="skip the tree / decode / prefill measurements")
    ap.add_argument("--extra-only", choices=["tree", "decode", "prefill", "replay"],
                    help="run only this secondary measurement (3 repetitions) and print it; for profiling")
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

    if args.extra_only:
        import torch
        torch.cuda.set_device(local_rank)
        dev = torch.device("cuda", local_rank)
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        rec = run_extra(dev, torch.cuda.current_stream(), flush, reps=3, only=args.extra_only)
        print(json.dumps({"extra_only": args.extra_only, **rec}), flush=True)
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
