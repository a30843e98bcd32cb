#!/usr/bin/env python3
"""Benchmark: fused grouped scaled activation + NVFP4/MXFP8 quantization,
forward and backward, GB/s of algorithmic HBM bytes and fraction of the HBM
roofline, on one GPU (N GPUs under torchrun run independent replicas).

Default workload: NVFP4 with the 16-point RHT on the columnwise copy,
SReLU and TanhSReLU(s=4), 32 experts, 65536 rows (Dirichlet(0.5) split),
width 2048, seeded synthetic inputs (X ~ N(0,1) BF16, p ~ U(0,1),
dY ~ N(0,1)).  One step = for each activation: forward (Y rowwise + columnwise
copies) + backward (dense dX, dX rowwise + columnwise copies, dprobs).
Inputs (X, dY: 268 MB each) are larger than L2, so no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gsa|reference]

After the timed region, "unfused_two_step" times the unfused path of the same
step (the activation kernel writing BF16, then a separate grouped quantizer
reading it back) against the fused kernel, with the algorithmic bytes of each,
and "graph_safe" times the graph-safe calls (split on the device) replayed from
a captured CUDA graph.

--impl reference times the CPU oracle (the slow, plain definition) on a
bounded sample of the same workload; it is a reported baseline, not a target.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_quantization_grouped_gb300 import inputs  # noqa: E402

METRIC = "fused grouped act+quant fwd/bwd GB/s and % of GB300 HBM peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
ACT_PARAMS = (4.0, 7.0, 1.702, 1.0)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gsa", choices=["gsa", "reference"])
    ap.add_argument("--workload", default="nvfp4_rht", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--acts", default=None, help="comma list; default: the workload's activations")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--rows", type=int, default=None, help="rescale the workload to this many rows (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused-steps", type=int, default=30,
                    help="iterations of the unfused two-step comparison (0: skip); outside the timed region")
    ap.add_argument("--configs", default="tiny_srelu_mxfp8,tanh_srelu_mxfp8_recompute,swiglu_mxfp8,"
                                         "moe_swiglu_mxfp8_recompute",
                    help="other workloads timed after the timed region ('' to skip)")
    ap.add_argument("--clock-seconds", type=float, default=1.0,
                    help="per headline kernel: seconds of back-to-back launches with clock sampling (0: skip)")
    return ap.parse_args()


# ----------------------------------------------------------------- bytes

def layout_bytes(split, width, recipe, rowwise, columnwise):
    """Bytes of the quantized copies, from the library's layout query."""
    from nvfp4_quantization_grouped_gb300 import gsa
    info, _, _ = gsa.gsa_layout(list(split), width, recipe)
    b = 0
    if rowwise:
        b += info.row_data_bytes + info.row_scale_bytes + 4 * info.amax_floats
    if columnwise:
        b += info.col_data_bytes + info.col_scale_bytes + 4 * info.amax_floats
    return b


def layout_bytes_oracle(split, width, recipe, rowwise, columnwise):
    """The same bytes from the oracle's layout (the reference arm loads nothing
    of the product library)."""
    import oracle
    M = int(sum(int(m) for m in split))
    bsz = oracle.block_size(recipe)
    amax = 4 * len(split) if recipe == oracle.NVFP4 else 0
    b = 0
    if rowwise:
        b += (M * width if recipe == oracle.MXFP8 else M * width // 2) + M * width // bsz + amax
    if columnwise:
        d, s = oracle.expert_col_offsets(split, width, recipe)
        b += int(d[-1]) + int(s[-1]) + amax
    return b


def algorithmic_bytes(wl, split, M, layout=layout_bytes):
    """Compulsory HBM bytes of one forward and one backward launch."""
    w, w_in = wl.width, wl.w_in
    recompute = wl.recompute
    fwd = M * w_in * 2 + M * 4 + layout(split, w, wl.recipe, True, not recompute)
    bwd = (M * w_in * 2 + M * w * 2 + M * 4            # X, dY, p
           + M * w_in * 2 + M * 4                      # dense dX, dprobs
           + layout(split, w_in, wl.recipe, True, True)
           + (layout(split, w, wl.recipe, False, True) if recompute else 0))
    return fwd, bwd


def two_step_bytes(wl, split, M):
    """Compulsory HBM bytes of the unfused two-step path (activation kernel
    writing BF16, then a separate grouped quantizer reading it back):
    forward and backward, each as (activation step, quantize step)."""
    w, w_in = wl.width, wl.w_in
    f_act = M * w_in * 2 + M * 4 + M * w * 2                  # X, p -> BF16 Y
    f_q = M * w * 2 + layout_bytes(split, w, wl.recipe, True, not wl.recompute)
    b_act = M * w_in * 2 + M * w * 2 + M * 4 + M * w_in * 2 + M * 4   # X, dY, p -> dX, dprobs
    b_q = M * w_in * 2 + layout_bytes(split, w_in, wl.recipe, True, True)
    return (f_act, f_q), (b_act, b_q)


def time_unfused(args, wl, acts, split, M, x, dy, p, prm, mask, ws, fwd_out, bwd_out, per, fb, bb, dev):
    """Unfused two-step path against the fused kernel: the activation kernel
    alone (dense BF16 output, no quantized copy), then the identity activation
    with p = 1 as a plain grouped quantizer of that BF16 tensor.  The fused
    times are the timed region's per-kernel averages."""
    import torch
    from nvfp4_quantization_grouped_gb300 import gsa

    stream = torch.cuda.current_stream()
    ws_q = gsa.Workspace(split, wl.w_in, inputs.ACT_IDENTITY, wl.recipe, dev)
    y = torch.empty((M, wl.width), dtype=torch.bfloat16, device=dev)
    y_q = gsa.alloc_qtensor(split, wl.width, wl.recipe, True, not wl.recompute, dev)
    dx_q = gsa.alloc_qtensor(split, wl.w_in, wl.recipe, True, True, dev)
    b1 = {"dx": bwd_out["dx"], "dprobs": bwd_out["dprobs"]}
    (f_act, f_q), (b_act, b_q) = two_step_bytes(wl, split, M)
    res = {}
    for a in acts:
        calls = {
            "fwd_act": lambda: gsa.fwd(x, p, split, a, wl.recipe, wl.rht, mask, False, False, True, prm, ws,
                                       {"y": y}),
            "fwd_quant": lambda: gsa.fwd(y, None, split, "identity", wl.recipe, wl.rht, mask, True,
                                         not wl.recompute, False, prm, ws_q, y_q),
            "bwd_act": lambda: gsa.bwd(dy, x, p, split, a, wl.recipe, wl.rht, mask, True, False, False, True, False,
                                       prm, ws, b1),
            "bwd_quant": lambda: gsa.fwd(b1["dx"], None, split, "identity", wl.recipe, wl.rht, mask, True, True,
                                         False, prm, ws_q, dx_q),
        }
        tm = {k: [] for k in calls}
        for it in range(args.unfused_steps + 2):
            for k, fn in calls.items():
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                if it >= 2:
                    tm[k].append((e0, e1))
        torch.cuda.synchronize()
        us = {k: 1e3 * sum(e0.elapsed_time(e1) for e0, e1 in v) / len(v) for k, v in tm.items()}
        for d, fused_bytes, nb in (("fwd", fb, (f_act, f_q)), ("bwd", bb, (b_act, b_q))):
            fused_us = 1e3 * sum(per[f"{d}_{a}"]) / len(per[f"{d}_{a}"])
            two = us[d + "_act"] + us[d + "_quant"]
            res[f"{d}_{a}"] = {"fused_us": round(fused_us, 2), "act_us": round(us[d + "_act"], 2),
                               "quant_us": round(us[d + "_quant"], 2), "two_step_us": round(two, 2),
                               "fused_speedup": round(two / fused_us, 3), "fused_bytes": fused_bytes,
                               "two_step_bytes": nb[0] + nb[1], "bytes_saved": nb[0] + nb[1] - fused_bytes}
    if ws_q.status() != 0:
        raise RuntimeError("device-side wait timed out in the unfused comparison")
    return res


def time_graph_safe(args, wl, acts, split, M, x, dy, p, prm, mask, fwd_out, bwd_out, per, dev):
    """The graph-safe calls (split on the device: counter memset, one-CTA plan
    kernel, fused kernel) captured once in a CUDA graph and replayed; per-call
    time against the host-split kernel's average from the timed region."""
    import torch
    from nvfp4_quantization_grouped_gb300 import gsa

    E = len(split)
    sd = torch.tensor(split, dtype=torch.int64, device=dev)
    res = {}
    for a in acts:
        aid = inputs.ACT_NAMES[a]
        ws = gsa.GraphSafeWorkspace(E, M, wl.w_in, aid, wl.recipe, dev)
        fo = gsa.fwd_graph_safe(x, p, sd, a, wl.recipe, wl.rht, mask, True, not wl.recompute, False, prm, ws)
        bo = gsa.bwd_graph_safe(dy, x, p, sd, a, wl.recipe, wl.rht, mask, True, True, True, True, wl.recompute,
                                prm, ws)
        torch.cuda.synchronize()
        for d, call in (("fwd", lambda: gsa.fwd_graph_safe(x, p, sd, a, wl.recipe, wl.rht, mask, True,
                                                            not wl.recompute, False, prm, ws, fo)),
                        ("bwd", lambda: gsa.bwd_graph_safe(dy, x, p, sd, a, wl.recipe, wl.rht, mask, True, True,
                                                            True, True, wl.recompute, prm, ws, bo))):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            for _ in range(3):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.unfused_steps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = 1e3 * e0.elapsed_time(e1) / args.unfused_steps
            host_us = 1e3 * sum(per[f"{d}_{a}"]) / len(per[f"{d}_{a}"])
            res[f"{d}_{a}"] = {"graph_replay_us": round(us, 2), "host_split_kernel_us": round(host_us, 2)}
        if ws.status() != 0:
            raise RuntimeError("graph-safe calls reported an error")
    return res


# ------------------------------------------------- other workloads, clocks

def time_launches(fn, reps, stream, flush=None):
    """Median µs of one launch (CUDA events on the launching stream); with
    flush, a buffer larger than L2 is written before every launch, outside the
    events; without, a short device-side sleep precedes each launch instead, so
    that the host has enqueued the call before the first event fires and the
    events time the device work alone (with L2 as the previous launch left it)."""
    import torch
    evs = []
    for i in range(reps + 3):
        if flush is not None:
            flush.zero_()
        else:
            torch.cuda._sleep(100000)   # about 50 µs of device time, no memory traffic
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        if i >= 3:
            evs.append((e0, e1))
    torch.cuda.synchronize()
    return 1e3 * statistics.median(a.elapsed_time(b) for a, b in evs)


L2_RESIDENT = ("tiny_srelu_mxfp8", "tanh_srelu_mxfp8_recompute")


def time_configs(names, dev, peak, peak_kind):
    """Fused forward and backward of the other workloads at full size, each as
    its configuration describes (recompute: forward rowwise only, backward with
    the regenerated columnwise copy).  The L2-resident ones are timed both hot
    (back to back) and with L2 flushed before every launch."""
    import torch
    from nvfp4_quantization_grouped_gb300 import gsa
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)   # 4 x L2
    prm = gsa.ActParams(*ACT_PARAMS)
    res = {}
    for name in names:
        wl, split, M, x, p, dy = inputs.device_problem(name, dev)
        fb, bb = algorithmic_bytes(wl, split, M)
        big = wl.rows * wl.w_in * 2 > (1 << 30)
        reps = {"tiny_srelu_mxfp8": 300, "tanh_srelu_mxfp8_recompute": 200}.get(name, 10 if big else 40)
        ent = {"rows": M, "experts": len(split), "empty_experts": int(sum(1 for v in split if v == 0)),
               "width": wl.width, "w_in": wl.w_in, "recipe": "nvfp4" if wl.recipe == inputs.RECIPE_NVFP4 else "mxfp8",
               "recompute": wl.recompute, "bytes": {"fwd": fb, "bwd": bb},
               "inputs": "split as in the parity tests; X, dY drawn on the device (seeded)",
               "l2": "flushed and hot" if name in L2_RESIDENT else "inputs larger than L2"}
        for a in wl.acts:
            ws = gsa.Workspace(split, wl.w_in, inputs.ACT_NAMES[a], wl.recipe, dev)
            fo = gsa.alloc_qtensor(split, wl.width, wl.recipe, True, not wl.recompute, dev)
            bo = gsa.alloc_qtensor(split, wl.w_in, wl.recipe, True, True, dev)
            bo["dx"] = torch.empty((M, wl.w_in), dtype=torch.bfloat16, device=dev)
            bo["dprobs"] = torch.empty(M, dtype=torch.float32, device=dev)
            if wl.recompute:
                for k, v in gsa.alloc_qtensor(split, wl.width, wl.recipe, False, True, dev).items():
                    bo["y_" + k] = v
            calls = {"fwd": (fb, lambda: gsa.fwd(x, p, split, a, wl.recipe, wl.rht, 0, True, not wl.recompute, False,
                                                 prm, ws, fo)),
                     "bwd": (bb, lambda: gsa.bwd(dy, x, p, split, a, wl.recipe, wl.rht, 0, True, True, True, True,
                                                 wl.recompute, prm, ws, bo))}
            ent[a] = {}
            for d, (nbytes, fn) in calls.items():
                r = {}
                modes = (("flushed", flush), ("hot", None)) if name in L2_RESIDENT else (("", None),)
                for tag, fl in modes:
                    us = time_launches(fn, reps, stream, fl)
                    sfx = "_" + tag if tag else ""
                    r["us" + sfx] = round(us, 2)
                    r["gbs" + sfx] = round(nbytes / (us * 1e-6) / 1e9, 1)
                    r["frac_of_" + peak_kind + sfx] = round(nbytes / (us * 1e-6) / 1e9 / peak, 4)
                ent[a][d] = r
            if ws.status() != 0:
                raise RuntimeError(f"device-side wait timed out on {name}")
            del fo, bo, ws
        res[name] = ent
        del x, p, dy
        torch.cuda.empty_cache()
    return res


def kernel_clocks(calls, seconds, local):
    """Each headline kernel back to back for about `seconds`, with the clock
    sampler running: average µs, SM clock samples and throttle reasons."""
    import torch
    stream = torch.cuda.current_stream()
    out = {}
    for key, fn in calls.items():
        us = time_launches(fn, 5, stream)
        n = max(10, int(seconds / (us * 1e-6)))
        sampler = ClockSampler(local)
        time.sleep(0.3)
        sampler.mark()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        c = sampler.stop() or {}
        out[key] = {"avg_us": round(1e3 * e0.elapsed_time(e1) / n, 2), "launches": n, **c}
    return out


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self):
        self.t0 = time.time()

    def stop(self):
        t1 = time.time()
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0 = getattr(self, "t0", 0.0)
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                if not (t0 - 0.05 <= ts <= t1 + 0.05):
                    continue
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if k in d and d[k]:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the kernel sources with comments and whitespace removed (a
    comment edit does not invalidate a recorded capture)."""
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "nvfp4_quantization_grouped_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode() + b"\0" + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(key):
    """DRAM bytes per launch from a committed ncu capture, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(key)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


def dist_setup(n):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def aggregate_gbs(world, step_bytes, steps, max_ms):
    """Whole-job throughput of N independent replicas: every rank processes
    step_bytes per step, the time is the slowest rank's."""
    return world * step_bytes * steps / (max_ms * 1e-3) / 1e9


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- CPU oracle

def oracle_sample(pr, rows_target):
    """Whole experts from the front of the workload (the NVFP4 scale is per
    expert) until about rows_target rows; the last one taken may be cut short
    and then counts as an expert of that many rows."""
    take, xs, ps, dys = [], [], [], []
    off = rows = 0
    for s in (int(v) for v in pr.split_sizes):
        if rows >= rows_target:
            break
        n = min(s, rows_target - rows)
        if n > 0:
            take.append(n)
            xs.append(pr.x[off:off + n]); ps.append(pr.probs[off:off + n]); dys.append(pr.dy[off:off + n])
            rows += n
        off += s
    return take, np.concatenate(xs), np.concatenate(ps), np.concatenate(dys)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_step(wl, acts, sample, mask, threads=1):
    """One step of the oracle on the sample: per activation the forward and the
    backward.  With threads > 1 the experts run concurrently (each expert is an
    independent problem; the oracle's C calls release the GIL).  Returns the
    outputs, concatenated in expert order."""
    import concurrent.futures
    import oracle
    split, x, p, dy = sample
    offs = np.concatenate([[0], np.cumsum(split)]).astype(np.int64)

    def one(a, e_lo, e_hi):
        lo, hi = offs[e_lo], offs[e_hi]
        aid = inputs.ACT_NAMES[a]
        sp = split[e_lo:e_hi]
        f = oracle.fwd(x[lo:hi], p[lo:hi], sp, aid, ACT_PARAMS, wl.recipe, wl.rht, mask, True, not wl.recompute)
        b = oracle.bwd(dy[lo:hi], x[lo:hi], p[lo:hi], sp, aid, ACT_PARAMS, wl.recipe, wl.rht, mask, True, True,
                       wl.recompute)
        return f, b

    out = {}
    for a in acts:
        if threads <= 1:
            parts = [one(a, 0, len(split))]
        else:
            with concurrent.futures.ThreadPoolExecutor(threads) as ex:
                parts = list(ex.map(lambda e: one(a, e, e + 1), range(len(split))))
        for d, i in (("fwd", 0), ("bwd", 1)):
            for k in parts[0][i]:
                out[(a, d, k)] = np.concatenate([np.asarray(pt[i][k]).reshape(-1) for pt in parts])
    return out


def time_oracle(wl, acts, pr, seconds_target, max_rows=None, layout=layout_bytes):
    """Oracle GB/s on a bounded sample of whole experts (about seconds_target
    of single-threaded work), timed on all host cores (threads over experts)
    and on one thread; the two results must be identical."""
    cores = host_cores()
    probe = oracle_sample(pr, 64)
    t0 = time.perf_counter()
    oracle_step(wl, acts, probe, pr.rht_mask)
    per_row = (time.perf_counter() - t0) / max(1, sum(probe[0]))
    rows = int(max(16, min(max_rows or 1 << 30, seconds_target / max(per_row, 1e-9))))
    sample = oracle_sample(pr, rows)
    t0 = time.perf_counter()
    multi = oracle_step(wl, acts, sample, pr.rht_mask, threads=cores)
    dt = time.perf_counter() - t0
    t0 = time.perf_counter()
    single = oracle_step(wl, acts, sample, pr.rht_mask, threads=1)
    dt1 = time.perf_counter() - t0
    same = multi.keys() == single.keys() and all(
        np.array_equal(multi[k].view(np.uint8), single[k].view(np.uint8)) for k in multi)
    if not same:
        raise RuntimeError("the threaded oracle disagrees with the single-threaded run")
    M = sum(sample[0])
    fb, bb = algorithmic_bytes(wl, sample[0], M, layout)
    nbytes = len(acts) * (fb + bb)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_thread_value": nbytes / dt1 / 1e9, "identical_to_single_thread": True,
            "sample": f"{len(sample[0])} expert(s), {M} rows x width {wl.w_in} of the workload, "
                      f"{len(acts)} activation(s) fwd+bwd; C oracle with {cores} threads over experts "
                      f"{dt:.1f} s, one thread {dt1:.1f} s, outputs identical"}, sample, dt


# ----------------------------------------------------------------- arms

def run_reference(args):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    wl = inputs.WORKLOADS[args.workload]
    acts = args.acts.split(",") if args.acts else list(wl.acts)
    pr = inputs.make_problem(args.workload, 0, rows=args.rows)
    budget = 150.0 / max(1, args.steps + args.warmup)
    base, sample, _ = time_oracle(wl, acts, pr, budget, layout=layout_bytes_oracle)
    cores = base["cores"]
    for _ in range(args.warmup):
        oracle_step(wl, acts, sample, pr.rht_mask, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, acts, sample, pr.rht_mask, threads=cores)
    dt = time.perf_counter() - t0
    M = sum(sample[0])
    fb, bb = algorithmic_bytes(wl, sample[0], M, layout_bytes_oracle)
    value = args.steps * len(acts) * (fb + bb) / dt / 1e9
    base["value"] = value
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config_of(wl, acts, pr),
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(wl, acts, pr):
    return {"workload": wl.name, "description": wl.description, "experts": wl.experts,
            "rows": int(pr.split_sizes.sum()), "width": wl.width, "w_in": wl.w_in,
            "empty_experts": int((pr.split_sizes == 0).sum()), "acts": acts,
            "recipe": "nvfp4" if wl.recipe == inputs.RECIPE_NVFP4 else "mxfp8", "rht_colwise": wl.rht,
            "recompute": wl.recompute,
            "step": "per activation: fwd (Y rowwise + columnwise) + bwd (dense dX, dX rowwise + columnwise, "
                    "dprobs" + (", regenerated Y columnwise" if wl.recompute else "") + ")",
            "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas"}


def run_gsa(args):
    import torch
    from nvfp4_quantization_grouped_gb300 import gsa

    rank, world, local = dist_setup(args.gpus)
    wl = inputs.WORKLOADS[args.workload]
    acts = args.acts.split(",") if args.acts else list(wl.acts)
    pr = inputs.make_problem(args.workload, rank, rows=args.rows)
    split = [int(s) for s in pr.split_sizes]
    M = int(pr.split_sizes.sum())
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    x = torch.from_numpy(pr.x.view(np.int16)).view(torch.bfloat16).to(dev)
    dy = torch.from_numpy(pr.dy.view(np.int16)).view(torch.bfloat16).to(dev)
    p = torch.from_numpy(pr.probs).to(dev)
    prm = gsa.ActParams(*ACT_PARAMS)
    a0 = inputs.ACT_NAMES[acts[0]]
    ws = gsa.Workspace(split, wl.w_in, a0, wl.recipe, dev)
    mask = pr.rht_mask
    fwd_out = gsa.alloc_qtensor(split, wl.width, wl.recipe, True, not wl.recompute, dev)
    bwd_out = gsa.alloc_qtensor(split, wl.w_in, wl.recipe, True, True, dev)
    bwd_out["dx"] = torch.empty((M, wl.w_in), dtype=torch.bfloat16, device=dev)
    bwd_out["dprobs"] = torch.empty(M, dtype=torch.float32, device=dev)
    if wl.recompute:
        for k, v in gsa.alloc_qtensor(split, wl.width, wl.recipe, False, True, dev).items():
            bwd_out["y_" + k] = v

    launches = [0]

    def step(events=None):
        for a in acts:
            if events is not None:
                events.append((a, "fwd", torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                events[-1][2].record(stream)
            gsa.fwd(x, p, split, a, wl.recipe, wl.rht, mask, True, not wl.recompute, False, prm, ws, fwd_out)
            launches[0] += gsa.gsa_last_launch_count()
            if events is not None:
                events[-1][3].record(stream)
                events.append((a, "bwd", torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                events[-1][2].record(stream)
            gsa.bwd(dy, x, p, split, a, wl.recipe, wl.rht, mask, True, True, True, True, wl.recompute, prm, ws,
                    bwd_out)
            launches[0] += gsa.gsa_last_launch_count()
            if events is not None:
                events[-1][3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if ws.status() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    fb, bb = algorithmic_bytes(wl, split, M)
    step_bytes = len(acts) * (fb + bb)

    # ---------------- timed region
    events = []
    launches[0] = 0
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    time.sleep(0.5)
    sampler.mark()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step(events)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    ms = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms, world)
    gpu_launches = launches[0]
    if ws.status() != 0:
        raise RuntimeError("device-side wait timed out in the timed region")

    per = {}
    for a, d, e0, e1 in events:
        per.setdefault(f"{d}_{a}", []).append(e0.elapsed_time(e1))
    kernels = {}
    peak, peak_kind = measured_peak()
    for key, v in per.items():
        avg_ms = sum(v) / len(v)
        nbytes = fb if key.startswith("fwd") else bb
        gbs = nbytes / (avg_ms * 1e-3) / 1e9
        kernels[key] = {"avg_us": round(avg_ms * 1e3, 2), "bytes": nbytes, "gbs": round(gbs, 1),
                        "frac_of_" + peak_kind: round(gbs / peak, 4), "launches": len(v)}
    dom = max(per, key=lambda k: sum(per[k]))
    dom_avg = sum(per[dom]) / len(per[dom])
    dom_bytes = fb if dom.startswith("fwd") else bb
    achieved = dom_bytes / (dom_avg * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                # the record is of the workload at its own size
                "traffic": recorded_traffic(f"{wl.name}:{dom}") if args.rows is None else None,
                "kernel": dom, "peak_source": peak_kind + (" (MEASURED_PEAKS.json hbm_gbs)" if peak_kind ==
                                                           "measured" else " (6.8 TB/s, profiling recipe)")}
    value = aggregate_gbs(world, step_bytes, args.steps, ms)

    # ---------------- end to end through the public API with host buffers
    # Every step copies its inputs in from pinned host memory and every output
    # back.  Two buffer sets alternate between steps and the copies run on
    # their own streams, so one step's copies overlap the other's kernels (the
    # usual input/output pipeline of a training loop); the calls are the
    # public fwd/bwd on the compute stream.
    e2e = None
    if args.e2e_steps > 0:
        hx = torch.from_numpy(pr.x.view(np.int16)).view(torch.bfloat16).pin_memory()
        hdy = torch.from_numpy(pr.dy.view(np.int16)).view(torch.bfloat16).pin_memory()
        hp = torch.from_numpy(pr.probs).pin_memory()

        def out_set():
            fo = gsa.alloc_qtensor(split, wl.width, wl.recipe, True, not wl.recompute, dev)
            bo = gsa.alloc_qtensor(split, wl.w_in, wl.recipe, True, True, dev)
            bo["dx"] = torch.empty((M, wl.w_in), dtype=torch.bfloat16, device=dev)
            bo["dprobs"] = torch.empty(M, dtype=torch.float32, device=dev)
            if wl.recompute:
                for k, v in gsa.alloc_qtensor(split, wl.width, wl.recipe, False, True, dev).items():
                    bo["y_" + k] = v
            return fo, bo

        sets = []
        for _ in range(2):
            sets.append({"x": torch.empty_like(x), "dy": torch.empty_like(dy), "p": torch.empty_like(p),
                         "out": {a: out_set() for a in acts}})
        def dev_outs(fo, bo):
            d = {("f", k): v for k, v in fo.items() if k != "_info"}
            d.update({("b", k): v for k, v in bo.items() if not k.endswith("_info")})
            return d
        sink = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                for k, v in dev_outs(*sets[0]["out"][acts[0]]).items()}
        h2d = hx.numel() * 2 + hdy.numel() * 2 + hp.numel() * 4
        d2h = len(acts) * sum(v.numel() * v.element_size() for v in sink.values())
        s_in = torch.cuda.Stream(device=dev)
        # the read-back is split over two streams (balanced by bytes) so that two copy engines share it
        s_outs = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
        load = [0, 0]
        lane_of = {}
        for key, v in sorted(sink.items(), key=lambda kv: -kv[1].numel() * kv[1].element_size()):
            j = 0 if load[0] <= load[1] else 1
            lane_of[key] = j
            load[j] += v.numel() * v.element_size()
        ev = {n: [torch.cuda.Event(), torch.cuda.Event()] for n in ("in", "comp", "out0", "out1")}
        for n in ev:
            for e in ev[n]:
                e.record(stream)

        def e2e_step(k):
            i = k % 2
            S = sets[i]
            s_in.wait_event(ev["comp"][i])          # the kernels of step k - 2 are done with these inputs
            with torch.cuda.stream(s_in):
                S["x"].copy_(hx, non_blocking=True)
                S["dy"].copy_(hdy, non_blocking=True)
                S["p"].copy_(hp, non_blocking=True)
                ev["in"][i].record(s_in)
            stream.wait_event(ev["in"][i])
            stream.wait_event(ev["out0"][i])        # the outputs of step k - 2 are back on the host
            stream.wait_event(ev["out1"][i])
            for a in acts:
                fo, bo = S["out"][a]
                gsa.fwd(S["x"], S["p"], split, a, wl.recipe, wl.rht, mask, True, not wl.recompute, False, prm, ws,
                        fo, stream)
                gsa.bwd(S["dy"], S["x"], S["p"], split, a, wl.recipe, wl.rht, mask, True, True, True, True,
                        wl.recompute, prm, ws, bo, stream)
                done = torch.cuda.Event()
                done.record(stream)
                for s_out in s_outs:
                    s_out.wait_event(done)
                for key, v in dev_outs(fo, bo).items():
                    with torch.cuda.stream(s_outs[lane_of[key]]):
                        sink[key].copy_(v, non_blocking=True)
            ev["comp"][i].record(stream)
            ev["out0"][i].record(s_outs[0])
            ev["out1"][i].record(s_outs[1])

        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_stream(stream)
        for k in range(args.e2e_steps):
            e2e_step(k)
        stream.wait_stream(s_in)
        for s_out in s_outs:
            stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), world)
        e2e = {"value": round(world * step_bytes * args.e2e_steps / (ems * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(ems / args.e2e_steps, 3),
               "pipeline": "inputs in on one copy stream, outputs out on two, two buffer sets alternating"}
        del sets, sink

    unfused = None
    if args.unfused_steps > 0:
        unfused = time_unfused(args, wl, acts, split, M, x, dy, p, prm, mask, ws, fwd_out, bwd_out, per, fb, bb,
                               dev)

    graph_safe = None
    if args.unfused_steps > 0:
        graph_safe = time_graph_safe(args, wl, acts, split, M, x, dy, p, prm, mask, fwd_out, bwd_out, per, dev)

    clk = None
    if args.clock_seconds > 0:
        kc = {}
        for a in acts:
            kc[f"fwd_{a}"] = (lambda a=a: gsa.fwd(x, p, split, a, wl.recipe, wl.rht, mask, True, not wl.recompute,
                                                  False, prm, ws, fwd_out))
            kc[f"bwd_{a}"] = (lambda a=a: gsa.bwd(dy, x, p, split, a, wl.recipe, wl.rht, mask, True, True, True, True,
                                                  wl.recompute, prm, ws, bwd_out))
        clk = kernel_clocks(kc, args.clock_seconds, local)

    configs = None
    names = [n for n in args.configs.split(",") if n and n != wl.name]
    if names and args.rows is None:
        configs = time_configs(names, dev, peak, peak_kind)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, _, _ = time_oracle(wl, acts, pr, 15.0)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": config_of(wl, acts, pr), "pct_hbm_peak": round(100 * value / world / peak, 2),
                "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "gpu_launches": gpu_launches, "bytes_per_step": step_bytes, "unfused_two_step": unfused,
                "graph_safe": graph_safe, "kernel_clocks": clk, "configs": configs}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gsa(args)


if __name__ == "__main__":
    main()
