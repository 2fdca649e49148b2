"""Benchmark of the GB300 shared-expert SwiGLU MLP library (one JSON line on rank 0).

Step = one pass of the hot path over one batch: the Kimi-K3 shared-expert layer
at decode, T = 64 tokens, hidden 7168, intermediate 6144, bf16
(mlp_swiglu_forward: gate_up + SiLU*mul kernel, down-projection kernel).
Headline: HBM TB/s = algorithmic bytes per step / device time per step, with the
same number also given as microseconds per layer.  Weights are cycled over
distinct copies (more bytes than L2), so no step reads its weights from L2.

Extra lines in the same JSON object: the T = 8192 prefill layer (TFLOP/s), the
TP8-sharded form (partials + shard_sum, and the partials summed inside the down
projection), one rank's partial at TP4/TP8/TP16 and the merged MLA q_a/kv_a projection.
`--only tp-sweep` prints instead the replicated-vs-sharded per-GPU time over token
counts and tp (kernels measured, collectives modelled).

`--impl reference` times the fp64 CPU oracle on the host cores instead.
Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run each rank runs an independent replica (the layer does not
need more than one GPU), timed between barriers, max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "shared-expert µs/layer & HBM TB/s at T=64; TFLOP/s at T=8192 (1 GB300)"
UNIT = "TB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
# GB300 vendor figures, reported beside the measured denominators: HBM3e 7.9 TB/s,
# dense bf16 2.25 PFLOP/s; and the tensor pipe's own rate, 152 SMs x 8192 dense bf16
# FLOP per SM per clock, scaled by the SM clock sampled during the run.
SPEC_HBM_GBS = 7900.0
SPEC_BF16_TFLOPS = 2250.0
N_SMS = 152
BF16_FLOP_PER_SM_CLK = 8192


# ------------------------------------------------------------------------------------------
# byte / flop models (algorithmic work per call)
# ------------------------------------------------------------------------------------------

def mlp_bytes(T, H, I):
    """Weights once + x read + y written (h stays on chip / in L2 and is not counted)."""
    return 2 * I * H * 2 + H * I * 2 + T * H * 2 + T * H * 2


def gate_up_bytes(T, H, I):
    """Bytes of the gate_up launch: W_gate_up + x + h written."""
    return 2 * I * H * 2 + T * H * 2 + T * I * 2


def mlp_flops(T, H, I):
    return 2 * T * (2 * I * H + H * I)


def gate_up_flops(T, H, I):
    return 2 * T * 2 * I * H


# ------------------------------------------------------------------------------------------
# environment helpers
# ------------------------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED, "source": "fallback"}


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ["tc.cu", "common.cuh", "tc.h"]:
        with open(os.path.join(ROOT, "moe_shared_expert_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key):
    """ncu DRAM bytes per launch recorded in profiles/traffic.json, if the kernel source
    still matches the one that was profiled; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_sha") != kernel_source_sha():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons around the timed region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.path = None
        self.windows = {}
        try:
            fd, self.path = tempfile.mkstemp(prefix="clk", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i", str(index),
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def mark(self, name, t0, t1):
        self.windows[name] = (t0, t1)

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()

    def summary(self, name, fallback_name=None):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
                except Exception:
                    continue
        if not rows:
            return None

        def pick(win):
            t0, t1 = self.windows[win]
            return [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]

        sel = pick(name) if name in self.windows else []
        window = name
        if len(sel) < 2 and fallback_name in self.windows:
            sel = pick(fallback_name)
            window = fallback_name
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": rows[-1][2], "reasons": [], "samples": 0, "window": window}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i, v in enumerate(r[4]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "power_w_max": max(r[3] for r in sel) if False else None,
                "reasons": reasons, "samples": len(sel), "window": window}


# ------------------------------------------------------------------------------------------
# distributed plumbing
# ------------------------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def done(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------

def dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def weight_copies(wgu0, wd0, n):
    """Copy 0 is the drawn weight; copies 1.. are row rotations of it (same distribution,
    distinct bytes and addresses), so consecutive steps stream different memory."""
    import torch
    gus, wds = [wgu0], [wd0]
    for i in range(1, n):
        gus.append(torch.roll(wgu0, shifts=977 * i, dims=0).contiguous())
        wds.append(torch.roll(wd0, shifts=331 * i, dims=0).contiguous())
    return gus, wds


# A device-side spin enqueued just before the start event, so that the host has queued
# the first steps before the timed region begins (the start event then records when
# the spin ends and the first step follows at once).  It is outside the timed region.
HOLD_CYCLES = 400_000   # about 0.2 ms at 2 GHz


def hold_device(stream):
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HOLD_CYCLES)


def time_loop(fn, K, stream, hold=True):
    """Device seconds of K steps: one event pair around all of them, no event between
    steps (an event between two kernels would cut the programmatic-dependent-launch
    overlap of consecutive layers)."""
    import torch
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    if hold:
        hold_device(stream)
    s.record(stream)
    for i in range(K):
        fn(i)
    e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) / 1e3   # seconds


def time_chunks(fn, K, stream, n_chunks=20):
    """time_loop in n_chunks consecutive chunks (an event between chunks, none between the
    steps of a chunk): (total seconds, seconds per step of each chunk).  Used only for the
    spread of per-step times, in a pass of its own with at least 50 steps per chunk."""
    import torch
    n_chunks = max(1, min(n_chunks, K))
    bounds = [K * c // n_chunks for c in range(n_chunks + 1)]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_chunks + 1)]
    hold_device(stream)
    evs[0].record(stream)
    for c in range(n_chunks):
        for i in range(bounds[c], bounds[c + 1]):
            fn(i)
        evs[c + 1].record(stream)
    evs[-1].synchronize()
    total = evs[0].elapsed_time(evs[-1]) / 1e3
    per = [evs[c].elapsed_time(evs[c + 1]) / 1e3 / (bounds[c + 1] - bounds[c]) for c in range(n_chunks)]
    return total, per


def percentiles(v, qs=(10, 50, 90)):
    s = sorted(v)
    return [s[min(len(s) - 1, max(0, int(round(q / 100 * (len(s) - 1)))))] for q in qs]


def one_launch_active() -> bool:
    import moe_shared_expert_gb300 as mse
    old = mse.set_tuning(mse.TUNE_ONE_LAUNCH, 1)
    mse.set_tuning(mse.TUNE_ONE_LAUNCH, old)
    return old == 1


# Library options for the decode leg.  The workload's x is a buffer that no kernel writes
# and each step's y and workspace are the same buffers, so a step's x never overlaps what
# the previous step writes: MSE_TUNE_X_EARLY lets each layer's gate_up weight stream start
# during the previous layer's split-K tail; with it, 12 k-blocks of L2 prefetch measured best,
# and MSE_TUNE_DOWN_FLAGS (the down kernel starts on each h block as soon as the gate_up
# kernel publishes it) took the layer from 53.6 to 50.2 us.  With these, the down projection
# on 128 CTAs (the library's rule takes 140, the largest grid near all SMs whose tiles are
# split at most three ways) measured 48.6 against 50.1 us, three alternating rounds on one
# box (144 and 152 CTAs: 48.3 and 48.5, but 144 also read 53.4 once).  It leaves 24 SMs to
# the next layer's first CTAs, which copy x in the host-buffer (e2e) step: 52.9 us there
# against 53.0-53.1 with 144.  The time with the library's default settings is reported
# beside the headline.
DECODE_TUNING = "x_early=1,l2_prefetch=12,down_flags=1,grid_down=128"
LIBRARY_DEFAULTS = (("x_early", 0), ("l2_prefetch", 8), ("down_flags", 0), ("grid_down", 0))


def bench_mlp(w, K, Wm, layers, dist, clocks=None, phase_steps=200, e2e_steps=None, spread_steps=2000,
              default_steps=0):
    """Replicated shared-expert layer: returns dict with device time, e2e time and phase times."""
    import torch
    import moe_shared_expert_gb300 as mse
    L = mse.lib()
    T, H, I = w.T, w.H, w.I
    x = dev_bf16(W.make_x(w))
    wgu_b, wd_b = W.make_mlp_weights(w)
    gus, wds = weight_copies(dev_bf16(wgu_b), dev_bf16(wd_b), layers)
    del wgu_b, wd_b
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ws = mse.new_mlp_workspace(T, H, I)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    px, py, pws, wsb = x.data_ptr(), y.data_ptr(), ws.data_ptr(), ws.numel()
    pgu = [g.data_ptr() for g in gus]
    pwd = [d.data_ptr() for d in wds]
    cap = T * H
    bad = [0]

    def step(i):
        j = i % layers
        bad[0] |= L.mlp_swiglu_forward(px, T, H, I, pgu[j], pwd[j], py, cap, pws, wsb, sp)

    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    dev_s = time_loop(step, K, stream)
    torch.cuda.synchronize()
    dist.barrier()
    t1 = time.time()
    if clocks:
        clocks.mark(f"{w.name}.timed", t0, t1)
    if bad[0]:
        raise RuntimeError(f"mlp_swiglu_forward returned an error status ({bad[0]})")
    st = mse.poll_device_error()
    if st:
        raise RuntimeError(f"device error {mse.STATUS.get(st)}")

    # the same loop with the library's default settings (no event inside its loop either)
    default_s = None
    if default_steps:
        saved = {k: mse.set_tuning(getattr(mse, "TUNE_" + k.upper()), d)
                 for k, d in LIBRARY_DEFAULTS}
        for i in range(Wm):
            step(i)
        torch.cuda.synchronize()
        default_s = time_loop(step, default_steps, stream) / default_steps
        for k, v in saved.items():
            mse.set_tuning(getattr(mse, "TUNE_" + k.upper()), v)
        for i in range(Wm):
            step(i)
        torch.cuda.synchronize()

    # spread of the per-step time: a separate pass of 20 chunks of >= 50 steps each
    # (the headline above has no event inside its loop)
    n_spread = 20 * max(50, spread_steps // 20) if spread_steps else 0
    chunk_s = time_chunks(step, n_spread, stream)[1] if n_spread else []

    # per-kernel durations: CUDA events recorded by the library between its two kernels
    n_ph = min(phase_steps, K)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_ph)]
    for trio in evs:            # torch only times events it has seen recorded; the
        for e in trio:          # library re-records them between its kernels below
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(n_ph):
        mse.set_phase_events(*evs[i])
        step(i)
    mse.set_phase_events(None, None, None)
    torch.cuda.synchronize()
    gate_up_ms = [e[0].elapsed_time(e[1]) for e in evs]
    down_ms = [e[1].elapsed_time(e[2]) for e in evs]
    layer_ms = [e[0].elapsed_time(e[2]) for e in evs]

    # end to end through the public API with host buffers: mlp_swiglu_forward_host reads x
    # from and writes y to page-locked host memory every step (the gate_up kernel copies x
    # from host memory itself, the down kernel writes y there; chained by programmatic
    # dependent launch)
    # at least 200 steps, so that start-up and the final synchronisation do not dominate
    n_e2e = e2e_steps if e2e_steps is not None else min(max(K, 200), 2000)
    xh = torch.from_numpy(W.make_x(w).view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    hws = mse.new_host_workspace(T, H, I)
    pxh, pyh, phws, hwsb = xh.data_ptr(), yh.data_ptr(), hws.data_ptr(), hws.numel()

    def e2e_step(i):
        j = i % layers
        bad[0] |= L.mlp_swiglu_forward_host(pxh, T, H, I, pgu[j], pwd[j], pyh, cap, phws, hwsb, sp)

    xd = torch.empty_like(x)

    def e2e_torch_step(i):   # the same with torch's host<->device copies around the device call
        j = i % layers
        xd.copy_(xh, non_blocking=True)
        bad[0] |= L.mlp_swiglu_forward(xd.data_ptr(), T, H, I, pgu[j], pwd[j], py, cap, pws, wsb, sp)
        yh.copy_(y, non_blocking=True)

    def host_timed(fn, n):
        # host wall clock from the first call to the final synchronize (host launch and
        # synchronisation costs included), and the stream's own events beside it
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        ev = time_loop(fn, n, stream, hold=False)
        torch.cuda.synchronize()
        return ev, time.perf_counter() - h0

    for i in range(min(Wm, 10)):
        e2e_step(i)
        e2e_torch_step(i)
    torch.cuda.synchronize()
    dist.barrier()
    e2e_s = e2e_host_s = e2e_torch_host_s = 0.0
    if n_e2e:
        e2e_s, e2e_host_s = host_timed(e2e_step, n_e2e)
        _, e2e_torch_host_s = host_timed(e2e_torch_step, n_e2e)
        if not torch.equal(yh.cuda(), y):
            raise RuntimeError("host-buffer output differs from the device output")
    if bad[0]:
        raise RuntimeError("error status in e2e loop")
    del gus, wds
    torch.cuda.empty_cache()
    return {"dev_s": dev_s, "K": K, "e2e_s": e2e_s, "e2e_host_s": e2e_host_s, "e2e_K": n_e2e, "chunk_s": chunk_s,
            "e2e_torch_host_s": e2e_torch_host_s, "default_s": default_s, "default_K": default_steps,
            "gate_up_ms": statistics.mean(gate_up_ms), "down_ms": statistics.mean(down_ms),
            "layer_ms": statistics.mean(layer_ms),
            "gate_up_ms_median": statistics.median(gate_up_ms), "h2d": T * H * 2, "d2h": T * H * 2}


def bench_tp8(w, K, Wm, layers):
    import torch
    import moe_shared_expert_gb300 as mse
    L = mse.lib()
    T, H, I, tp = w.T, w.H, w.I, w.tp
    x = dev_bf16(W.make_x(w))
    wgu_b, wd_b = W.make_mlp_weights(w)
    gus, wds = weight_copies(dev_bf16(wgu_b), dev_bf16(wd_b), layers)
    parts = torch.empty((tp, T, H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ws = mse.new_mlp_workspace(T, H, I)
    sp = torch.cuda.current_stream().cuda_stream
    pgu = [g.data_ptr() for g in gus]
    pwd = [d.data_ptr() for d in wds]
    bad = [0]

    def step(i):
        j = i % layers
        bad[0] |= L.mlp_swiglu_shard_partial(x.data_ptr(), T, H, I, pgu[j], pwd[j], tp, 0, tp, parts.data_ptr(),
                                             0, parts.numel(), ws.data_ptr(), ws.numel(), sp)
        bad[0] |= L.shard_sum(parts.data_ptr(), 0, tp, T, H, out.data_ptr(), out.numel(), sp)

    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    s = time_loop(step, K, torch.cuda.current_stream())
    if bad[0]:
        raise RuntimeError("tp8 error status")
    del gus, wds
    torch.cuda.empty_cache()
    return s / K


def bench_tp8_summed(w, K, Wm, layers):
    """All shards' partials summed inside the down projection (mlp_swiglu_shard_forward):
    no partial round trip, one [T x H] bf16 output."""
    import torch
    import moe_shared_expert_gb300 as mse
    L = mse.lib()
    T, H, I, tp = w.T, w.H, w.I, w.tp
    x = dev_bf16(W.make_x(w))
    wgu_b, wd_b = W.make_mlp_weights(w)
    gus, wds = weight_copies(dev_bf16(wgu_b), dev_bf16(wd_b), layers)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ws = mse.new_mlp_workspace(T, H, I)
    sp = torch.cuda.current_stream().cuda_stream
    pgu = [g.data_ptr() for g in gus]
    pwd = [d.data_ptr() for d in wds]
    bad = [0]

    def step(i):
        j = i % layers
        bad[0] |= L.mlp_swiglu_shard_forward(x.data_ptr(), T, H, I, pgu[j], pwd[j], tp, 0, tp, out.data_ptr(), 0,
                                             out.numel(), ws.data_ptr(), ws.numel(), sp)

    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    s = time_loop(step, K, torch.cuda.current_stream())
    if bad[0]:
        raise RuntimeError("summed shard forward error status")
    del gus, wds
    torch.cuda.empty_cache()
    return s / K


class RankShapes:
    """Decode weights (2 distinct copies, 528 MB) and tokens for per-rank timings: a step
    of one rank r of a tp-way split reads that rank's slices only, so steps cycle through
    the ranks and copies and no step finds its slice in L2.

    Steps are captured in a CUDA graph (every rank and copy once) and the graph is
    replayed: a rank's step is a few microseconds of device work, less than the host
    needs to issue it, so an eager loop would time the host.  Decode serving replays
    graphs in the same way."""

    def __init__(self, max_T, copies=2):
        import moe_shared_expert_gb300 as mse
        w = W.DECODE_T64
        self.H, self.I = w.H, w.I
        wgu_b, wd_b = W.make_mlp_weights(w)
        self.gus, self.wds = weight_copies(dev_bf16(wgu_b), dev_bf16(wd_b), copies)
        self.copies = copies
        self.x = dev_bf16(W.make_custom(77, 0, (max_T, self.H)))
        self.ws = {}
        self.mse = mse

    def workspace(self, T):
        if T not in self.ws:
            self.ws.clear()
            import torch
            torch.cuda.empty_cache()
            self.ws[T] = self.mse.new_mlp_workspace(T, self.H, self.I)
        return self.ws[T]

    def _time(self, step, n_steps, K, Wm, bad, graph=True):
        """Device seconds per step: steps 0..n_steps-1 captured once, replayed (or, with
        graph=False, K eager steps)."""
        import torch
        for i in range(max(Wm, n_steps)):      # eager warm-up (also sets kernel attributes)
            step(i)
        torch.cuda.synchronize()
        if not graph:
            K = K or 200
            return time_loop(step, K, torch.cuda.current_stream()) / K
        side = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(n_steps):
                step(i)
        if bad[0]:
            raise RuntimeError("error status while capturing")
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        if K is None:      # size the replay loop to about 0.15 s
            t = time_loop(lambda i: g.replay(), 5, torch.cuda.current_stream()) / 5
            K = int(max(10, min(4000, 0.15 / max(t, 1e-7))))
        else:
            K = max(1, K // n_steps)
        t = time_loop(lambda i: g.replay(), K, torch.cuda.current_stream())
        return t / (K * n_steps)

    def rank_partial(self, T, tp, K=None, Wm=5, graph=True):
        """One rank's partial [T x H] bf16 over its 1/tp of the weights (T gathered tokens)."""
        import torch
        L = self.mse.lib()
        H, I = self.H, self.I
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        ws = self.workspace(T)
        bad = [0]

        def step(i):
            r, c = i % tp, (i // tp) % self.copies
            sp = torch.cuda.current_stream().cuda_stream
            bad[0] |= L.mlp_swiglu_shard_partial(self.x.data_ptr(), T, H, I, self.gus[c].data_ptr(),
                                                 self.wds[c].data_ptr(), tp, r, 1, out.data_ptr(), 0, out.numel(),
                                                 ws.data_ptr(), ws.numel(), sp)

        t = self._time(step, tp * self.copies, K, Wm, bad, graph)
        if bad[0]:
            raise RuntimeError("rank partial error status")
        return t

    def replicated(self, T, K=None, Wm=5):
        """The full layer on T tokens (a replicated rank on its own tokens)."""
        import torch
        L = self.mse.lib()
        H, I = self.H, self.I
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        ws = self.workspace(T)
        bad = [0]

        def step(i):
            c = i % self.copies
            sp = torch.cuda.current_stream().cuda_stream
            bad[0] |= L.mlp_swiglu_forward(self.x.data_ptr(), T, H, I, self.gus[c].data_ptr(),
                                           self.wds[c].data_ptr(), out.data_ptr(), out.numel(), ws.data_ptr(),
                                           ws.numel(), sp)

        t = self._time(step, 2 * self.copies, K, Wm, bad)
        if bad[0]:
            raise RuntimeError("replicated error status")
        return t


def apply_tuning(spec: str) -> dict:
    """Set library tuning keys from 'name=value,...' (names of the binding's TUNE_* constants)."""
    import moe_shared_expert_gb300 as mse
    done = {}
    for item in filter(None, (t.strip() for t in spec.split(","))):
        name, value = item.split("=")
        key = getattr(mse, "TUNE_" + name.strip().upper())
        if mse.set_tuning(key, int(value)) < 0:
            raise ValueError(f"tuning {item} rejected")
        done[name.strip().lower()] = int(value)
    return done


def rank_bench(args):
    """One rank's partial alone (first of --sweep-tokens / --sweep-tp), eager launches:
    the small command that profiles of the per-rank kernels are taken on."""
    import torch
    torch.cuda.set_device(0)
    from moe_shared_expert_gb300 import _build
    _build.build()
    import moe_shared_expert_gb300 as mse
    mse.lib()
    tuning = apply_tuning(args.tune)
    T = int(args.sweep_tokens.split(",")[0])
    tp = int(args.sweep_tp.split(",")[0])
    rs = RankShapes(T)
    t = rs.rank_partial(T, tp, K=args.steps, Wm=args.warmup, graph=False)
    b = mlp_bytes(T, rs.H, rs.I // tp)
    print(json.dumps({"metric": "one rank's shard partial", "value": t * 1e6, "unit": "us", "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": f"rank_partial_tp{tp}_t{T}", "T": T, "tp": tp, "slice": rs.I // tp,
                                 "timing": "eager launches", "tuning": tuning},
                      "tbps_algorithmic": b / t / 1e12, "gpu_launches": 2 * args.steps}), flush=True)


def mla_bench(args):
    """The merged MLA projection alone (logical + rank-major outputs, T = 128, TP16 layout),
    eager launches cycling 24 weight copies: the small command that profiles of its kernel
    are taken on."""
    import torch
    torch.cuda.set_device(0)
    from moe_shared_expert_gb300 import _build
    _build.build()
    import moe_shared_expert_gb300 as mse
    mse.lib()
    tuning = apply_tuning(args.tune)
    w = W.MLA_MERGED
    t = bench_mla(w, args.steps, args.warmup)
    C = w.q_dim + w.kv_dim
    b = C * w.H * 2 + w.T * w.H * 2 + w.T * C * 2
    print(json.dumps({"metric": "merged MLA projection", "value": t * 1e6, "unit": "us", "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": w.name, "T": w.T, "H": w.H, "q_dim": w.q_dim, "kv_dim": w.kv_dim,
                                 "tp": w.tp, "timing": "eager launches", "tuning": tuning},
                      "tbps_algorithmic": b / t / 1e12, "gpu_launches": args.steps}), flush=True)


def collectives_model_s(T, H, tp, alpha_s, beta_Bps):
    """Modelled time of the block's two collectives (all-gather of the tokens, reduce-scatter
    of the bf16 partials): each alpha + (tp-1)/tp * T*H*2 bytes / beta."""
    return 2 * (alpha_s + (tp - 1) / tp * T * H * 2 / beta_Bps)


def crossovers(points, tps):
    """First group size T at which the replicated block is at least as fast, kernels only and
    with the modelled collectives (None: sharding faster at every T measured)."""
    out = {}
    for tp in tps:
        pts = sorted((p for p in points if p["tp"] == tp), key=lambda p: p["T"])
        k = [p["T"] for p in pts if p["sharded_kernel_us"] >= p["replicated_us"]]
        c = [p["T"] for p in pts if p["sharded_with_collectives_us"] >= p["replicated_us"]]
        out[str(tp)] = {"kernel_only_first_T_replicated_wins": min(k) if k else None,
                        "with_modelled_collectives_first_T_replicated_wins": min(c) if c else None}
    return out


def crossover_sensitivity(points, tps, H, alphas_us=(5.0, 10.0, 20.0), betas_gbs=(400.0, 800.0, 1600.0)):
    """The crossover (first T at which the replicated block is at least as fast as the
    sharded one with its two modelled collectives) for each collective model (alpha,
    beta), from the same measured kernel times: {tp: {"a{alpha}_b{beta}": T or None}}."""
    out = {}
    for tp in tps:
        pts = sorted((p for p in points if p["tp"] == tp), key=lambda p: p["T"])
        row = {}
        for a in alphas_us:
            for b in betas_gbs:
                c = [p["T"] for p in pts
                     if (p["sharded_kernel_us"] * 1e-6 + collectives_model_s(p["T"], H, tp, a * 1e-6, b * 1e9))
                     >= p["replicated_us"] * 1e-6]
                row[f"a{a:g}us_b{b:g}GBps"] = min(c) if c else None
        out[str(tp)] = row
    return out


def tp_sweep(args):
    """Per-GPU time of the replicated and the TP-sharded MLP block under sequence
    parallelism, over the group's token count T and tp.  Replicated: each rank runs the
    full layer on its T/tp own tokens.  Sharded: each rank runs its 1/tp slice on all T
    gathered tokens, plus an all-gather of the tokens and a reduce-scatter of the bf16
    partials.  Kernel times are measured; the two collectives are MODELLED (this library
    runs on one GPU): per collective  alpha + (tp-1)/tp * T*H*2 bytes / beta."""
    import torch
    torch.cuda.set_device(0)
    from moe_shared_expert_gb300 import _build
    _build.build()
    import moe_shared_expert_gb300 as mse
    mse.lib()
    tuning = apply_tuning(args.tune)
    Ts = [int(v) for v in args.sweep_tokens.split(",")]
    tps = [int(v) for v in args.sweep_tp.split(",")]
    rs = RankShapes(max(Ts))
    H, I = rs.H, rs.I
    alpha, beta = args.coll_alpha_us * 1e-6, args.coll_link_gbs * 1e9
    points = []
    for tp in tps:
        for T in Ts:
            if T % tp:
                continue
            t_rep = rs.replicated(T // tp)
            t_shard = rs.rank_partial(T, tp)
            coll = collectives_model_s(T, H, tp, alpha, beta)
            points.append({"tp": tp, "T": T, "replicated_us": t_rep * 1e6, "sharded_kernel_us": t_shard * 1e6,
                           "sharded_with_collectives_us": (t_shard + coll) * 1e6,
                           "collectives_model_us": coll * 1e6})
    cross = crossovers(points, tps)
    line = {"metric": "per-GPU µs of the MLP block: replicated vs TP-sharded under sequence parallelism",
            "unit": "us", "n_gpus": 1, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "tp_crossover_sweep", "H": H, "I": I, "tokens": Ts, "tp": tps,
                       "timing": "CUDA graph replay of every rank and weight copy", "tuning": tuning,
                       "weights": "decode weights, 2 copies cycled (and ranks cycled for the sharded slices)",
                       "collective_model": {"alpha_us": args.coll_alpha_us, "link_GBps": args.coll_link_gbs,
                                            "kind": "modelled, not measured"}},
            "points": points, "crossover": cross,
            "crossover_sensitivity": {
                "what": "first T at which replication wins, per collective model alpha (us) x beta (GB/s), "
                        "from the same measured kernel times",
                "by_tp": crossover_sensitivity(points, tps, H)}}
    print(json.dumps(line), flush=True)


def bench_mla(w, K, Wm, copies=24):
    import torch
    import moe_shared_expert_gb300 as mse
    L = mse.lib()
    T, H, q, kv, tp = w.T, w.H, w.q_dim, w.kv_dim, w.tp
    C = q + kv
    x = dev_bf16(W.make_x(w))
    w0 = dev_bf16(W.make_merged_weight(w))
    ws_ = [w0] + [torch.roll(w0, shifts=13 * i, dims=0).contiguous() for i in range(1, copies)]
    lo = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    rm = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    wsp = mse.new_merged_workspace(T, H, q, kv)
    sp = torch.cuda.current_stream().cuda_stream
    pw = [t.data_ptr() for t in ws_]
    bad = [0]

    def step(i):
        bad[0] |= L.merged_proj_forward(x.data_ptr(), T, H, pw[i % copies], q, kv, tp, lo.data_ptr(), rm.data_ptr(),
                                        T * C, wsp.data_ptr(), wsp.numel(), sp)

    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    s = time_loop(step, K, torch.cuda.current_stream())
    if bad[0]:
        raise RuntimeError("mla error status")
    return s / K


def cpu_oracle_baseline(w, max_rows=None):
    """The oracle as it stands on the host cores: the full decode step (all T token rows)."""
    import oracle
    x = W.make_x(w)
    wgu, wd = W.make_mlp_weights(w)
    rows = None if max_rows is None else np.arange(min(max_rows, w.T))
    n = w.T if rows is None else len(rows)
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.mlp_forward(x, wgu, wd, rows=rows, nthreads=threads)
    dt = time.perf_counter() - t0
    frac = n / w.T
    value = frac * mlp_bytes(w.T, w.H, w.I) / dt / 1e12
    return {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} of {w.T} token rows of the {w.name} layer (H={w.H}, I={w.I}), fp64, "
                      f"{dt:.2f} s wall on {threads} threads"}


def decode_config(w, layers, n_gpus):
    """The workload description shared by the GPU arm and the reference arm."""
    return {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "weights": "N(0,1/fan_in) bf16, seed 1",
            "x": "N(0,1) bf16", "l2": f"inputs larger than L2: {layers} distinct weight copies "
            f"({layers * 264.2:.0f} MB) cycled across steps", "parallelism": f"replicas x{n_gpus}"}


def tensor_peak_at_clock(sm_mhz):
    """Dense bf16 tensor-pipe rate of the whole GPU at the given SM clock (TFLOP/s)."""
    return N_SMS * BF16_FLOP_PER_SM_CLK * sm_mhz * 1e6 / 1e12 if sm_mhz else None


def gpu_arm(args):
    import torch
    dist = Dist()
    torch.cuda.set_device(dist.local)
    dist.init("nccl")
    from moe_shared_expert_gb300 import _build
    if dist.local == 0:
        _build.build()
    dist.barrier()
    import moe_shared_expert_gb300 as mse
    mse.lib()
    if args.two_launch:
        mse.set_tuning(mse.TUNE_ONE_LAUNCH, 0)
    tuning = apply_tuning(args.tune)
    peaks = load_peaks()
    clocks = ClockSampler(dist.local) if dist.rank == 0 else None

    w = W.DECODE_T64
    extra = {}
    if args.only == "prefill":
        r = None
    else:
        t_w0 = time.time()
        decode_tuning = {}
        saved = {}
        if not args.tune and not args.library_defaults:
            for item in DECODE_TUNING.split(","):
                name, v = item.split("=")
                saved[name] = mse.set_tuning(getattr(mse, "TUNE_" + name.upper()), int(v))
                decode_tuning[name] = int(v)
        r = bench_mlp(w, args.steps, args.warmup, args.layers, dist, clocks=clocks, spread_steps=args.spread_steps,
                      default_steps=max(args.steps, 2000) if decode_tuning else 0)
        for name, v in saved.items():
            mse.set_tuning(getattr(mse, "TUNE_" + name.upper()), v)
        tuning = {**decode_tuning, **tuning}
        dev_s = dist.max(r["dev_s"])
        e2e_s = dist.max(r["e2e_s"])
        if clocks:
            clocks.mark("decode.all", t_w0, time.time())

    if args.only != "decode":
        wp = W.PREFILL_T8192
        if args.prefill_tokens != wp.T:
            wp = dataclasses.replace(wp, T=args.prefill_tokens, name=f"prefill_t{args.prefill_tokens}")
        t_p0 = time.time()
        rp = bench_mlp(wp, args.prefill_steps, max(3, min(args.warmup, 5)), 2, dist, clocks=clocks,
                       phase_steps=min(10, args.prefill_steps), e2e_steps=0, spread_steps=0)
        if clocks:
            clocks.mark("prefill.all", t_p0, time.time())
        ps = dist.max(rp["dev_s"]) / args.prefill_steps
        gu_fl = gate_up_flops(wp.T, wp.H, wp.I)
        ach = gu_fl / (rp["gate_up_ms"] * 1e-3) / 1e12
        layer_tf = mlp_flops(wp.T, wp.H, wp.I) / ps / 1e12
        pclk = clocks.summary(f"{wp.name}.timed", "prefill.all") if clocks else None
        clk_peak = tensor_peak_at_clock(pclk.get("sm_mhz") if pclk else None)
        pkey = "pair_gate_up_prefill" if args.prefill_tokens >= 512 else "std_gate_up_prefill"
        extra[wp.name] = {
            "ms_per_layer": ps * 1e3, "tflops": layer_tf,
            "frac_of_bf16_peak_sustained": layer_tf / peaks["bf16_tflops_sustained"],
            "frac_of_bf16_peak_burst": layer_tf / peaks["bf16_tflops"],
            "frac_of_bf16_spec_2250": layer_tf / SPEC_BF16_TFLOPS,
            "frac_of_tensor_pipe_at_sampled_clock": layer_tf / clk_peak if clk_peak else None,
            "gate_up_ms": rp["gate_up_ms"], "down_ms": rp["down_ms"],
            "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": ach / peaks["bf16_tflops"], "traffic": profiled_traffic(pkey),
                         "peak_kind": f"burst bf16 ({peaks['source']})",
                         "frac_of_spec_2250": ach / SPEC_BF16_TFLOPS,
                         "frac_of_tensor_pipe_at_sampled_clock": ach / clk_peak if clk_peak else None},
            "clocks": pclk,
            "gpu_launches": 2 * args.prefill_steps,
        }
    if args.only == "all":
        w3 = W.TP8_EMULATED
        s3 = bench_tp8(w3, args.aux_steps, args.warmup, args.layers)
        b3 = mlp_bytes(w3.T, w3.H, w3.I)
        extra["tp8_emulated_t128"] = {"us": s3 * 1e6, "tbps_algorithmic": b3 / s3 / 1e12,
                                      "frac_of_hbm": b3 / s3 / 1e9 / peaks["hbm_gbs"],
                                      "partials_roundtrip_bytes": 2 * w3.tp * w3.T * w3.H * 2,
                                      "gpu_launches_per_step": 3}
        s3b = bench_tp8_summed(w3, args.aux_steps, args.warmup, args.layers)
        extra["tp8_summed_in_down_t128"] = {"us": s3b * 1e6, "tbps_algorithmic": b3 / s3b / 1e12,
                                            "frac_of_hbm": b3 / s3b / 1e9 / peaks["hbm_gbs"],
                                            "partials_roundtrip_bytes": 0, "gpu_launches_per_step": 2,
                                            "entry": "mlp_swiglu_shard_forward"}
        rs = RankShapes(64)
        per_rank = {}
        for tp in (4, 8, 16):
            t = rs.rank_partial(64, tp, K=args.aux_steps, Wm=args.warmup)
            # the same steps with early token loads (the steps are independent: x is a buffer
            # no kernel writes), as in the decode leg
            old = mse.set_tuning(mse.TUNE_X_EARLY, 1)
            te = rs.rank_partial(64, tp, K=args.aux_steps, Wm=args.warmup)
            mse.set_tuning(mse.TUNE_X_EARLY, old)
            b = mlp_bytes(64, w.H, w.I // tp)
            per_rank[f"tp{tp}"] = {"us": t * 1e6, "us_x_early": te * 1e6, "slice": w.I // tp,
                                   "tbps_algorithmic": b / t / 1e12, "frac_of_hbm": b / t / 1e9 / peaks["hbm_gbs"],
                                   "timing": "CUDA graph replay; us: library defaults, us_x_early: x_early=1"}
        extra["one_rank_partial_t64"] = per_rank
        del rs
        torch.cuda.empty_cache()
        w4 = W.MLA_MERGED
        s4 = bench_mla(w4, args.aux_steps, args.warmup)
        old = mse.set_tuning(mse.TUNE_X_EARLY, 1)
        s4e = bench_mla(w4, args.aux_steps, args.warmup)
        mse.set_tuning(mse.TUNE_X_EARLY, old)
        C = w4.q_dim + w4.kv_dim
        b4 = C * w4.H * 2 + w4.T * w4.H * 2 + w4.T * C * 2
        extra["mla_merged_tp16_t128"] = {"us": s4 * 1e6, "us_x_early": s4e * 1e6, "tbps_algorithmic": b4 / s4 / 1e12,
                                         "frac_of_hbm": b4 / s4 / 1e9 / peaks["hbm_gbs"],
                                         "outputs": "logical + rank-major", "weight_copies_cycled": 24}
    if clocks:
        clocks.stop()

    if dist.rank != 0:
        dist.done()
        return
    if r is None:   # prefill only: report the prefill measurement as the line
        pf = extra[wp.name]
        line = {"metric": METRIC, "value": pf["tflops"], "unit": "TFLOP/s", "n_gpus": dist.world,
                "steps": args.prefill_steps, "warmup": args.warmup, "ms_per_step": pf["ms_per_layer"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": {"workload": wp.name, "T": wp.T, "H": wp.H, "I": wp.I},
                "roofline": pf["roofline"], "gpu_launches": pf["gpu_launches"]}
        print(json.dumps(line), flush=True)
        dist.done()
        return
    N = dist.world
    K = args.steps
    bytes_step = mlp_bytes(w.T, w.H, w.I)
    ms = dev_s / K * 1e3
    value = N * bytes_step * K / dev_s / 1e12
    if one_launch_active():
        # one launch per layer: the dominant kernel is the whole layer
        k_bytes, k_ms, launches = bytes_step, r["layer_ms"], K
        k_name = "swapab_mlp_kernel<EPI_BF16> (gate_up + SiLU*mul, then down; one launch)"
        k_key = "swapab_mlp_decode"
    else:
        k_bytes, k_ms, launches = gate_up_bytes(w.T, w.H, w.I), r["gate_up_ms"], 2 * K
        k_name = "swapab_kernel<EPI_SWIGLU> (gate_up + SiLU*mul)"
        k_key = "swapab_gate_up_decode"
    ach = k_bytes / (k_ms * 1e-3) / 1e9
    e2e_host_s = dist.max(r["e2e_host_s"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": N, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "us_per_layer": ms * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": decode_config(w, args.layers, N),
        "library_tuning": tuning or None,
        "timing": "one CUDA event pair around all timed steps on the launching stream (no event between steps)",
        "clocks": clocks.summary(f"{w.name}.timed", "decode.all") if clocks else None,
        "e2e": {"value": N * bytes_step * r["e2e_K"] / e2e_host_s / 1e12 if r["e2e_K"] else None, "unit": UNIT,
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "steps": r["e2e_K"],
                "us_per_layer_host_clock": e2e_host_s / r["e2e_K"] * 1e6 if r["e2e_K"] else None,
                "us_per_layer_stream_events": e2e_s / r["e2e_K"] * 1e6 if r["e2e_K"] else None,
                "us_per_layer_torch_copies_host_clock":
                    r["e2e_torch_host_s"] / r["e2e_K"] * 1e6 if r["e2e_K"] else None,
                "entry": "mlp_swiglu_forward_host (x read from and y written to page-locked host memory)",
                "timing": "host wall clock from the first call to the final synchronize; stream events beside it"},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": profiled_traffic(k_key),
                     "kernel": k_name, "kernel_ms": k_ms, "algorithmic_bytes": k_bytes,
                     "peak_kind": f"HBM copy ({peaks['source']})",
                     "frac_of_spec_7900": ach / SPEC_HBM_GBS},
        "step_frac_of_hbm": bytes_step / (dev_s / K) / 1e9 / peaks["hbm_gbs"],
        "step_frac_of_hbm_spec_7900": bytes_step / (dev_s / K) / 1e9 / SPEC_HBM_GBS,
    }
    if r.get("default_s"):
        line["us_per_layer_library_defaults"] = r["default_s"] * 1e6
        line["library_defaults"] = (f"{r['default_K']} steps timed the same way with the library's default "
                                    f"settings ({', '.join(f'{k}={v}' for k, v in LIBRARY_DEFAULTS)})")
    if r["chunk_s"]:
        line["us_per_layer_p10_p50_p90"] = [v * 1e6 for v in percentiles(r["chunk_s"])]
        line["us_per_layer_spread"] = (f"per-step time of {len(r['chunk_s'])} consecutive chunks of a separate "
                                       f"pass after the timed region")
    if launches == 2 * K:
        line["down_kernel_ms"] = r["down_ms"]
    if extra:
        line["also"] = extra
    if not args.no_cpu_baseline and N == 1:
        line["cpu_baseline"] = cpu_oracle_baseline(w)
    print(json.dumps(line), flush=True)
    dist.done()


# ------------------------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ------------------------------------------------------------------------------------------

def reference_arm(args):
    dist = Dist()
    if dist.rank != 0:
        return
    import oracle
    oracle.build()
    w = W.DECODE_T64
    x = W.make_x(w)
    wgu, wd = W.make_mlp_weights(w)
    threads = oracle.default_threads()
    # calibrate one token row, then size each step's sample so the whole run stays
    # within a few minutes: r token rows of the layer, or one row of one intermediate
    # slice (a shard partial) when even one full row per step is too much.
    t0 = time.perf_counter()
    oracle.mlp_forward(x, wgu, wd, rows=np.array([0]), nthreads=threads)
    t_row = time.perf_counter() - t0
    budget = float(args.ref_budget_s)
    per_step = budget / max(1, args.steps + args.warmup)
    if per_step >= t_row:
        rows = int(min(w.T, max(1, per_step // t_row)))
        tp = 1
    else:
        rows = 1
        tp = 96                                    # one 64-wide intermediate slice
    sample_rows = np.arange(rows)
    frac = rows / w.T / tp

    def step(i):
        if tp == 1:
            oracle.mlp_forward(x, wgu, wd, rows=sample_rows, nthreads=threads)
        else:
            oracle.shard_partial(x, wgu, wd, tp, i % tp, oracle.BF16, rows=sample_rows, nthreads=threads)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = frac * mlp_bytes(w.T, w.H, w.I) * args.steps / dt / 1e12
    sample = (f"{rows} of {w.T} token rows" if tp == 1 else f"1 token row x 1/{tp} intermediate slice") + \
             f" of the {w.name} layer per step, fp64 oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(w, args.layers, dist.world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=4, help="distinct weight copies cycled")
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--aux-steps", type=int, default=2000)
    ap.add_argument("--decode-only", action="store_true", help="same as --only decode")
    ap.add_argument("--only", default="all", choices=["all", "decode", "prefill", "tp-sweep", "rank", "mla"])
    ap.add_argument("--sweep-tokens", default="16,32,64,128,256,512,1024,2048")
    ap.add_argument("--sweep-tp", default="4,8,16")
    ap.add_argument("--coll-alpha-us", type=float, default=10.0,
                    help="modelled fixed cost of one collective (tp-sweep)")
    ap.add_argument("--coll-link-gbs", type=float, default=800.0,
                    help="modelled per-GPU link bandwidth of one collective (tp-sweep)")
    ap.add_argument("--tune", default="",
                    help="library tuning for the run, e.g. one_launch=2,grid=144 (names of mse.TUNE_*)")
    ap.add_argument("--prefill-tokens", type=int, default=8192)
    ap.add_argument("--library-defaults", action="store_true",
                    help="time the decode leg with the library's default settings only (no DECODE_TUNING)")
    ap.add_argument("--spread-steps", type=int, default=2000,
                    help="steps of the separate pass that gives the p10/p50/p90 spread (0: none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget-s", type=float, default=120.0)
    ap.add_argument("--two-launch", action="store_true",
                    help="decode layer as two launches (gate_up, down) instead of one")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.decode_only:
        args.only = "decode"
    if args.impl == "reference":
        reference_arm(args)
    elif args.only == "tp-sweep":
        tp_sweep(args)
    elif args.only == "rank":
        rank_bench(args)
    elif args.only == "mla":
        mla_bench(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
