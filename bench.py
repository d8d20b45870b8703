#!/usr/bin/env python3
"""Benchmark of the gated-delta SSM layer step on GB300.

Headline (``value``): batched decode, 64 sequences x 48 V heads x 128x128 fp32
state (192 MiB), conv_dim 10240, input rows 20480 apart with z inside the row,
one fused launch per step: recurrent-state HBM GB/s (state bytes read + written
per step / device time per step). The same JSON line carries the other
workloads measured in the same run (single-sequence decode in a CUDA graph over
64 rotating state buffers, K=2 verify + commit, chunked prefill tokens/s), the
roofline of the dominant kernel, an end-to-end figure through the C ABI with
host buffers, the clock record, and the fp64 CPU oracle timed on a bounded
sample of the headline workload on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

For N > 1 launch under torch.distributed.run: each rank runs its own replica
of the workload on its own GPU (sequences are independent: no collective on
the data path); value = all ranks' state bytes / the slowest rank's time.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_ssm_gb300 import synth  # noqa: E402

METRIC = "GDN decode: state HBM GB/s (% of peak), seqs/s; prefill tokens/s"
HEADLINE = "decode_b64"
KERNEL_SOURCES = ["gated_delta_ssm_gb300/csrc/decode.cu", "gated_delta_ssm_gb300/csrc/gdn_device.cuh",
                  "gated_delta_ssm_gb300/csrc/cluster.cuh"]


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def reduce_max(dist, value: float, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank processes the same units; time is the slowest rank's."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during a region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def src_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


NOMINAL_HBM_GBS = 8000.0   # the GB300's nominal HBM3e bandwidth, for a second denominator


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("src_sha") != src_hash():
        return None
    return d.get("bytes_per_launch")


def e2e_group_sizes(n_steps: int, group: int) -> list:
    """Steps per group of the end-to-end loop: groups of `group` steps, except one step
    in the first and in the last group (the first group's input copy and the last
    group's output copy are the ones that nothing overlaps)."""
    if n_steps <= 2:
        return [1] * n_steps
    mid = n_steps - 2
    return [1] + [group] * (mid // group) + ([mid % group] if mid % group else []) + [1]


def decode_bytes(shape: synth.Shape) -> dict:
    """Algorithmic HBM bytes of one fused decode step (each compulsory byte counted once)."""
    B, Hv, Hq, d, W, cd = shape.B, shape.Hv, shape.Hq, shape.d, shape.W, shape.conv_dim
    act = 2 if shape.act_dtype == "bf16" else 4
    state = 2 * B * Hv * d * d * 4
    hist = 2 * B * cd * (W - 1) * 4
    acts = B * (cd + Hv * d + 2 * Hv) * act
    out = B * Hv * d * 4
    params = cd * W * 4 + (2 * Hv + d) * 4
    return {"state": state, "total": state + hist + acts + out + params}


def prefill_work(shape: synth.Shape) -> dict:
    """Algorithmic work of one chunked prefill call: the chunk form's dense products
    (5 x 2C^2 d + 3 x 2 C d^2 per (chunk, V head), C = 64, d = 128: ~11.6 MFLOP,
    counted once per product) and the compulsory HBM bytes (x read, z read, outputs
    written, state read + written, conv history read + written)."""
    C, d = 64, shape.d
    n_units = shape.B * shape.Hv * ((shape.T + C - 1) // C)
    flops = n_units * (5 * 2 * C * C * d + 3 * 2 * C * d * d)
    act = 2 if shape.act_dtype == "bf16" else 4
    rows = shape.B * shape.T
    nbytes = (rows * (shape.conv_dim + shape.Hv * d + 2 * shape.Hv) * act + rows * shape.Hv * d * 4
              + 2 * shape.B * shape.Hv * d * d * 4 + 2 * shape.B * shape.conv_dim * (shape.W - 1) * 4)
    return {"flops": float(flops), "bytes": float(nbytes)}


# ------------------------------------------------------------------ GPU measurements
class Gpu:
    def __init__(self, local_rank: int):
        import torch
        import gated_delta_ssm_gb300 as gdn
        from gated_delta_ssm_gb300 import build as gbuild
        self.torch, self.gdn = torch, gdn
        gbuild.build()
        gdn.load()
        torch.cuda.set_device(local_rank)
        self.dev = torch.device("cuda", local_rank)
        self.stream = torch.cuda.current_stream()
        self.launches = 0

    def upload(self, shape, inp, copies=1):
        torch = self.torch
        dt = shape.act_dtype

        def t(a, dtype="f32"):
            if dtype == "bf16":
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(self.dev)
            return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(self.dev)

        d = {"x": t(inp["x"], dt), "alpha": t(inp["alpha"], dt), "beta_logit": t(inp["beta_logit"], dt)}
        d["z"] = d["x"][..., shape.conv_dim:shape.conv_dim + shape.Hv * shape.d] if shape.z_in_x else t(inp["z"], dt)
        for k in ("conv_w", "dt", "A_log", "norm_w"):
            d[k] = t(inp[k])
        st, hi = t(inp["state"]), t(inp["hist"])
        d["states"] = [st] + [st.clone() for _ in range(copies - 1)]
        d["hists"] = [hi] + [hi.clone() for _ in range(copies - 1)]
        d["accept"] = torch.from_numpy(inp["accept"]).to(self.dev)
        return d

    def dims(self, shape):
        return self.gdn.Dims(shape.B, shape.Hq, shape.Hv, shape.d, shape.W, shape.xs,
                             shape.xs if shape.z_in_x else shape.Hv * shape.d, shape.Hv)

    def params(self, d):
        return self.gdn.Params(d["conv_w"], d["dt"], d["A_log"], d["norm_w"], 1e-6, 1e-6)

    def time_steps(self, fn, steps, warmup):
        """Device time (s) of `steps` calls issued back to back after `warmup` untimed
        ones: one pair of CUDA events on the launching stream around all of them, so
        consecutive launches overlap as they do in a serving loop (each decode launch is a
        programmatic dependent of the one before it). Returns the mean per call, once per
        call. The callable receives the step index (used to rotate buffers)."""
        torch = self.torch
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        for i in range(steps):
            fn(warmup + i)
        b.record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) * 1e-3 / steps] * steps

    def time_each(self, fn, steps, warmup):
        """Per-call device times (s), an event pair around each call. The event recorded
        between two launches keeps the second from starting before the first ends, so
        this is the serialised time of one launch."""
        torch = self.torch
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record(self.stream)
            fn(warmup + i)
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) * 1e-3 for a, b in ev]

    # -- headline: batched decode
    def decode_b64(self, steps, warmup, dist=None):
        torch, gdn = self.torch, self.gdn
        shape = synth.WORKLOADS["decode_b64"]
        inp = synth.make_inputs(shape, seed=2)
        nbuf = 3                                   # 3 x 192 MiB state: every step reads cold state
        d = self.upload(shape, inp, copies=nbuf)
        dims, prm = self.dims(shape), self.params(d)
        out = torch.empty(shape.B, shape.Hv, shape.d, device=self.dev)

        def step(i):
            gdn.decode_step(d["states"][i % nbuf], d["hists"][i % nbuf], d["x"], d["z"], d["alpha"],
                            d["beta_logit"], prm, out, dims)

        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        times = self.time_steps(step, steps, warmup)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        self.launches += steps
        self.per_launch_s = statistics.mean(self.time_each(step, steps, warmup))
        self.launches += steps
        # end to end through the C ABI: inputs from pinned host memory each step, output back
        hx = torch.from_numpy(np.ascontiguousarray(inp["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
        ha = torch.from_numpy(np.ascontiguousarray(inp["alpha"]).view(np.int16)).view(torch.bfloat16).pin_memory()
        hb = torch.from_numpy(np.ascontiguousarray(inp["beta_logit"]).view(np.int16)).view(torch.bfloat16).pin_memory()
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = hx.numel() * 2 + ha.numel() * 2 + hb.numel() * 2
        d2h = hout.numel() * 4

        def e2e_step(i):
            d["x"].copy_(hx, non_blocking=True)
            d["alpha"].copy_(ha, non_blocking=True)
            d["beta_logit"].copy_(hb, non_blocking=True)
            step(i)
            hout.copy_(out, non_blocking=True)

        serial_times = self.time_steps(e2e_step, steps, max(3, warmup // 2))
        self.launches += steps

        # The serving loop: every step's inputs still come from pinned host memory and
        # its output still goes back to pinned host memory, but the copies run on a
        # second stream while the kernels run. Steps go in groups (of G, except one step
        # in the first and the last): the inputs of group g+1 (its steps' inputs, back
        # to back in pinned host memory) travel in one copy while group g runs, and the
        # outputs of a group come back in one copy.
        # The kernels of a group follow one another with nothing between them in the
        # stream, so each is a programmatic dependent of the one before, as in the
        # kernel-only loop, and the host issues one call per step. A step's three
        # inputs are its x rows, then its alpha rows, then its beta-logit rows; the step
        # reads views of its slot. Two sets of slots alternate.
        G = 4
        cd = shape.conv_dim
        copy = torch.cuda.Stream(device=self.dev)
        comp = self.stream
        nx, na = hx.numel(), ha.numel()
        one = torch.cat([hx.reshape(-1), ha.reshape(-1), hb.reshape(-1)])
        per = one.numel()
        hpk = one.repeat(G).pin_memory()                         # G steps' inputs
        dpk = [torch.empty_like(hpk, device=self.dev) for _ in range(2)]
        slot = [[dpk[sset][u * per:(u + 1) * per] for u in range(G)] for sset in range(2)]
        dx = [[t[:nx].view(d["x"].shape) for t in slot[sset]] for sset in range(2)]
        da = [[t[nx:nx + na].view(d["alpha"].shape) for t in slot[sset]] for sset in range(2)]
        db = [[t[nx + na:].view(d["beta_logit"].shape) for t in slot[sset]] for sset in range(2)]
        dz = [[t[..., cd:cd + shape.Hv * shape.d] for t in dx[sset]] for sset in range(2)]
        outs = [torch.empty((G,) + tuple(out.shape), dtype=out.dtype, device=self.dev) for _ in range(2)]
        houts = [torch.empty((G,) + tuple(out.shape), dtype=out.dtype).pin_memory() for _ in range(2)]
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]     # a slot set's inputs are in
        ev_k = [torch.cuda.Event(), torch.cuda.Event()]      # its kernels are done
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]    # its outputs are back on the host
        assert per * one.element_size() == h2d

        def pipelined(n_steps, first):
            size = e2e_group_sizes(n_steps, G)
            n_groups = len(size)
            start = [sum(size[:g]) for g in range(n_groups)]

            def h2d_group(g):
                sset = g % 2
                with torch.cuda.stream(copy):
                    if g >= 2:
                        copy.wait_event(ev_k[sset])          # group g-2 has read these slots
                    dpk[sset][:size[g] * per].copy_(hpk[:size[g] * per], non_blocking=True)
                    ev_in[sset].record(copy)

            h2d_group(0)
            for g in range(n_groups):
                sset = g % 2
                if g + 1 < n_groups:
                    h2d_group(g + 1)
                comp.wait_event(ev_in[sset])
                if g >= 2:
                    comp.wait_event(ev_out[sset])            # group g-2's outputs have left
                xs, zs, als, bls, os_ = dx[sset], dz[sset], da[sset], db[sset], outs[sset]
                for u in range(size[g]):
                    i = start[g] + u
                    gdn.decode_step(d["states"][(first + i) % nbuf], d["hists"][(first + i) % nbuf],
                                    xs[u], zs[u], als[u], bls[u], prm, os_[u], dims, stream=comp)
                ev_k[sset].record(comp)
                with torch.cuda.stream(copy):
                    copy.wait_event(ev_k[sset])
                    houts[sset][:size[g]].copy_(outs[sset][:size[g]], non_blocking=True)
                    ev_out[sset].record(copy)

        pipelined(max(3, warmup), 0)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(copy)
        comp.wait_event(t0)
        pipelined(steps, 0)
        comp_done = torch.cuda.Event()
        comp_done.record(comp)
        copy.wait_event(comp_done)
        t1.record(copy)
        torch.cuda.synchronize()
        self.launches += steps
        e2e_total = t0.elapsed_time(t1) * 1e-3
        return shape, times, e2e_total, h2d, d2h, sum(serial_times)

    # -- single-sequence decode: 1000 steps in one CUDA graph, 64 rotating state buffers
    def decode_b1(self, n_steps=1000, nbuf=64, reps=3):
        torch, gdn = self.torch, self.gdn
        shape = synth.WORKLOADS["decode_b1"]
        inp = synth.make_inputs(shape, seed=1)
        d = self.upload(shape, inp, copies=nbuf)
        dims, prm = self.dims(shape), self.params(d)
        out = torch.empty(shape.B, shape.Hv, shape.d, device=self.dev)
        for i in range(nbuf):                       # warm the kernels before capture
            gdn.decode_step(d["states"][i], d["hists"][i], d["x"], d["z"], d["alpha"],
                            d["beta_logit"], prm, out, dims)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(n_steps):
                    gdn.decode_step(d["states"][i % nbuf], d["hists"][i % nbuf], d["x"], d["z"],
                                    d["alpha"], d["beta_logit"], prm, out, dims)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) * 1e-3)
            self.launches += n_steps
        per = best / n_steps
        st = decode_bytes(shape)["state"]
        return {"us_per_step": per * 1e6, "state_GBps": st / per / 1e9, "steps_in_graph": n_steps,
                "state_buffers": nbuf}

    # -- the batched decode with bf16 state and output (serving option)
    def decode_b64_bf16_state(self, steps, warmup):
        torch, gdn = self.torch, self.gdn
        shape = synth.WORKLOADS["decode_b64"]
        inp = synth.make_inputs(shape, seed=2)
        d = self.upload(shape, inp)
        bits = torch.from_numpy(synth.bf16_round(inp["state"]).view(np.int16)).view(torch.bfloat16)
        nbuf = 3                                   # 3 x 96 MiB bf16 state: beyond L2
        states = [bits.to(self.dev) for _ in range(nbuf)]
        dims = self.dims(shape)
        prm = self.params(d)
        out = torch.empty(shape.B, shape.Hv, shape.d, device=self.dev, dtype=torch.bfloat16)

        def step(i):
            gdn.decode_step_bf16_state(states[i % nbuf], d["hists"][0], d["x"], d["z"], d["alpha"],
                                       d["beta_logit"], prm, out, dims)

        t = self.time_steps(step, steps, warmup)
        self.launches += steps
        m = statistics.mean(t)
        sb = 2 * shape.B * shape.Hv * shape.d * shape.d * 2
        hbm_peak, _, _ = measured_peaks()
        return {"us_per_step": m * 1e6, "state_GBps": sb / m / 1e9,
                "pct_of_peak": 100.0 * sb / m / 1e9 / hbm_peak, "seqs_per_s": shape.B / m}

    # -- K=2 verify + commit
    def verify_k2(self, steps, warmup):
        torch, gdn = self.torch, self.gdn
        shape = synth.WORKLOADS["verify_k2"]
        inp = synth.make_inputs(shape, seed=3)
        nbuf = 3
        d = self.upload(shape, inp, copies=nbuf)
        snaps = [torch.empty_like(d["states"][0]) for _ in range(nbuf)]
        hsnaps = [torch.empty_like(d["hists"][0]) for _ in range(nbuf)]
        dims, prm = self.dims(shape), self.params(d)
        out = torch.empty(shape.B, 2, shape.Hv, shape.d, device=self.dev)

        def vstep(i):
            j = i % nbuf
            gdn.verify_k2(d["states"][j], d["hists"][j], snaps[j], hsnaps[j], d["x"], d["z"],
                          d["alpha"], d["beta_logit"], prm, out, dims)

        def cstep(i):
            j = i % nbuf
            gdn.verify_commit(d["states"][j], d["hists"][j], snaps[j], hsnaps[j], d["accept"], dims)

        # the token after the verify: with the rollback folded in (each sequence reads the
        # snapshot its accepted count selects), or the plain step that follows a commit;
        # one token row of the two-token buffers is the step's input
        zs = shape.xs if shape.z_in_x else shape.Hv * shape.d
        step_dims = gdn.Dims(shape.B, shape.Hq, shape.Hv, shape.d, shape.W, 2 * shape.xs, 2 * zs, 2 * shape.Hv)
        sout = torch.empty(shape.B, shape.Hv, shape.d, device=self.dev)
        tok = {k: d[k][:, 0] for k in ("x", "z", "alpha", "beta_logit")}

        def sstep(i):
            j = i % nbuf
            gdn.decode_step_select(d["states"][j], d["hists"][j], snaps[j], hsnaps[j], 1, d["accept"], 2,
                                   tok["x"], tok["z"], tok["alpha"], tok["beta_logit"], prm, sout, step_dims)

        def pstep(i):
            j = i % nbuf
            gdn.decode_step(d["states"][j], d["hists"][j], tok["x"], tok["z"], tok["alpha"],
                            tok["beta_logit"], prm, sout, step_dims)

        tv = self.time_steps(vstep, steps, warmup)
        tc = self.time_steps(cstep, steps, warmup)
        ts = self.time_steps(sstep, steps, warmup)
        tp = self.time_steps(pstep, steps, warmup)
        self.launches += 4 * steps
        sb = shape.B * shape.Hv * shape.d * shape.d * 4
        n_rb = int((inp["accept"] == 1).sum())
        mv, mc, ms, mp = (statistics.mean(t) for t in (tv, tc, ts, tp))
        return {"verify_us": mv * 1e6, "verify_state_GBps": 3 * sb / mv / 1e9,
                "commit_us": mc * 1e6, "commit_GBps": 2 * n_rb * (sb // shape.B) / mc / 1e9,
                "rollbacks": n_rb, "select_step_us": ms * 1e6, "step_us": mp * 1e6,
                "verify_commit_step_us": (mv + mc + mp) * 1e6, "verify_select_step_us": (mv + ms) * 1e6}

    # -- generic-K draft verification (K = 4) + commit, K=2 verify's batch
    def verify_kn(self, steps, warmup, K=4):
        torch, gdn = self.torch, self.gdn
        shape = synth.Shape(B=32, T=K, Hq=16, Hv=32, warm=True)
        inp = synth.make_inputs(shape, seed=5)
        nbuf = 3                                   # 3 x 64 MiB state (+ snapshots): beyond L2
        d = self.upload(shape, inp, copies=nbuf)
        B, Hv, dd = shape.B, shape.Hv, shape.d
        snaps = [torch.empty(B, K - 1, Hv, dd, dd, device=self.dev) for _ in range(nbuf)]
        hsnaps = [torch.empty((B, K) + tuple(d["hists"][0].shape[1:]), device=self.dev)
                  for _ in range(nbuf)]
        dims, prm = self.dims(shape), self.params(d)
        out = torch.empty(B, K, Hv, dd, device=self.dev)
        accept = torch.arange(B, dtype=torch.int32, device=self.dev) % K + 1

        def vstep(i):
            j = i % nbuf
            gdn.verify_kn(d["states"][j], d["hists"][j], snaps[j], hsnaps[j], d["x"], d["z"],
                          d["alpha"], d["beta_logit"], prm, out, dims, K)

        def cstep(i):
            j = i % nbuf
            gdn.verify_commit_kn(d["states"][j], d["hists"][j], snaps[j], hsnaps[j], accept, dims, K)

        tv = self.time_steps(vstep, steps, warmup)
        tc = self.time_steps(cstep, steps, warmup)
        self.launches += 2 * steps
        sb = B * Hv * dd * dd * 4
        mv, mc = statistics.mean(tv), statistics.mean(tc)
        n_rb = int((accept < K).sum())
        # state bytes: read once, the K-1 snapshots and the committed state written
        return {"K": K, "verify_us": mv * 1e6, "verify_state_GBps": (1 + K) * sb / mv / 1e9,
                "commit_us": mc * 1e6, "commit_GBps": 2 * n_rb * (sb // B) / mc / 1e9,
                "rollbacks": n_rb}

    # -- token-parallel conv + SiLU + Q/K L2 over the prefill workload
    def conv_tokens(self, steps, warmup):
        torch, gdn = self.torch, self.gdn
        shape = synth.WORKLOADS["prefill"]
        inp = synth.make_inputs(shape, seed=6)
        d = self.upload(shape, inp)
        B, T, cd = shape.B, shape.T, shape.conv_dim
        out = torch.empty(B, T, cd, device=self.dev)
        dims = self.dims(shape)

        def step(i):
            gdn.conv_update(d["hists"][0], d["x"], d["conv_w"], out, dims, T, 1e-6)

        t = self.time_steps(step, steps, warmup)
        self.launches += steps
        m = statistics.mean(t)
        act = 2 if shape.act_dtype == "bf16" else 4
        nbytes = B * T * cd * (act + 4) + 2 * B * cd * (shape.W - 1) * 4 + cd * shape.W * 4
        return {"us": m * 1e6, "GBps": nbytes / m / 1e9, "algorithmic_bytes": nbytes}

    # -- chunked prefill
    def prefill(self, steps, warmup, tokens=None):
        torch, gdn = self.torch, self.gdn
        shape = synth.WORKLOADS["prefill"]
        if tokens:
            shape = dataclasses.replace(shape, T=int(tokens))
        inp = synth.make_inputs(shape, seed=4)
        d = self.upload(shape, inp)
        dims, prm = self.dims(shape), self.params(d)
        out = torch.empty(shape.B, shape.T, shape.Hv, shape.d, device=self.dev)
        ws_bytes = gdn.prefill_workspace_bytes(dims, shape.T)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.dev)

        def pstep(i):
            gdn.prefill_chunked(d["states"][0], d["hists"][0], d["x"], d["z"], d["alpha"],
                                d["beta_logit"], prm, out, dims, shape.T, 64, workspace=ws)

        try:
            t = self.time_steps(pstep, steps, warmup)
        except gdn.GdnError as e:
            return {"unavailable": str(e)}
        self.launches += 3 * steps           # transform pass, sequential pass, history update
        m = statistics.mean(t)
        toks = shape.B * shape.T
        nb = prefill_work(shape)
        hbm_peak, tc_peak, peak_kind = measured_peaks()
        tflops, gbs = nb["flops"] / m / 1e12, nb["bytes"] / m / 1e9
        return {"ms": m * 1e3, "tokens_per_s": toks / m, "chunk_TFLOPs": tflops,
                "workspace_bytes": ws_bytes,
                "roofline": {"bound": "tensor", "flops_per_launch": nb["flops"],
                             "bytes_per_launch": nb["bytes"], "achieved": tflops, "peak": tc_peak,
                             "unit": "TFLOP/s", "frac": tflops / tc_peak,
                             "hbm_achieved": gbs, "hbm_peak": hbm_peak, "hbm_frac": gbs / hbm_peak,
                             "peak_kind": peak_kind,
                             "note": "whole call (3 launches); per-kernel shares in "
                                     "profiles/prefill_*__prefill_4x8192.md"}}


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_decode_b64_sample(n_seqs: int = 64, n_steps: int = 40, threads: int | None = None,
                             min_seconds: float = 10.0):
    """fp64 oracle on a bounded sample of the headline workload: n_steps
    consecutive decode steps of n_seqs of the 64 sequences (same shapes and
    distributions), parallel over sequences on the host cores."""
    import oracle
    shape = synth.WORKLOADS["decode_b64"]
    inp = synth.make_inputs(shape, seed=2, T=n_steps)
    f = lambda a: synth.bf16_to_f32(np.ascontiguousarray(a))
    x, z = f(inp["x"]), f(np.ascontiguousarray(inp["z"]))
    al, bl = f(inp["alpha"]), f(inp["beta_logit"])
    threads = threads or os.cpu_count() or 1
    seqs = list(range(n_seqs))
    oracle.lib()

    def once():
        t0 = time.perf_counter()
        oracle.layer(x, z, al, bl, inp["conv_w"], inp["dt"], inp["A_log"], inp["norm_w"],
                     inp["state"], inp["hist"], Hq=shape.Hq, W=shape.W, seqs=seqs, threads=threads)
        return time.perf_counter() - t0

    dt = once()
    reps = 1
    while dt < min_seconds and reps < 64:      # repeat the same sample to ~min_seconds of CPU work
        dt += once()
        reps += 1
    state_bytes = decode_bytes(shape)["state"] / shape.B * n_seqs * n_steps * reps
    return {"value": state_bytes / dt / 1e9, "unit": "GB/s", "cores": min(threads, n_seqs),
            "kind": "oracle", "seconds": dt,
            "sample": f"{n_steps} decode steps of {n_seqs} of the 64 sequences (48 V heads, fp64), "
                      f"run {reps}x ({dt:.1f} s)"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    times = []
    res = None
    for i in range(args.warmup + args.steps):
        res = oracle_decode_b64_sample(n_seqs=64, n_steps=2, min_seconds=0.0)
        if i >= args.warmup:
            times.append(res["seconds"])
    shape = synth.WORKLOADS[HEADLINE]
    per_step_bytes = decode_bytes(shape)["state"] * 2
    value = per_step_bytes / statistics.mean(times) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.mean(times) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "batched decode 64 seq x 48 V heads x 128x128 fp32 state, "
                                   "conv_dim 10240, qkvz row stride 20480 (oracle: each step = 2 decode steps "
                                   "of all 64 sequences)"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": res["cores"], "kind": "oracle",
                             "sample": res["sample"]},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-extra", action="store_true", help="headline workload only")
    ap.add_argument("--only", choices=["decode_b1", "decode_b64_bf16_state", "verify_k2",
                                       "verify_kn", "verify_kn8", "conv_tokens", "prefill"],
                    help="run one secondary workload alone and print its figures (for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-tokens", type=int, default=None,
                    help="with --only prefill: tokens per sequence (a smaller case for profiler captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    world, rank, local = dist_env()
    if args.only:
        gpu = Gpu(local)
        fn = {"decode_b1": lambda: gpu.decode_b1(), "verify_k2": lambda: gpu.verify_k2(args.steps, args.warmup),
              "verify_kn": lambda: gpu.verify_kn(args.steps, args.warmup),
              "verify_kn8": lambda: gpu.verify_kn(args.steps, args.warmup, K=8),
              "decode_b64_bf16_state": lambda: gpu.decode_b64_bf16_state(args.steps, args.warmup),
              "conv_tokens": lambda: gpu.conv_tokens(args.steps, args.warmup),
              "prefill": lambda: gpu.prefill(args.steps, args.warmup, args.prefill_tokens)}[args.only]
        print(json.dumps({"workload": args.only, **fn()}), flush=True)
        return 0
    dist = init_dist(world, "nccl")
    gpu = Gpu(local)
    shape = synth.WORKLOADS[HEADLINE]
    with ClockSampler(local) as clocks:
        _, times, e2e_total, h2d, d2h, e2e_serial = gpu.decode_b64(args.steps, args.warmup, dist)
    total_s = sum(times)
    max_s = reduce_max(dist, total_s, gpu.dev)
    nb = decode_bytes(shape)
    mean = max_s / args.steps
    value = aggregate(nb["state"] * args.steps, world, max_s) / 1e9
    e2e_max = reduce_max(dist, e2e_total, gpu.dev)
    e2e_value = aggregate(nb["state"] * args.steps, world, e2e_max) / 1e9
    hbm_peak, _, peak_kind = measured_peaks()
    achieved = nb["total"] / statistics.mean(times) / 1e9
    extra = {}
    if not args.skip_extra:
        extra["decode_b1"] = gpu.decode_b1()
        extra["decode_b64_bf16_state"] = gpu.decode_b64_bf16_state(args.steps, args.warmup)
        extra["verify_k2"] = gpu.verify_k2(max(5, args.steps // 2), args.warmup)
        extra["verify_kn"] = gpu.verify_kn(max(5, args.steps // 2), args.warmup)
        # K = 8: past the fused forms, the token-serial scan with snapshots
        extra["verify_kn8"] = gpu.verify_kn(max(5, args.steps // 4), args.warmup, K=8)
        extra["conv_tokens"] = gpu.conv_tokens(max(5, args.steps // 2), args.warmup)
        extra["prefill"] = gpu.prefill(max(10, args.steps // 2), 3)
    if rank != 0:
        if dist is not None:
            dist.barrier()
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = oracle_decode_b64_sample()
        cpu.pop("seconds")
        # the same oracle on one host thread (a smaller sample: 8 steps of 8 sequences)
        one = oracle_decode_b64_sample(n_seqs=8, n_steps=8, threads=1, min_seconds=2.0)
        cpu["single_thread"] = {"value": one["value"], "unit": one["unit"], "sample": one["sample"]}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "batched decode: 64 seq x 48 V heads (16 QK heads) x 128x128 fp32 "
                               "state, conv_dim 10240, d_conv 4, bf16 activations, qkvz row stride "
                               "20480, one fused launch per step",
                   "global_batch": 64 * world, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: 3 rotating state sets of 192 MiB",
                   "timing": "one pair of CUDA events on the launching stream around the K "
                             "back-to-back steps (each launch a programmatic dependent of the one "
                             "before, as in a serving loop)"},
        "ms_per_launch_serialized": gpu.per_launch_s * 1e3,
        "pct_of_peak": 100.0 * value / world / hbm_peak,
        "pct_of_nominal": 100.0 * value / world / NOMINAL_HBM_GBS,
        "seqs_per_s": shape.B * world / mean,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "traffic": recorded_traffic("decode_fused_kernel"),
                     "kernel": "decode_fused_kernel", "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": nb["total"]},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_max / args.steps * 1e3,
                "copies": "each step's inputs (x, alpha, beta logits packed back to back) from pinned "
                          "host memory in one copy and its output back to pinned host memory, on a "
                          "second stream overlapping the previous step's kernel",
                "serialized_ms_per_step": e2e_serial / args.steps * 1e3},
        "gpu_launches": gpu.launches,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "workloads": extra,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
