#!/usr/bin/env python3
"""Throughput of tree/chain verification + accepted-path commit, per GDN layer.

Metric: draft nodes verified per second per GDN layer = B * N / t_layer, where
t_layer is the device time of one decode step of one layer: the pending
commit of the previous step's accepted path fused into the verification of
the new draft (the delayed state update of the SpecLA review, "Core claim").

Protocol (layer-major decode, inputs larger than L2): R distinct layer
instances, each with its own fp32 state, inputs and ping-pong factor buffers,
R chosen so their footprint is at least 4x the L2 size; one step runs the R
layers back to back, captured once as a CUDA graph and replayed.  Between two
visits of a layer every other layer's data has streamed through L2, so each
visit reads its state from HBM.  Steps are timed with CUDA events on the
launching stream; W untimed warm-up steps come first.

Also reported in the same JSON line:
  roofline      algorithmic bytes of one layer call / measured t_layer, against
                the measured HBM copy bandwidth
  e2e           the same metric through the public API with pinned host inputs
                copied in and outputs copied out inside every timed step
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample
  clocks        SM clocks and throttle reasons sampled while timing

``--impl reference`` times the oracle itself as the reference arm.
Multi-GPU (torchrun): every rank runs its own replica (weak scaling, no
data-path collective); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft nodes verified/sec per GDN layer"
UNIT = "nodes/s"


# ---------------------------------------------------------------------------
# algorithmic traffic of one layer call (bytes that must cross HBM)
# ---------------------------------------------------------------------------
def algorithmic_bytes(B, N, H, dk, dv, esz, L_total, Lmax, chain):
    """Bytes one fused commit+verify layer call must move: L_total = accepted nodes summed over B."""
    state = 2 * B * H * dv * dk * 4                       # read S, write committed S
    inputs = B * N * H * (2 * dk + dv) * esz + 2 * B * N * H * 4 + (0 if chain else B * N * 4)
    outputs = B * N * H * dv * 4                           # o_t
    factors_out = B * H * N * (dv * 4 + dk * esz + 4) + B * N * 4
    commit_in = L_total * H * (dv * 4 + dk * esz + 4) + B * Lmax * 4   # accepted rows of prev factors + path
    return state + inputs + outputs + factors_out + commit_in


# DRAM traffic of one layer call (dram__bytes_read.sum + dram__bytes_write.sum of
# every kernel the call launches) from one ncu capture per workload, with the
# hash of the kernel sources it was taken on: a changed kernel reports null.
NCU_TRAFFIC = {
    "chain8_b1_h8_d256": (2.276e6, ("gdn_chain.cu", "gdn_internal.cuh", "gdn_tc_ptx.cuh"), "4369be9a62c19566"),
    "tree32_depth6_b1_h8_d256": (2.615e6, ("gdn_tree_tc.cu", "gdn_prep_common.cuh", "gdn_tc_ptx.cuh",
                                           "gdn_internal.cuh"), "1ca8894d6f526df8"),
    "tree64_depth8_b16_h8_d256": (47.74e6, ("gdn_tree_tc.cu", "gdn_prep_common.cuh", "gdn_tc_ptx.cuh",
                                            "gdn_internal.cuh"), "1ca8894d6f526df8"),
}


def ncu_traffic(workload):
    import hashlib
    if workload not in NCU_TRAFFIC:
        return None
    nbytes, files, digest = NCU_TRAFFIC[workload]
    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "speculative_decoding_linear_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return nbytes if m.hexdigest()[:16] == digest else None


def max_over_ranks(x, dist, world, device="cpu"):
    """The largest value of x over all ranks (x itself on one rank): step times are the max over ranks."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, seconds):
    """Units processed by all ranks per second of the slowest rank (weak scaling: every rank runs
    its own replica of the workload)."""
    return units_per_rank * world / seconds


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", "clocks_bench_%d.csv" % os.getpid())

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())}


# ---------------------------------------------------------------------------
# the workload: R layer instances on one GPU
# ---------------------------------------------------------------------------
class Layer:
    """One GDN layer instance: its state, this step's draft inputs, ping-pong factors."""

    def __init__(self, w, device, torch, gdnspec):
        def qkv(x):
            if x.dtype == np.uint16:
                return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).to(device)
            return torch.from_numpy(x.copy()).to(device)
        self.w = w
        self.q, self.k, self.v = qkv(w.q), qkv(w.k), qkv(w.v)
        self.alpha = torch.from_numpy(w.alpha).to(device)
        self.beta = torch.from_numpy(w.beta).to(device)
        self.parent = torch.from_numpy(w.parent).to(device)
        self.path = torch.from_numpy(w.path).to(device)
        self.S = torch.from_numpy(w.S0).to(device)
        self.out = torch.empty((w.B, w.N, w.H, w.dv), dtype=torch.float32, device=device)
        self.fac = [gdnspec.empty_factors(w.B, w.N, w.H, w.dk, w.dv, w.dtype, device) for _ in range(2)]
        self.ws = gdnspec.empty_workspace(w.B, w.N, w.H, w.dk, w.dv, device)

    def nbytes(self):
        ts = [self.q, self.k, self.v, self.alpha, self.beta, self.parent, self.path, self.S, self.out,
              self.ws] + self.fac
        return sum(t.numel() * t.element_size() for t in ts)


def make_layers(cfg, R, seed0, device, torch, gdnspec, wl, batch=None):
    return [Layer(wl.make_workload(cfg, seed=seed0 + 7919 * r, B=batch), device, torch, gdnspec)
            for r in range(R)]


def layer_call(gdnspec, ly, parity, chain):
    """One decode step of one layer: commit the previous accepted path inside the new verify."""
    prev, nxt = ly.fac[parity], ly.fac[1 - parity]
    w = ly.w
    if chain:
        gdnspec.gdn_commit_chain_verify(ly.S, prev, w.N, ly.path, ly.q, ly.k, ly.v, ly.alpha, ly.beta,
                                        ly.out, nxt)
    else:
        gdnspec.gdn_commit_tree_verify(ly.S, prev, w.N, ly.path, ly.q, ly.k, ly.v, ly.alpha, ly.beta,
                                       ly.parent, ly.out, nxt, ly.ws)


def first_verify(gdnspec, ly, chain):
    w = ly.w
    if chain:
        gdnspec.gdn_chain_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.S, ly.out, ly.fac[0])
    else:
        gdnspec.gdn_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out, ly.fac[0],
                                ly.ws)


def run_gpu(cfg, steps, warmup, rank, world, device_index, torch, dist, profile=False, batch=None, layers=None):
    from speculative_decoding_linear_gb300 import gdnspec
    from speculative_decoding_linear_gb300 import workloads as wl

    torch.cuda.set_device(device_index)
    device = torch.device("cuda", device_index)
    spec = wl.SPECS[cfg]
    chain = spec.tree == "chain"
    props = torch.cuda.get_device_properties(device_index)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 2 ** 20

    probe = Layer(wl.make_workload(cfg, B=batch), device, torch, gdnspec)
    per_layer = probe.nbytes()
    del probe
    R = max(2, -(-4 * l2 // per_layer)) if layers is None else max(2, layers)
    layers = make_layers(cfg, R, 1000 * (rank + 1) + cfg, device, torch, gdnspec, wl, batch)
    footprint = sum(ly.nbytes() for ly in layers)

    stream = torch.cuda.Stream(device=device)
    # consecutive calls of the sweep touch different layers: launch overlap is safe
    gdnspec.gdn_set_launch_overlap(True)
    with torch.cuda.stream(stream):
        for ly in layers:
            first_verify(gdnspec, ly, chain)
        assert gdnspec.gdn_last_error(stream) == 0
        for parity in (0, 1):                    # eager warm-up of both parities before capture
            for ly in layers:
                layer_call(gdnspec, ly, parity, chain)
        assert gdnspec.gdn_last_error(stream) == 0
        graphs = []
        for parity in (0, 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for ly in layers:
                    layer_call(gdnspec, ly, parity, chain)
            graphs.append(g)
        for i in range(max(warmup, 3)):
            graphs[i % 2].replay()
        stream.synchronize()
        assert gdnspec.gdn_last_error(stream) == 0

        # soak ~1 s so the clock sampler sees the GPU under this load, then time exactly K steps
        sampler = ClockSampler(device_index)
        sampler.start()
        t_soak = time.time()
        i = 0
        while not profile and time.time() - t_soak < 1.0:
            graphs[i % 2].replay()
            i += 1
            if i % 16 == 0:
                stream.synchronize()
        stream.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(steps):
            graphs[s % 2].replay()
        e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        clocks = sampler.stop()
        ms_local = e0.elapsed_time(e1)
        assert gdnspec.gdn_last_error(stream) == 0

    ms = max_over_ranks(ms_local, dist, world, device)

    # ---- end to end through the public API: pinned host inputs in, outputs out, every step
    e2e = None if profile else run_e2e(layers, steps, chain, gdnspec, torch, stream, world, dist, device)
    baselines = None if (profile or chain) else run_replay_baselines(layers, gdnspec, torch, stream,
                                                                     max(5, min(steps, 20)))
    hybrid = None if (profile or chain) else run_hybrid_comparison(layers, gdnspec, torch, stream,
                                                                   max(5, min(steps, 20)), device, wl)
    prune = None if (profile or chain) else run_prune_timing(gdnspec, torch, stream, device, wl, B=layers[0].w.B,
                                                             N=layers[0].w.N)

    w0 = layers[0].w
    B, N, H, dk, dv = w0.B, w0.N, w0.H, w0.dk, w0.dv
    esz = 2 if w0.dtype == wl.BF16 else 4
    per_call = float(np.mean([algorithmic_bytes(B, N, H, dk, dv, esz, int(np.sum(ly.w.path >= 0)),
                                                ly.w.path.shape[1], chain) for ly in layers]))
    t_layer_s = ms / 1e3 / (steps * R)
    peak, peak_kind = measured_peaks()
    achieved = per_call / t_layer_s / 1e9
    value = whole_job_rate(B * N * R * steps, world, ms / 1e3)
    # one launch per call: the chain kernel, or the single-kernel tree verifier (d_k = d_v = 256)
    fused_tree = not chain and dk == 256 and dv == 256
    launches_per_call = 1 if (chain or fused_tree) else 2
    return dict(
        value=value, ms=ms / steps, R=R, footprint=footprint, l2=l2, clocks=clocks, e2e=e2e,
        spec=spec, B=B, N=N, H=H, dk=dk, dv=dv, chain=chain,
        roofline={"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                  "frac": round(achieved / peak, 4), "traffic": ncu_traffic(spec.name),
                  "peak_kind": peak_kind + " hbm_gbs (copy)",
                  "kernel": "gdn_commit_chain_verify (chain_g8_kernel)" if chain else
                            "gdn_commit_tree_verify (tree_fused_tc_kernel)" if fused_tree else
                            "gdn_commit_tree_verify (prologue + contraction kernels)",
                  "algorithmic_bytes_per_call": per_call, "t_call_us": round(t_layer_s * 1e6, 3)},
        gpu_launches=launches_per_call * R * steps, baselines=baselines, hybrid=hybrid, prune=prune,
    )


# ---------------------------------------------------------------------------
# replay baselines: what tree verification and the factor-buffer commit replace
# ---------------------------------------------------------------------------
def run_replay_baselines(layers, gdnspec, torch, stream, steps):
    """Per-call device time of tree verification vs replaying every root-to-leaf path, and of the
    factor-buffer commit vs replaying the accepted tokens, on the same layer rotation (no launch
    overlap for either side).  Commits write to a scratch state so the inputs stay unchanged."""
    prev = gdnspec.gdn_set_launch_overlap(False)
    scratch = [torch.empty_like(ly.S) for ly in layers]
    w0 = layers[0].w

    def variant(name):
        def call(ly, sc):
            w = ly.w
            if name == "tree_verify":
                gdnspec.gdn_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out, ly.fac[0], ly.ws)
            elif name == "replay_verify":
                gdnspec.gdn_replay_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out)
            elif name == "factor_commit":
                gdnspec.gdn_commit(ly.S, ly.fac[0], ly.path, sc, w.N, w.dtype)
            else:
                gdnspec.gdn_replay_commit(ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.path, sc)
        with torch.cuda.stream(stream):
            for ly, sc in zip(layers, scratch):
                call(ly, sc)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for ly, sc in zip(layers, scratch):
                    call(ly, sc)
            for _ in range(3):
                g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
        assert gdnspec.gdn_last_error(stream) == 0
        return e0.elapsed_time(e1) * 1e3 / (steps * len(layers))

    with torch.cuda.stream(stream):
        for ly in layers:                 # the factor record the commits read
            gdnspec.gdn_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out, ly.fac[0], ly.ws)
    us = {n: variant(n) for n in ("tree_verify", "replay_verify", "factor_commit", "replay_commit")}
    gdnspec.gdn_set_launch_overlap(prev)
    del scratch
    return {"us_per_call": {k: round(v, 3) for k, v in us.items()},
            "replay_verify_over_tree_verify": round(us["replay_verify"] / us["tree_verify"], 2),
            "replay_commit_over_factor_commit": round(us["replay_commit"] / us["factor_commit"], 2),
            "what": "per layer call, %s, same rotation of %d layers; replay = every root-to-leaf path "
                    "(verify) or the accepted tokens (commit) run token by token from S0"
                    % (w0.spec.name, len(layers))}


# ---------------------------------------------------------------------------
# chain-decomposed (hybrid) verification vs the tree verifier
# ---------------------------------------------------------------------------
def time_calls(calls, torch, stream, steps):
    """Device time per call of a list of zero-argument launches, replayed as one CUDA graph."""
    with torch.cuda.stream(stream):
        for c in calls:
            c()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c()
        for _ in range(3):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (steps * len(calls))


def run_hybrid_comparison(layers, gdnspec, torch, stream, steps, device, wl):
    """Tree verifier vs chain-decomposed verification on the bench's trees and on deep, narrow trees of
    the same size (a trunk of 8 nodes and 4 chains below it), launch overlap off for both."""
    prev = gdnspec.gdn_set_launch_overlap(False)
    w0 = layers[0].w
    res = {}
    narrow = [Layer(wl.custom_workload(w0.B, w0.N, w0.H, w0.dk, w0.dv, wl.narrow_tree(w0.N, 4, 8), seed=9000 + r),
                    device, torch, gdnspec) for r in range(len(layers))]
    for name, lys in (("bench_trees", layers), ("narrow_trees", narrow)):
        tree = [lambda ly=ly: gdnspec.gdn_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out,
                                                      ly.fac[0], ly.ws) for ly in lys]
        hyb = [lambda ly=ly: gdnspec.gdn_hybrid_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S,
                                                            ly.out, ly.fac[0]) for ly in lys]
        t_tree = time_calls(tree, torch, stream, steps)
        t_hyb = time_calls(hyb, torch, stream, steps)
        rc = gdnspec.gdn_last_error(stream)
        res[name] = {"tree_verify_us": round(t_tree, 3),
                     "hybrid_verify_us": round(t_hyb, 3) if rc == 0 else None,
                     "hybrid_status": gdnspec.strerror(rc) if rc else "ok"}
    gdnspec.gdn_set_launch_overlap(prev)
    res["what"] = ("per call, %d sequences x %d nodes; narrow_trees = a trunk of 8 nodes and 4 chains of %d "
                   "hanging from it" % (w0.B, w0.N, (w0.N - 8) // 4))
    return res


# ---------------------------------------------------------------------------
# full GDN layer decode step: projections, ancestor-window conv, gates, tree
# verification with the pending commit fused in, output gate, o_proj
# ---------------------------------------------------------------------------
def layer_flops(B, N, H, hidden, dk, dv):
    """Dense tensor-core work of one layer call: input and output projections (useful flops)."""
    rows = 2 * H * dk + 2 * H * dv + 2 * H
    return 2.0 * B * N * hidden * rows + 2.0 * B * N * H * dv * hidden


class LayerStep:
    """One full-layer instance: weights, state, conv history, this step's draft, ping-pong records."""

    def __init__(self, w, device, torch, gdnspec):
        def bf(bits):
            return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(device)

        def f(x):
            return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)
        self.w = w
        self.X, self.W_in, self.W_o, self.conv_w = bf(w.X), bf(w.W_in), bf(w.W_o), f(w.conv_w)
        self.parent = torch.from_numpy(w.parent).to(device)
        self.path = torch.from_numpy(w.path).to(device)
        self.S, self.conv_state = f(w.S0), f(w.conv_state)
        nb = gdnspec.gdn_layer_record_bytes(w.B, w.N, w.H, w.hidden, w.dk, w.dv)
        self.rec = [torch.empty(nb, dtype=torch.uint8, device=device) for _ in range(2)]
        self.ws = torch.empty(gdnspec.gdn_layer_workspace_bytes(w.B, w.N, w.H, w.hidden, w.dk, w.dv),
                              dtype=torch.uint8, device=device)
        self.out = torch.empty((w.B, w.N, w.hidden), dtype=torch.float32, device=device)

    def nbytes(self):
        ts = [self.X, self.W_in, self.W_o, self.conv_w, self.parent, self.path, self.S, self.conv_state,
              self.ws, self.out] + self.rec
        return sum(t.numel() * t.element_size() for t in ts)

    def call(self, gdnspec, parity, first=False):
        w = self.w
        if first:
            gdnspec.gdn_layer_tree_step(self.X, self.W_in, self.conv_w, self.W_o, self.parent, self.S,
                                        self.conv_state, None, 0, None, self.out, self.rec[0], self.ws,
                                        w.H, w.dk, w.dv)
        else:
            gdnspec.gdn_layer_tree_step(self.X, self.W_in, self.conv_w, self.W_o, self.parent, self.S,
                                        self.conv_state, self.rec[parity], w.N, self.path, self.out,
                                        self.rec[1 - parity], self.ws, w.H, w.dk, w.dv)


def run_gpu_layer(steps, warmup, rank, world, device_index, torch, dist, profile=False, layers=None):
    from speculative_decoding_linear_gb300 import gdnspec
    from speculative_decoding_linear_gb300 import workloads as wl

    torch.cuda.set_device(device_index)
    device = torch.device("cuda", device_index)
    spec = wl.SPECS[4]
    props = torch.cuda.get_device_properties(device_index)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 2 ** 20
    first = LayerStep(wl.make_layer_workload(4, seed=1000 * (rank + 1) + 4), device, torch, gdnspec)
    per_layer = first.nbytes()
    R = max(2, -(-4 * l2 // per_layer)) if layers is None else max(2, layers)
    lys = [first] + [LayerStep(wl.make_layer_workload(4, seed=1000 * (rank + 1) + 4 + 7919 * r), device, torch,
                               gdnspec) for r in range(1, R)]
    footprint = sum(ly.nbytes() for ly in lys)
    stream = torch.cuda.Stream(device=device)
    with torch.cuda.stream(stream):
        for ly in lys:
            ly.call(gdnspec, 0, first=True)
        assert gdnspec.gdn_last_error(stream) == 0
        for parity in (0, 1):
            for ly in lys:
                ly.call(gdnspec, parity)
        assert gdnspec.gdn_last_error(stream) == 0
        graphs = []
        for parity in (0, 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for ly in lys:
                    ly.call(gdnspec, parity)
            graphs.append(g)
        for i in range(max(warmup, 3)):
            graphs[i % 2].replay()
        stream.synchronize()
        assert gdnspec.gdn_last_error(stream) == 0
        sampler = ClockSampler(device_index)
        sampler.start()
        t_soak = time.time()
        i = 0
        while not profile and time.time() - t_soak < 1.0:
            graphs[i % 2].replay()
            i += 1
            if i % 4 == 0:
                stream.synchronize()
        stream.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s_ in range(steps):
            graphs[s_ % 2].replay()
        e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        clocks = sampler.stop()
        ms_local = e0.elapsed_time(e1)
        assert gdnspec.gdn_last_error(stream) == 0

        seq = None if profile else run_sequential_baseline(lys[0], gdnspec, torch, stream, steps=3)
        model = None if profile else run_model_step(gdnspec, torch, stream, device, wl)
    ms = max_over_ranks(ms_local, dist, world, device)

    e2e = None if profile else run_e2e_layer(lys, steps, gdnspec, torch, stream, world, dist, device)
    w0 = lys[0].w
    t_layer_s = ms / 1e3 / (steps * R)
    flops = layer_flops(w0.B, w0.N, w0.H, w0.hidden, w0.dk, w0.dv)
    peak, peak_kind = measured_tensor_peak()
    achieved = flops / t_layer_s / 1e12
    return dict(
        value=whole_job_rate(w0.B * w0.N * R * steps, world, ms / 1e3), ms=ms / steps, R=R, footprint=footprint, l2=l2, clocks=clocks, e2e=e2e,
        spec=spec, B=w0.B, N=w0.N, H=w0.H, dk=w0.dk, dv=w0.dv, hidden=w0.hidden, chain=False, layer=True,
        sequential=seq, model=model,
        roofline={"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                  "frac": round(achieved / peak, 4), "traffic": None, "peak_kind": peak_kind,
                  "kernel": "gdn_layer_tree_step (input/output projection GEMMs on tcgen05, conv, "
                            "tree verify + commit, gate)",
                  "algorithmic_flops_per_call": flops, "t_call_us": round(t_layer_s * 1e6, 3)},
        # GEMM, conv, tree verifier (one kernel at d_k = d_v = 256, else two), gate, GEMM
        gpu_launches=(5 if w0.dk == 256 and w0.dv == 256 else 6) * R * steps,
    )


def run_model_step(gdnspec, torch, stream, device, wl, n_layers=4, steps=5):
    """n_layers full layers back to back on a residual stream (h_{l+1} = h_l + out_l), each step committing
    the previous step's accepted path in every layer: time per model step as one CUDA graph per parity."""
    lys = [LayerStep(wl.make_layer_workload(4, seed=5000 + 11 * l), device, torch, gdnspec) for l in range(n_layers)]
    w = lys[0].w
    ws = torch.empty(gdnspec.gdn_model_workspace_bytes(n_layers, w.B, w.N, w.H, w.hidden, w.dk, w.dv),
                     dtype=torch.uint8, device=device)
    out = torch.empty((w.B, w.N, w.hidden), dtype=torch.float32, device=device)
    per = dict(W_in=[ly.W_in for ly in lys], conv_w=[ly.conv_w for ly in lys], W_o=[ly.W_o for ly in lys],
               S=[ly.S for ly in lys], conv_state=[ly.conv_state for ly in lys])

    def step(parity, first=False):
        gdnspec.gdn_model_tree_step(lys[0].X, per["W_in"], per["conv_w"], per["W_o"], lys[0].parent, per["S"],
                                    per["conv_state"], None if first else [ly.rec[parity] for ly in lys], w.N,
                                    None if first else lys[0].path, out, [ly.rec[1 - parity] for ly in lys], ws,
                                    w.H, w.dk, w.dv)
    with torch.cuda.stream(stream):
        step(1, first=True)                    # writes rec[0]
        step(0)
        step(1)
        graphs = []
        for parity in (0, 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(parity)
            graphs.append(g)
        for i in range(3):
            graphs[i % 2].replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            graphs[i % 2].replay()
        e1.record(stream)
        e1.synchronize()
    assert gdnspec.gdn_last_error(stream) == 0
    ms = e0.elapsed_time(e1) / steps
    del lys, ws
    torch.cuda.empty_cache()
    return {"layers": n_layers, "ms_per_model_step": round(ms, 4), "us_per_layer": round(1e3 * ms / n_layers, 2),
            "nodes_per_s_per_layer": round(w.B * w.N * n_layers / (ms / 1e3), 1),
            "what": "gdn_model_tree_step: %d layers back to back on a residual stream h_(l+1) = h_l + out_l, "
                    "every layer committing the previous step's accepted path" % n_layers}


def run_prune_timing(gdnspec, torch, stream, device, wl, B, N, steps=50):
    """Device time of one gdn_prune_tree call on B random trees of N nodes."""
    rng = np.random.default_rng(77)
    parent = torch.from_numpy(np.stack([wl.random_tree(rng, N, 8) for _ in range(B)])).to(device)
    logp = torch.from_numpy((-rng.exponential(1.0, (B, N))).astype(np.float32)).to(device)
    idx = torch.empty((B, N), dtype=torch.int32, device=device)
    npar = torch.empty((B, N), dtype=torch.int32, device=device)
    nk = torch.empty(B, dtype=torch.int32, device=device)
    us = time_calls([lambda: gdnspec.gdn_prune_tree(parent, logp, 1.0, N // 2, idx, npar, nk)], torch, stream, steps)
    assert gdnspec.gdn_last_error(stream) == 0
    return {"us_per_call": round(us, 3), "B": B, "N": N, "tau": 1.0, "budget": N // 2}


def measured_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops_sustained"]), "measured bf16_tflops_sustained (cuBLAS, long loop)"
    return 1700.0, "fallback"


def pack_tensors(objs, names, torch, device):
    """Move the named tensors of every object into one device buffer (each view 256-byte aligned) and
    re-point the objects at the views; returns (device buffer, pinned host buffer with the same bytes)."""
    ts = [getattr(o, n) for o in objs for n in names]
    offs, total = [], 0
    for t in ts:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    buf = torch.empty(total, dtype=torch.uint8, device=device)
    i = 0
    for o in objs:
        for n in names:
            t = ts[i]
            v = buf[offs[i]: offs[i] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            v.copy_(t)
            setattr(o, n, v)
            i += 1
    return buf, buf.cpu().pin_memory()


def run_e2e_layer(lys, steps, gdnspec, torch, stream, world, dist, device):
    """Layer step through the public API with every instance's X, parent_idx and accepted path copied
    in from pinned host memory (one transfer) and the layer outputs copied out (one transfer), every
    step."""
    dev_in, host_in = pack_tensors(lys, ["X", "parent", "path"], torch, device)
    dev_out, host_out = pack_tensors(lys, ["out"], torch, device)
    h2d = host_in.numel()
    d2h = host_out.numel()
    k = max(1, min(steps, 5))
    with torch.cuda.stream(stream):
        def one(parity):
            dev_in.copy_(host_in, non_blocking=True)
            for ly in lys:
                ly.call(gdnspec, parity)
            host_out.copy_(dev_out, non_blocking=True)
        one(0)
        one(1)
        stream.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for s_ in range(k):
            one(s_ % 2)
        stream.synchronize()
        t1 = time.perf_counter()
    sec = max_over_ranks(t1 - t0, dist, world, device)
    w = lys[0].w
    return {"value": whole_job_rate(w.B * w.N * len(lys) * k, world, sec), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": k, "ms_per_step": 1e3 * sec / k}


def run_sequential_baseline(ly, gdnspec, torch, stream, steps=3):
    """The same layer decoded node by node (gdn_layer_token_step for t = 0 .. N-1), each node from its
    parent's materialised state: the per-token decoder the tree step replaces.  One pass over the N
    nodes is captured as a CUDA graph and replayed; returns nodes/s and ms per layer step."""
    w = ly.w
    dev = ly.S.device
    S_nodes = torch.empty((w.N, w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    rec = torch.empty(gdnspec.gdn_layer_record_bytes(w.B, w.N, w.H, w.hidden, w.dk, w.dv), dtype=torch.uint8,
                      device=dev)
    ws = torch.empty(gdnspec.gdn_layer_workspace_bytes(w.B, w.N, w.H, w.hidden, w.dk, w.dv), dtype=torch.uint8,
                     device=dev)
    out = torch.empty_like(ly.out)

    def one_pass():
        for t in range(w.N):
            gdnspec.gdn_layer_token_step(ly.X, ly.W_in, ly.conv_w, ly.W_o, ly.parent, ly.S, ly.conv_state, S_nodes,
                                         t, out, rec, ws, w.H, w.dk, w.dv)
    one_pass()
    assert gdnspec.gdn_last_error(stream) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        one_pass()
    g.replay()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.replay()
    e1.record(stream)
    e1.synchronize()
    assert gdnspec.gdn_last_error(stream) == 0
    ms = e0.elapsed_time(e1) / steps
    res = {"value": w.B * w.N / (ms / 1e3), "unit": UNIT, "ms_per_layer_step": round(ms, 4), "passes": steps,
           "gpu_launches_per_layer_step": 5 * w.N, "node_state_bytes": S_nodes.numel() * 4,
           "what": "gdn_layer_token_step for t = 0..N-1: per-node projection, conv, one delta-rule step "
                   "from the parent's materialised state, gate, o_proj"}
    del S_nodes, rec, ws, out
    torch.cuda.empty_cache()
    return res


def run_e2e(layers, steps, chain, gdnspec, torch, stream, world, dist, device):
    """Same metric through the public API: every layer call made from the host each step, with all
    layers' draft inputs copied in from pinned host memory (one transfer) and their outputs copied
    out (one transfer) inside the timed region."""
    names = ["q", "k", "v", "alpha", "beta", "path"] + ([] if chain else ["parent"])
    dev_in, host_in = pack_tensors(layers, names, torch, device)
    dev_out, host_out = pack_tensors(layers, ["out"], torch, device)
    h2d = host_in.numel()
    d2h = host_out.numel()
    k = max(1, min(steps, 10))
    with torch.cuda.stream(stream):
        def one(parity):
            dev_in.copy_(host_in, non_blocking=True)
            for ly in layers:
                layer_call(gdnspec, ly, parity, chain)
            host_out.copy_(dev_out, non_blocking=True)
        one(0)
        one(1)
        stream.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for s in range(k):
            one(s % 2)
        stream.synchronize()
        t1 = time.perf_counter()
    sec = max_over_ranks(t1 - t0, dist, world, device)
    w = layers[0].w
    return {"value": whole_job_rate(w.B * w.N * len(layers) * k, world, sec), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k, "ms_per_step": 1e3 * sec / k}


# ---------------------------------------------------------------------------
# oracle on the host cores
# ---------------------------------------------------------------------------
def oracle_layer_seconds(w, nthreads):
    """Verify every node of one layer instance and commit its accepted path with the fp64 oracle."""
    import oracle
    x = dict(q=w.widened("q"), k=w.widened("k"), v=w.widened("v"), alpha=w.alpha.astype(np.float64),
             beta=w.beta.astype(np.float64), parent=w.parent, S0=w.S0.astype(np.float64))
    t0 = time.perf_counter()
    oracle.tree_verify(**x, nthreads=nthreads)
    oracle.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path, nthreads=nthreads)
    return time.perf_counter() - t0


def oracle_full_layer_seconds(w, nthreads):
    """One full-layer decode step of a layer workload with the fp64 layer oracle, plus its commit."""
    from oracle import layer
    X, W_in, cw, cs, W_o, S0 = (w.widened(n) for n in ("X", "W_in", "conv_w", "conv_state", "W_o", "S0"))
    t0 = time.perf_counter()
    r = layer.layer_step(X, W_in, cw, cs, W_o, w.parent, S0, w.H, w.dk, w.dv, nthreads=nthreads)
    layer.layer_commit(r, w.parent, S0, cs, w.path, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(cfg, budget_s=10.0):
    import oracle
    from speculative_decoding_linear_gb300 import workloads as wl
    oracle.build()
    cores = os.cpu_count() or 1
    if cfg == 4:
        w = wl.make_layer_workload(4, B=2)
        n, sec = 0, 0.0
        while sec < budget_s:
            sec += oracle_full_layer_seconds(w, cores)
            n += 1
        return {"value": w.B * w.N * n / sec, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": "%d repetitions of one full-layer step of 2 of the 64 sequences of %s (numpy "
                          "fp64 projections/conv/o_proj + path-walk recurrence + commit), %d threads"
                          % (n, w.spec.name, cores)}
    w = wl.make_workload(cfg)
    n, sec = 0, 0.0
    while sec < budget_s:
        sec += oracle_layer_seconds(w, cores)
        n += 1
    return {"value": w.B * w.N * n / sec, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d repetitions of one layer instance of %s (verify all %d nodes x %d heads "
                      "by path walks + commit), fp64, %d threads" % (n, w.spec.name, w.B * w.N, w.H, cores)}


def run_reference(args):
    """Reference arm: the oracle as it stands, timed on the host cores (rank 0 only)."""
    from speculative_decoding_linear_gb300 import workloads as wl
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle.build()
    cores = os.cpu_count() or 1
    if args.config == 4:
        w = wl.make_layer_workload(4, B=2)
        timer = oracle_full_layer_seconds
    else:
        w = wl.make_workload(args.config)
        timer = oracle_layer_seconds
    for _ in range(max(args.warmup, 1)):
        timer(w, cores)
    sec = sum(timer(w, cores) for _ in range(args.steps))
    value = w.B * w.N * args.steps / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.spec.name, "B": w.spec.B, "N": w.N, "H": w.H, "dk": w.dk, "dv": w.dv},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "one layer instance of %s per step (verify all nodes by path "
                                       "walks + commit), fp64, %d threads" % (w.spec.name, cores)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=1, choices=[1, 2, 3, 4])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch size")
    ap.add_argument("--profile", action="store_true",
                    help="for profiler runs: no clock soak, no e2e leg, no CPU baseline")
    ap.add_argument("--layers", type=int, default=None,
                    help="for profiler runs: rotate this many layers instead of >= 4x L2 of them")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    if args.config == 4:
        r = run_gpu_layer(args.steps, args.warmup, rank, world, local, torch, dist, args.profile, args.layers)
    else:
        r = run_gpu(args.config, args.steps, args.warmup, rank, world, local, torch, dist, args.profile,
                    args.batch, args.layers)

    if rank == 0:
        cpu = None if args.no_cpu_baseline or args.profile or world > 1 else cpu_baseline(args.config)
        spec = r["spec"]
        line = {
            "metric": METRIC, "value": round(r["value"], 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms"], 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": spec.name, "B": r["B"], "N": r["N"], "H": r["H"], "dk": r["dk"],
                       "dv": r["dv"], "qkv": spec.dtype, "state": "f32",
                       "step": ("full GDN layer step: projections, ancestor-window conv, gates, tree "
                                "verify with the pending commit (state + conv history) fused in, output "
                                "gate, o_proj") if r.get("layer") else
                               "per layer: pending commit fused into the next %s verify"
                               % ("chain" if r["chain"] else "tree"),
                       "layers_rotated": r["R"], "footprint_bytes": r["footprint"], "l2_bytes": r["l2"],
                       "l2_policy": ("inputs larger than L2: %d-layer rotation, footprint >= 4x L2" % r["R"])
                       if r["footprint"] >= 4 * r["l2"] else
                       "profiling rotation of %d layers (footprint below 4x L2)" % r["R"],
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r["e2e"],
            "gpu_launches": r["gpu_launches"], "clocks": r["clocks"],
        }
        if r.get("baselines"):
            line["replay_baselines"] = r["baselines"]
        if r.get("hybrid"):
            line["hybrid_verify"] = r["hybrid"]
        if r.get("prune"):
            line["prune_tree"] = r["prune"]
        if r.get("model"):
            line["model_step"] = r["model"]
        if r.get("layer"):
            line["config"]["hidden"] = r["hidden"]
            seq = r["sequential"]
            if seq:
                seq["tree_step_speedup"] = round(r["value"] / seq["value"], 2)
            line["sequential_decode"] = seq
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
