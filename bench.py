#!/usr/bin/env python3
"""Throughput of tree verification + accepted-path commit, per GDN layer.

Metric: draft nodes verified per second per GDN layer = B * N / t_layer, where
t_layer is the device time of one decode step of one layer.  The default
workload is the full GDN layer step over 64 draft trees of 64 nodes (hidden
2048, 8 heads of d_k = d_v = 256): input projection, ancestor-window conv,
gates, tree verification with the previous accepted path's commit fused in
(the delayed state update of the SpecLA review, "Core claim"), output gate and
output projection.  The same line carries a sub-record for 16 trees of 64
nodes through gdn_commit_tree_verify alone (the verifier + commit kernel).

Protocol (layer-major decode, inputs larger than L2): R distinct layer
instances, each with its own state, inputs and ping-pong records, R chosen so
their footprint is at least 4x the L2 size; one step runs the R layers back
to back, captured once as a CUDA graph and replayed.  Between two visits of a
layer every other layer's data has streamed through L2, so each visit reads
its state from HBM.  W untimed warm-up steps, then exactly K timed steps
bracketed by a barrier and a device synchronize, timed with CUDA events on
the launching stream (max over ranks).

Also reported in the same JSON line:
  roofline      the dominant kernel's algorithmic bytes (or flops) per launch /
                its CUDA-event time, against the measured peak; per_kernel
                lists every kernel of the step the same way
  replays       median / p10 / p90 per layer call over >= 100 graph replays,
                the cold single-call latency (L2 flushed) and the L2-warm figure
  e2e           the same metric through the public API with pinned host inputs
                copied in and outputs copied out inside every timed step
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample
  clocks        SM clocks and throttle reasons sampled while timing

``--impl reference`` times the oracle itself as the reference arm.
Multi-GPU: ``--gpus N`` launches N ranks (one per GPU) through torchrun when
not already under it.  ``--shard replicas`` (default): every rank runs its own
replica (weak scaling).  ``--shard sequences``: the batch's sequences are split
across ranks (strong scaling).  Neither needs a collective on the data path;
the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import socket
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft nodes verified/sec per GDN layer"
UNIT = "nodes/s"
LAYER_KERNELS = ("gemm_in", "conv", "tree_verify", "gate", "gemm_out")
LAYER_KERNEL_NAMES = {
    "gemm_in": "gemm_bf16_kernel<1,256> (input projection)",
    "conv": "layer_conv_kernel (ancestor-window conv, norms, gates)",
    "tree_verify": "tree_fused_tc_kernel<1,2> (+ <1,1> for the pairs past whole waves; tree verify + pending commit)",
    "gate": "layer_gate_kernel (o * SiLU(z))",
    "gemm_out": "gemm_bf16_kernel<2,256> (output projection, two bf16 terms)",
}


# ---------------------------------------------------------------------------
# algorithmic work of one call (bytes that must cross HBM, or tensor flops)
# ---------------------------------------------------------------------------
def algorithmic_bytes(B, N, H, dk, dv, esz, L_total, Lmax, chain):
    """Bytes one fused commit+verify layer call must move: L_total = accepted nodes summed over B."""
    state = 2 * B * H * dv * dk * 4                       # read S, write committed S
    inputs = B * N * H * (2 * dk + dv) * esz + 2 * B * N * H * 4 + (0 if chain else B * N * 4)
    outputs = B * N * H * dv * 4                           # o_t
    factors_out = B * H * N * (dv * 4 + dk * esz + 4) + B * N * 4
    commit_in = L_total * H * (dv * 4 + dk * esz + 4) + B * Lmax * 4   # accepted rows of prev factors + path
    return state + inputs + outputs + factors_out + commit_in


def layer_flops(B, N, H, hidden, dk, dv):
    """Dense tensor-core work of one layer call: input and output projections (useful flops)."""
    rows = 2 * H * dk + 2 * H * dv + 2 * H
    return 2.0 * B * N * hidden * rows + 2.0 * B * N * H * dv * hidden


def layer_kernel_work(B, N, H, hidden, dk, dv, L_total, Lmax):
    """Per kernel of one layer step: (bound, algorithmic amount, unit).  HBM kernels count the bytes
    their function needs to move (inputs read once, outputs written once); the GEMMs count useful
    flops (the output GEMM issues twice as many: two bf16 terms of its fp32 left operand)."""
    M = B * N
    C = H * (2 * dk + dv)
    conv = (M * C * 4                                  # read the pre-conv q|k|v projections
            + 2 * B * 3 * C * 4                        # conv history: read, write the committed rows
            + min(L_total, 3 * B) * C * 4              # accepted rows entering the history
            + M * 2 * H * 4                            # gate pre-activations
            + M * H * (dk + dv) * 4                    # k, v (fp32) for the verifier
            + 4 * M * H * dk * 2                       # bf16 hi/lo terms of q and k
            + 2 * M * H * 4)                           # alpha, beta
    verify = (2 * B * H * dv * dk * 4                  # state read + committed state written
              + 4 * M * H * dk * 2 + M * H * (dk + dv) * 4 + 2 * M * H * 4 + M * 4   # q/k terms, k, v, gates, parents
              + M * H * dv * 4                         # o
              + B * H * N * (dv * 4 + dk * 4 + 4) + M * 4   # factor record (fp32 keys)
              + L_total * H * (dv * 4 + dk * 4 + 4) + B * Lmax * 4)   # pending commit's rows + path
    gate = M * H * dv * 4 * 2 + 2 * M * H * dv * 2     # read o, z; write y hi, lo
    rows = 2 * H * dk + 2 * H * dv + 2 * H
    return {"gemm_in": ("tensor", 2.0 * M * hidden * rows, "flop"),
            "conv": ("hbm", float(conv), "B"),
            "tree_verify": ("hbm", float(verify), "B"),
            "gate": ("hbm", float(gate), "B"),
            "gemm_out": ("tensor", 2.0 * M * H * dv * hidden, "flop")}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a kernel from one ncu
# capture, keyed by (workload, kernel), with the hash of the kernel sources it was taken on: a changed
# kernel reports null.  How each figure was taken is in profiles/.
_TREE_SRC = ("gdn_tree_tc.cu", "gdn_prep_common.cuh", "gdn_tc_ptx.cuh", "gdn_internal.cuh")
_GEMM_SRC = ("gdn_gemm.cu", "gdn_tc_ptx.cuh", "gdn_internal.cuh")
_GLA_VERIFY_SRC = ("gdn_gla.cu",) + _TREE_SRC
_GLA_COMMIT_SRC = ("gdn_gla.cu", "gdn_internal.cuh")
NCU_TRAFFIC = {
    ("chain8_b1_h8_d256", "chain_g8_kernel"): (2.274e6, ("gdn_chain.cu", "gdn_internal.cuh", "gdn_tc_ptx.cuh"),
                                               "10502adcdbd91ed8"),
    ("tree32_depth6_b1_h8_d256", "tree_fused_tc_kernel"): (2.627e6, _TREE_SRC, "91888a95b7896ca6"),
    ("tree64_depth8_b16_h8_d256", "tree_fused_tc_kernel"): (47.81e6, _TREE_SRC, "91888a95b7896ca6"),
    ("layer_tree64_depth8_b64_hid2048", "tree_verify"): (358.8e6, _TREE_SRC + ("gdn_layer.cu",), "ac989d0002dee1a9"),
    ("layer_tree64_depth8_b64_hid2048", "gemm_in"): (134.6e6, _GEMM_SRC, "e61b6b4b2b2a32d8"),
    ("layer_tree64_depth8_b64_hid2048", "gemm_out"): (43.08e6, _GEMM_SRC, "e61b6b4b2b2a32d8"),
    ("layer_tree64_depth8_b64_hid2048", "conv"): (188.2e6, ("gdn_layer.cu", "gdn_layer.cuh", "gdn_internal.cuh"),
                                                  "066e72e5baf0efbc"),
    ("gla_tree64_depth8_b16_h8_d256", "gla_verify"): (75.80e6, _GLA_VERIFY_SRC, "5cb5e2ac463bfd31"),
    ("gla_tree64_depth8_b16_h8_d256", "gla_commit"): (35.29e6, _GLA_COMMIT_SRC, "e2c276b3adf2e905"),
}
NCU_TRAFFIC_NOTE = ("dram read + write bytes per launch from a serialised ncu capture (cold L2 at kernel "
                    "start; writes still held in L2 when the kernel ends are not counted)")


def source_digest(files):
    import hashlib
    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "speculative_decoding_linear_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    entry = NCU_TRAFFIC.get((workload, kernel))
    if entry is None:
        return None
    nbytes, files, digest = entry
    return nbytes if source_digest(files) == digest else None


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------
def max_over_ranks(x, dist, world, device="cpu"):
    """The largest value of x over all ranks (x itself on one rank): step times are the max over ranks."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, dist, world, device="cpu"):
    """The sum of x over all ranks (units processed by the whole job)."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_rate(units_per_rank, world, seconds):
    """Units processed by all ranks per second of the slowest rank (weak scaling: every rank runs
    its own replica of the workload)."""
    return units_per_rank * world / seconds


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launcher_command(argv, gpus, port):
    """The torchrun command that runs this script on `gpus` ranks of one node."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(gpus),
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)


def check_world(args, world):
    """--gpus must match the launched world: a lone process asked for N > 1 GPUs relaunches itself
    under torchrun (returns the exit code to propagate); a mismatch under a launcher is an error."""
    if world == args.gpus:
        return None
    if world == 1 and "WORLD_SIZE" not in os.environ and args.gpus > 1:
        import torch
        have = torch.cuda.device_count()
        if have < args.gpus:
            sys.stderr.write("bench.py: --gpus %d but only %d GPU(s) visible\n" % (args.gpus, have))
            return 2
        return subprocess.call(launcher_command(sys.argv[1:], args.gpus, _free_port()))
    sys.stderr.write("bench.py: --gpus %d does not match WORLD_SIZE=%d\n" % (args.gpus, world))
    return 2


# ---------------------------------------------------------------------------
# peaks
# ---------------------------------------------------------------------------
def measured_peaks():
    """HBM GB/s and bf16 TFLOP/s (burst and sustained) from MEASURED_PEAKS.json, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d["bf16_tflops_sustained"]), "kind": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "kind": "fallback"}


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
        fd, self.path = tempfile.mkstemp(prefix="gdn_clocks_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
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
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())}


# ---------------------------------------------------------------------------
# timing helpers (CUDA events on the launching stream)
# ---------------------------------------------------------------------------
def soak(graphs, stream, seconds=1.0, sync_every=8):
    """Replay the step graphs for about `seconds` so the clock sampler sees the GPU under this load."""
    t0 = time.time()
    i = 0
    while time.time() - t0 < seconds:
        graphs[i % 2].replay()
        i += 1
        if i % sync_every == 0:
            stream.synchronize()
    stream.synchronize()
    return i


def timed_steps(graphs, steps, stream, torch, dist, world):
    """Exactly `steps` replays between a barrier + synchronize on both sides; the total device time
    (ms, this rank) from CUDA events on `stream`."""
    torch.cuda.synchronize()
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
    return e0.elapsed_time(e1)


def replay_distribution(graphs, n, calls_per_step, stream, torch):
    """Per-call device time of `n` graph replays, each bracketed by its own events: median, p10, p90."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(n):
            graphs[i % 2].replay()
            ev[i + 1].record(stream)
        ev[-1].synchronize()
    us = np.array([ev[i].elapsed_time(ev[i + 1]) * 1e3 / calls_per_step for i in range(n)])
    return {"replays": n, "median_us_per_call": round(float(np.median(us)), 3),
            "p10_us": round(float(np.percentile(us, 10)), 3), "p90_us": round(float(np.percentile(us, 90)), 3)}


def cold_and_warm(call, stream, torch, l2_bytes, reps=5, warm_reps=50):
    """Cold single-call latency (L2 flushed by writing a buffer of twice its size before each call) and
    the L2-warm figure (the same instance called back to back), in microseconds."""
    flush = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device="cuda")
    cold = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            cold.append(e0.elapsed_time(e1) * 1e3)
        call()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(warm_reps):
                call()
        g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
    del flush, g
    return float(np.median(cold)), e0.elapsed_time(e1) * 1e3 / warm_reps


# ---------------------------------------------------------------------------
# tree / chain workloads: R layer instances on one GPU
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


def draw_tree_workload(wl, cfg, seed, batch, shard_mode, world, rank):
    from speculative_decoding_linear_gb300 import shard
    w = wl.make_workload(cfg, seed=seed, B=batch)
    return shard.shard_workload(w, world, rank) if shard_mode == "sequences" else w


def layer_call(gdnspec, ly, parity, chain):
    """One decode step of one layer: the previous accepted path's commit fused into the new verify."""
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


def l2_size(torch, device_index):
    props = torch.cuda.get_device_properties(device_index)
    return int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 2 ** 20


def run_tree(cfg, steps, warmup, rank, world, device_index, torch, dist, profile=False, batch=None, layers=None,
             shard_mode="replicas", extras=True, side=True):
    """Commit + verify calls of workload `cfg` over a rotation of layer instances."""
    from speculative_decoding_linear_gb300 import gdnspec
    from speculative_decoding_linear_gb300 import workloads as wl

    torch.cuda.set_device(device_index)
    device = torch.device("cuda", device_index)
    spec = wl.SPECS[cfg]
    chain = spec.tree == "chain"
    l2 = l2_size(torch, device_index)
    # replicas: every rank its own draws; sequences: one global draw per layer, sliced by rank
    seed_base = 1000 * (rank + 1) + cfg if shard_mode == "replicas" else 1000 + cfg

    probe = Layer(draw_tree_workload(wl, cfg, None, batch, shard_mode, world, rank), device, torch, gdnspec)
    per_layer = probe.nbytes()
    del probe
    R = max(2, -(-4 * l2 // per_layer)) if layers is None else max(2, layers)
    lys = [Layer(draw_tree_workload(wl, cfg, seed_base + 7919 * r, batch, shard_mode, world, rank), device, torch,
                 gdnspec) for r in range(R)]
    footprint = sum(ly.nbytes() for ly in lys)

    stream = torch.cuda.Stream(device=device)
    # consecutive calls of the sweep touch different layers: launch overlap is safe
    gdnspec.gdn_set_launch_overlap(True)
    with torch.cuda.stream(stream):
        for ly in lys:
            first_verify(gdnspec, ly, chain)
        assert gdnspec.gdn_last_error(stream) == 0
        for parity in (0, 1):                    # eager warm-up of both parities before capture
            for ly in lys:
                layer_call(gdnspec, ly, parity, chain)
        assert gdnspec.gdn_last_error(stream) == 0
        graphs = []
        for parity in (0, 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for ly in lys:
                    layer_call(gdnspec, ly, parity, chain)
            graphs.append(g)
        for i in range(max(warmup, 3)):
            graphs[i % 2].replay()
        stream.synchronize()
        assert gdnspec.gdn_last_error(stream) == 0

        sampler = ClockSampler(device_index)
        sampler.start()
        if not profile:
            soak(graphs, stream, 1.0, 16)
        ms_local = timed_steps(graphs, steps, stream, torch, dist, world)
        clocks = sampler.stop()
        assert gdnspec.gdn_last_error(stream) == 0
        dist_rec = None if profile else replay_distribution(graphs, max(100, steps), R, stream, torch)
    ms = max_over_ranks(ms_local, dist, world, device)

    w0 = lys[0].w
    B, N, H, dk, dv = w0.B, w0.N, w0.H, w0.dk, w0.dv
    units = sum_over_ranks(B * N * R * steps, dist, world, device)
    cold = warm = None
    if not profile and extras:
        ly0 = lys[0]
        parity = [0]

        def one():
            layer_call(gdnspec, ly0, parity[0], chain)
            parity[0] ^= 1
        # the single-call figures without launch overlap: one call has nothing to overlap with
        prev = gdnspec.gdn_set_launch_overlap(False)
        cold, warm = cold_and_warm(one, stream, torch, l2)
        gdnspec.gdn_set_launch_overlap(prev)
    e2e = None if profile or not (extras and side) else run_e2e(lys, steps, chain, gdnspec, torch, stream, world,
                                                               dist, device, shard_mode)
    more = extras and side and not profile and not chain
    baselines = run_replay_baselines(lys, gdnspec, torch, stream, max(5, min(steps, 20))) if more else None
    hybrid = run_hybrid_comparison(lys, gdnspec, torch, stream, max(5, min(steps, 20)), device, wl) if more else None
    prune = run_prune_timing(gdnspec, torch, stream, device, wl, B=B, N=N) if more else None

    esz = 2 if w0.dtype == wl.BF16 else 4
    per_call = float(np.mean([algorithmic_bytes(B, N, H, dk, dv, esz, int(np.sum(ly.w.path >= 0)),
                                                ly.w.path.shape[1], chain) for ly in lys]))
    t_call_s = ms / 1e3 / (steps * R)
    peaks = measured_peaks()
    achieved = per_call / t_call_s / 1e9
    fused_tree = not chain and dk == 256 and dv == 256
    kernel = "chain_g8_kernel" if chain else "tree_fused_tc_kernel" if fused_tree else "tree_contract_tc_kernel"
    launches = 1 if chain else verifier_launches(lys[0].w, torch, device_index)
    replays = None
    if dist_rec is not None:
        replays = dict(dist_rec)
        replays["cold_single_call_us"] = None if cold is None else round(cold, 3)
        replays["l2_warm_us_per_call"] = None if warm is None else round(warm, 3)
        replays["what"] = ("median over graph replays of the %d-layer rotation (each visit reads its state from "
                           "HBM); cold = one call after writing a 2x-L2 buffer, launch overlap off; warm = one "
                           "layer instance called back to back (footprint %.0f MB vs %.0f MB of L2)"
                           % (R, per_layer / 1e6, l2 / 1e6))
    return dict(
        value=units / (ms / 1e3), ms=ms / steps, R=R, footprint=footprint, l2=l2, clocks=clocks, e2e=e2e,
        spec=spec, B=B, N=N, H=H, dk=dk, dv=dv, chain=chain, replays=replays,
        roofline={"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm"], "unit": "GB/s",
                  "frac": round(achieved / peaks["hbm"], 4), "traffic": ncu_traffic(spec.name, kernel),
                  "traffic_note": NCU_TRAFFIC_NOTE, "peak_kind": peaks["kind"] + " hbm_gbs (copy)",
                  "kernel": "gdn_commit_%s_verify (%s, %d launch%s per call)"
                            % ("chain" if chain else "tree", kernel, launches, "" if launches == 1 else "es"),
                  "algorithmic_bytes_per_call": per_call, "t_call_us": round(t_call_s * 1e6, 3),
                  "t_call_from": "CUDA events around the timed graph replays / calls (launch overlap on)"},
        gpu_launches=launches * R * steps, baselines=baselines, hybrid=hybrid, prune=prune,
    )


# ---------------------------------------------------------------------------
# replay baselines: what tree verification and the factor-buffer commit replace
# ---------------------------------------------------------------------------
def run_replay_baselines(layers, gdnspec, torch, stream, steps):
    """Per-call device time of tree verification vs replaying every root-to-leaf path, and of the
    factor-buffer commit vs replaying the accepted tokens and vs restoring a snapshot of the accepted
    node's state, on the same layer rotation (no launch overlap for any side).  Commits write to a
    scratch state so the inputs stay unchanged."""
    prev = gdnspec.gdn_set_launch_overlap(False)
    scratch = [torch.empty_like(ly.S) for ly in layers]
    w0 = layers[0].w
    # every node's state, for the snapshot baseline (one buffer shared by the rotation)
    S_nodes = torch.empty((w0.N, w0.B, w0.H, w0.dv, w0.dk), dtype=torch.float32, device=layers[0].S.device)

    def variant(name):
        def call(ly, sc):
            w = ly.w
            if name == "tree_verify":
                gdnspec.gdn_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out, ly.fac[0], ly.ws)
            elif name == "replay_verify":
                gdnspec.gdn_replay_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out)
            elif name == "factor_commit":
                gdnspec.gdn_commit(ly.S, ly.fac[0], ly.path, sc, w.N, w.dtype)
            elif name == "snapshot_verify":
                gdnspec.gdn_snapshot_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out, S_nodes)
            elif name == "snapshot_commit":
                gdnspec.gdn_snapshot_commit(S_nodes, ly.S, ly.parent, ly.path, sc)
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
    us = {n: variant(n) for n in ("tree_verify", "replay_verify", "factor_commit", "replay_commit",
                                  "snapshot_verify", "snapshot_commit")}
    gdnspec.gdn_set_launch_overlap(prev)
    del scratch, S_nodes
    return {"us_per_call": {k: round(v, 3) for k, v in us.items()},
            "replay_verify_over_tree_verify": round(us["replay_verify"] / us["tree_verify"], 2),
            "replay_commit_over_factor_commit": round(us["replay_commit"] / us["factor_commit"], 2),
            "snapshot_verify_over_tree_verify": round(us["snapshot_verify"] / us["tree_verify"], 2),
            "snapshot_commit_over_factor_commit": round(us["snapshot_commit"] / us["factor_commit"], 2),
            "what": "per layer call, %s, same rotation of %d layers; replay = every root-to-leaf path "
                    "(verify) or the accepted tokens (commit) run token by token from S0; snapshot = every "
                    "node's state built from its parent's and stored (verify, one launch per node index), "
                    "then the accepted node's state copied (commit)" % (w0.spec.name, len(layers))}


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
    hws_bytes = gdnspec.gdn_hybrid_workspace_bytes(w0.B, w0.N, w0.H, w0.dk, w0.dv)
    hws = torch.empty(hws_bytes, dtype=torch.uint8, device=device) if hws_bytes else None   # calls in stream order
    for name, lys in (("bench_trees", layers), ("narrow_trees", narrow)):
        tree = [lambda ly=ly: gdnspec.gdn_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S, ly.out,
                                                      ly.fac[0], ly.ws) for ly in lys]
        hyb = [lambda ly=ly: gdnspec.gdn_hybrid_tree_verify(ly.q, ly.k, ly.v, ly.alpha, ly.beta, ly.parent, ly.S,
                                                            ly.out, ly.fac[0], hws) for ly in lys]
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


# ---------------------------------------------------------------------------
# gated linear attention (per-channel gates): verify and commit of its own record
# ---------------------------------------------------------------------------
def gla_bytes(B, N, H, dk, dv, esz, L_total, Lmax):
    """Algorithmic bytes of one GLA verify and of one GLA commit call."""
    verify = (B * H * dv * dk * 4                                   # read S0
              + B * N * H * (2 * dk + dv) * esz + B * N * H * (dk + 1) * 4 + B * N * 4   # q k v, gates, beta, parents
              + B * N * H * dv * 4                                   # o
              + B * H * N * (dv * 4 + dk * esz + dk * 4) + B * N * 4)   # record: delta, key, g per channel, parent
    commit = 2 * B * H * dv * dk * 4 + L_total * H * (dv * 4 + dk * esz + dk * 4) + B * Lmax * 4 + B * N * 4
    return verify, commit


def run_gla(steps, rank, world, device_index, torch, shard_mode, l2):
    """gdn_gla_tree_verify and gdn_gla_commit on the 16 x 64-node, 8-head, d = 256 batch with per-channel gates,
    each timed over a rotation of layer instances (footprint >= 4x L2) replayed as a CUDA graph."""
    from speculative_decoding_linear_gb300 import gdnspec, shard
    from speculative_decoding_linear_gb300 import workloads as wl
    device = torch.device("cuda", device_index)

    def draw(seed):
        w = wl.make_gla_workload(3, seed=seed)
        return shard.shard_workload(w, world, rank) if shard_mode == "sequences" else w

    class G:
        def __init__(self, w):
            bf = lambda x: torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).to(device)
            self.w = w
            self.q, self.k, self.v = bf(w.q), bf(w.k), bf(w.v)
            self.alpha = torch.from_numpy(w.alpha).to(device)
            self.beta = torch.from_numpy(w.beta).to(device)
            self.parent = torch.from_numpy(w.parent).to(device)
            self.path = torch.from_numpy(w.path).to(device)
            self.S = torch.from_numpy(w.S0).to(device)
            self.S_new = torch.empty_like(self.S)
            self.out = torch.empty((w.B, w.N, w.H, w.dv), dtype=torch.float32, device=device)
            self.fac = torch.empty(gdnspec.gdn_gla_factors_bytes(w.B, w.N, w.H, w.dk, w.dv, w.dtype),
                                   dtype=torch.uint8, device=device)
            self.ws = torch.empty(gdnspec.gdn_gla_workspace_bytes(w.B, w.N, w.H, w.dk, w.dv), dtype=torch.uint8,
                                  device=device)

        def nbytes(self):
            ts = [self.q, self.k, self.v, self.alpha, self.beta, self.parent, self.path, self.S, self.S_new, self.out,
                  self.fac, self.ws]
            return sum(t.numel() * t.element_size() for t in ts)

    first = G(draw(2000 + rank))
    R = max(2, -(-4 * l2 // first.nbytes()))
    gs = [first] + [G(draw(2000 + rank + 7919 * r)) for r in range(1, R)]
    stream = torch.cuda.Stream(device=device)
    verify = [lambda g=g: gdnspec.gdn_gla_tree_verify(g.q, g.k, g.v, g.alpha, g.beta, g.parent, g.S, g.out, g.fac,
                                                      g.ws) for g in gs]
    commit = [lambda g=g: gdnspec.gdn_gla_commit(g.S, g.fac, g.path, g.S_new, g.w.N, g.w.dtype) for g in gs]
    t_v = time_calls(verify, torch, stream, max(5, min(steps, 20)))
    t_c = time_calls(commit, torch, stream, max(5, min(steps, 20)))
    assert gdnspec.gdn_last_error(stream) == 0
    w = gs[0].w
    L_total = float(np.mean([int(np.sum(g.w.path >= 0)) for g in gs]))
    vb, cb = gla_bytes(w.B, w.N, w.H, w.dk, w.dv, 2, L_total, w.path.shape[1])
    peaks = measured_peaks()

    def rl(nbytes, us, kernel, key):
        ach = nbytes / (us * 1e-6) / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm"], 4), "algorithmic_bytes_per_call": nbytes, "t_call_us": round(us, 3),
                "kernel": kernel, "traffic": ncu_traffic(w.spec.name, key), "traffic_note": NCU_TRAFFIC_NOTE,
                "peak_kind": peaks["kind"] + " hbm_gbs (copy)"}
    units = (w.B * world if shard_mode == "replicas" else wl.SPECS[3].B) * w.N     # sequences of the whole job
    res = {"workload": w.spec.name, "B": w.B, "N": w.N, "H": w.H, "dk": w.dk, "dv": w.dv, "layers_rotated": R,
           "verify": rl(vb, t_v, "gdn_gla_tree_verify (gla_prep_kernel + tree_contract_tc_kernel<1> in linear mode)",
                        "gla_verify"),
           "commit": rl(cb, t_c, "gdn_gla_commit (gla_commit_kernel)", "gla_commit"),
           "nodes_per_s_verify_plus_commit": round(units / ((t_v + t_c) * 1e-6), 1),
           "what": "per call, launch overlap off, CUDA-graph replays of the rotation; per-channel gates "
                   "alpha = exp(-softplus(U(-3, 1))) per key channel"}
    del gs
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# full GDN layer decode step: projections, ancestor-window conv, gates, tree
# verification with the pending commit fused in, output gate, o_proj
# ---------------------------------------------------------------------------
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


def draw_layer_workload(wl, seed, shard_mode, world, rank):
    from speculative_decoding_linear_gb300 import shard
    w = wl.make_layer_workload(4, seed=seed)
    return shard.shard_workload(w, world, rank) if shard_mode == "sequences" else w


def layer_kernel_times(lys, gdnspec, torch, stream, steps, parity0):
    """Average device time (us) of each of the layer step's five stages (the verifier one or two launches)
    over `steps` passes of the
    rotation, from CUDA events the library records on the launching stream between the kernels
    (gdn_layer_stage_events); calls are eager, so kernels of consecutive calls do not overlap."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(LAYER_KERNELS) + 1)]
          for _ in range(steps * len(lys))]
    i = 0
    with torch.cuda.stream(stream):
        for e in ev:                      # torch creates the CUDA event at its first record
            for x in e:
                x.record(stream)
        for s in range(steps):
            for ly in lys:
                gdnspec.gdn_layer_stage_events(ev[i])
                ly.call(gdnspec, (parity0 + s) % 2)
                i += 1
        gdnspec.gdn_layer_stage_events(None)
        stream.synchronize()
    assert gdnspec.gdn_last_error(stream) == 0
    tot = np.zeros(len(LAYER_KERNELS))
    for e in ev:
        tot += [e[k].elapsed_time(e[k + 1]) for k in range(len(LAYER_KERNELS))]
    return {k: float(t) * 1e3 / len(ev) for k, t in zip(LAYER_KERNELS, tot)}, (parity0 + steps) % 2


def run_layer(steps, warmup, rank, world, device_index, torch, dist, profile=False, layers=None,
              shard_mode="replicas"):
    from speculative_decoding_linear_gb300 import gdnspec
    from speculative_decoding_linear_gb300 import workloads as wl

    torch.cuda.set_device(device_index)
    device = torch.device("cuda", device_index)
    spec = wl.SPECS[4]
    l2 = l2_size(torch, device_index)
    seed_base = 1000 * (rank + 1) + 4 if shard_mode == "replicas" else 1004
    first = LayerStep(draw_layer_workload(wl, seed_base, shard_mode, world, rank), device, torch, gdnspec)
    per_layer = first.nbytes()
    R = max(2, -(-4 * l2 // per_layer)) if layers is None else max(2, layers)
    lys = [first] + [LayerStep(draw_layer_workload(wl, seed_base + 7919 * r, shard_mode, world, rank), device, torch,
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
        if not profile:
            soak(graphs, stream, 1.0, 4)
        ms_local = timed_steps(graphs, steps, stream, torch, dist, world)
        clocks = sampler.stop()
        assert gdnspec.gdn_last_error(stream) == 0
        dist_rec = None if profile else replay_distribution(graphs, max(100, steps), R, stream, torch)
        # replays end on graph parity (n - 1) % 2; the next eager call takes the other parity
        parity = 0 if dist_rec is None else max(100, steps) % 2
        kt, parity = (None, parity) if profile else layer_kernel_times(lys, gdnspec, torch, stream,
                                                                      max(3, min(steps, 10)), parity)
        seq = None if profile else run_sequential_baseline(lys[0], gdnspec, torch, stream, steps=3)
        model = None if profile else run_model_step(gdnspec, torch, stream, device, wl)
    ms = max_over_ranks(ms_local, dist, world, device)
    cold = warm = None
    if not profile:
        ly0 = lys[0]
        par = [parity]

        def one():
            ly0.call(gdnspec, par[0])
            par[0] ^= 1
        cold, warm = cold_and_warm(one, stream, torch, l2, reps=3, warm_reps=5)

    e2e = None if profile else run_e2e_layer(lys, steps, gdnspec, torch, stream, world, dist, device, shard_mode)
    w0 = lys[0].w
    units = sum_over_ranks(w0.B * w0.N * R * steps, dist, world, device)
    t_call_s = ms / 1e3 / (steps * R)
    flops = layer_flops(w0.B, w0.N, w0.H, w0.hidden, w0.dk, w0.dv)
    peaks = measured_peaks()
    step_tensor = {"achieved": round(flops / t_call_s / 1e12, 1), "peak": peaks["bf16_sustained"],
                   "unit": "TFLOP/s", "frac": round(flops / t_call_s / 1e12 / peaks["bf16_sustained"], 4),
                   "algorithmic_flops_per_call": flops, "t_call_us": round(t_call_s * 1e6, 3),
                   "what": "whole layer step: useful projection flops / step time (graph replays), against the "
                           "measured sustained bf16 peak"}
    roofline = {"bound": "tensor", "kernel": "gdn_layer_tree_step (whole step)", **step_tensor, "traffic": None}
    if kt is not None:
        L_total = float(np.mean([int(np.sum(ly.w.path >= 0)) for ly in lys]))
        work = layer_kernel_work(w0.B, w0.N, w0.H, w0.hidden, w0.dk, w0.dv, L_total, w0.path.shape[1])
        total = sum(kt.values())
        per = []
        for k in LAYER_KERNELS:
            bound, amount, unit = work[k]
            t = kt[k] * 1e-6
            if bound == "hbm":
                ach, peak, u = amount / t / 1e9, peaks["hbm"], "GB/s"
                pk = peaks["kind"] + " hbm_gbs (copy)"
            else:
                ach, peak, u = amount / t / 1e12, peaks["bf16_sustained"], "TFLOP/s"
                pk = peaks["kind"] + " bf16_tflops_sustained (cuBLAS, long loop)"
            per.append({"kernel": LAYER_KERNEL_NAMES[k], "bound": bound, "t_us": round(kt[k], 2),
                        "share": round(kt[k] / total, 4), "achieved": round(ach, 1), "peak": peak, "unit": u,
                        "frac": round(ach / peak, 4), "peak_kind": pk,
                        ("algorithmic_bytes" if bound == "hbm" else "algorithmic_flops"): amount,
                        "traffic": ncu_traffic(spec.name, k)})
        top = max(per, key=lambda r: r["t_us"])
        roofline = {"bound": top["bound"], "achieved": top["achieved"], "peak": top["peak"], "unit": top["unit"],
                    "frac": top["frac"], "traffic": top["traffic"], "traffic_note": NCU_TRAFFIC_NOTE,
                    "peak_kind": top["peak_kind"], "kernel": top["kernel"] + " -- the step's dominant kernel",
                    "t_kernel_us": top["t_us"],
                    "t_kernel_from": "CUDA events recorded by the library between the step's kernels "
                                     "(gdn_layer_stage_events), eager calls over the same rotation",
                    "per_kernel": per, "step": step_tensor}
    replays = None
    if dist_rec is not None:
        replays = dict(dist_rec)
        replays["cold_single_call_us"] = None if cold is None else round(cold, 3)
        replays["l2_warm_us_per_call"] = None if warm is None else round(warm, 3)
        replays["what"] = ("median over graph replays of the %d-layer rotation; cold = one layer step after "
                           "writing a 2x-L2 buffer; warm = one instance called back to back (its %.0f MB "
                           "footprint exceeds the %.0f MB L2, so this is not L2-resident)"
                           % (R, per_layer / 1e6, l2 / 1e6))
    return dict(
        value=units / (ms / 1e3), ms=ms / steps, R=R, footprint=footprint, l2=l2, clocks=clocks, e2e=e2e,
        spec=spec, B=w0.B, N=w0.N, H=w0.H, dk=w0.dk, dv=w0.dv, hidden=w0.hidden, chain=False, layer=True,
        sequential=seq, model=model, roofline=roofline, replays=replays,
        # GEMM, conv, tree verifier, gate, GEMM
        gpu_launches=(4 + verifier_launches(w0, torch, device_index)) * R * steps,
    )


def verifier_launches(w, torch, device_index):
    """Kernels of one tree verification: one at d_k = d_v = 256 (a second launch when the (sequence,
    head) pairs fill whole waves of the SMs plus a remainder that fits one wave as two CTAs per pair),
    else the prologue and the contraction."""
    if not (w.dk == 256 and w.dv == 256):
        return 2
    sms = torch.cuda.get_device_properties(device_index).multi_processor_count
    pairs = w.B * w.H
    rest = pairs % sms
    return 2 if pairs > sms // 2 and 0 < rest and 2 * rest <= sms else 1


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


def _e2e_rate(units_local, sec, world, dist, device):
    units = sum_over_ranks(units_local, dist, world, device)
    return units / sec


def pipelined_e2e(objs, in_names, out_names, run_step, k, torch, stream, world, dist, device):
    """k steps through the public API, each step's inputs copied in from pinned host memory and its
    outputs copied out, inside the timed region.  The copies run on their own streams (host-to-device
    and device-to-host) against two device copies of the packed inputs and outputs, ordered by
    events: step s + 1's inputs go in and step s's outputs come out while the neighbouring step
    computes.  Returns (seconds for k steps, bytes in per step, bytes out per step)."""
    dev_in, host_in = pack_tensors(objs, in_names, torch, device)
    dev_out, host_out = pack_tensors(objs, out_names, torch, device)
    bufs = {"in": [dev_in, torch.empty_like(dev_in)], "out": [dev_out, torch.empty_like(dev_out)]}
    views = [{}, {}]
    for o in objs:
        for kind, names in (("in", in_names), ("out", out_names)):
            for n in names:
                v = getattr(o, n)
                off = v.data_ptr() - bufs[kind][0].data_ptr()
                nb = v.numel() * v.element_size()
                views[0][(id(o), n)] = v
                views[1][(id(o), n)] = bufs[kind][1][off: off + nb].view(v.dtype).view(v.shape)
    h2d, d2h = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]      # set b's inputs have landed
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]    # the step on set b has computed
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]     # set b's outputs have been copied out
    used = [False, False]

    def step(s):
        b = s % 2
        if used[b]:                                       # set b is read until its last step computed
            h2d.wait_event(ev_done[b])
        with torch.cuda.stream(h2d):
            bufs["in"][b].copy_(host_in, non_blocking=True)
            ev_in[b].record(h2d)
        stream.wait_event(ev_in[b])
        if used[b]:                                       # and its outputs are out before they are rewritten
            stream.wait_event(ev_out[b])
        for o in objs:
            for n in in_names + out_names:
                setattr(o, n, views[b][(id(o), n)])
        with torch.cuda.stream(stream):
            run_step(s)
            ev_done[b].record(stream)
        d2h.wait_event(ev_done[b])
        with torch.cuda.stream(d2h):
            host_out.copy_(bufs["out"][b], non_blocking=True)
            ev_out[b].record(d2h)
        used[b] = True

    step(0)
    step(1)
    for st in (h2d, stream, d2h):
        st.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for s_ in range(k):
        step(s_)
    for st in (h2d, stream, d2h):
        st.synchronize()
    t1 = time.perf_counter()
    return t1 - t0, host_in.numel(), host_out.numel()


def run_e2e_layer(lys, steps, gdnspec, torch, stream, world, dist, device, shard_mode="replicas"):
    """Layer step through the public API with every instance's X, parent_idx and accepted path copied
    in from pinned host memory (one transfer) and the layer outputs copied out (one transfer), every
    step; the transfers overlap the neighbouring steps' compute (pipelined_e2e)."""
    k = max(4, min(steps, 10))

    def run_step(s_):
        for ly in lys:
            ly.call(gdnspec, s_ % 2)
    sec, h2d, d2h = pipelined_e2e(lys, ["X", "parent", "path"], ["out"], run_step, k, torch, stream, world, dist,
                                  device)
    sec = max_over_ranks(sec, dist, world, device)
    w = lys[0].w
    return {"value": _e2e_rate(w.B * w.N * len(lys) * k, sec, world, dist, device), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k, "ms_per_step": 1e3 * sec / k,
            "copies": "host-to-device and device-to-host on their own streams, double-buffered device packs, "
                      "overlapping the neighbouring steps' compute"}


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


def run_e2e(layers, steps, chain, gdnspec, torch, stream, world, dist, device, shard_mode="replicas"):
    """Same metric through the public API: every layer call made from the host each step, with all
    layers' draft inputs copied in from pinned host memory (one transfer) and their outputs copied
    out (one transfer) inside the timed region; the transfers overlap the neighbouring steps'
    compute (pipelined_e2e)."""
    names = ["q", "k", "v", "alpha", "beta", "path"] + ([] if chain else ["parent"])
    k = max(4, min(steps, 10))

    def run_step(s_):
        for ly in layers:
            layer_call(gdnspec, ly, s_ % 2, chain)
    sec, h2d, d2h = pipelined_e2e(layers, names, ["out"], run_step, k, torch, stream, world, dist, device)
    sec = max_over_ranks(sec, dist, world, device)
    w = layers[0].w
    return {"value": _e2e_rate(w.B * w.N * len(layers) * k, sec, world, dist, device), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k, "ms_per_step": 1e3 * sec / k,
            "copies": "host-to-device and device-to-host on their own streams, double-buffered device packs, "
                      "overlapping the neighbouring steps' compute"}


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


def reference_config(cfg, wl):
    """The workload keys of the GPU arm's `config` (config_record), for the full workload; the reference
    times a bounded sample of it, described in its cpu_baseline.sample."""
    spec = wl.SPECS[cfg]
    layer = cfg == 4
    out = {"workload": spec.name, "B": spec.B, "N": spec.N, "H": spec.H, "dk": spec.dk, "dv": spec.dv,
           "qkv": spec.dtype, "state": "f32",
           "step": ("full GDN layer step: projections, ancestor-window conv, gates, tree verify with the "
                    "pending commit (state + conv history) fused in, output gate, o_proj") if layer else
                   "per layer: pending commit fused into the next %s verify" % ("chain" if cfg == 1 else "tree")}
    if layer:
        out["hidden"] = spec.hidden
    return out


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
        sample = ("one full-layer step of 2 of the 64 sequences of %s per step (numpy fp64 projections/conv/"
                  "o_proj + path-walk recurrence + commit), %d threads" % (w.spec.name, cores))
    else:
        w = wl.make_workload(args.config)
        timer = oracle_layer_seconds
        sample = ("one layer instance of %s per step (verify all nodes by path walks + commit), fp64, %d threads"
                  % (w.spec.name, cores))
    for _ in range(max(args.warmup, 1)):
        timer(w, cores)
    sec = sum(timer(w, cores) for _ in range(args.steps))
    value = w.B * w.N * args.steps / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": reference_config(args.config, wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def config_record(r, spec, world, shard_mode):
    cfg = {"workload": spec.name, "B": r["B"], "N": r["N"], "H": r["H"], "dk": r["dk"], "dv": r["dv"],
           "qkv": spec.dtype, "state": "f32",
           "step": ("full GDN layer step: projections, ancestor-window conv, gates, tree verify with the "
                    "pending commit (state + conv history) fused in, output gate, o_proj") if r.get("layer") else
                   "per layer: pending commit fused into the next %s verify" % ("chain" if r["chain"] else "tree"),
           "layers_rotated": r["R"], "footprint_bytes": r["footprint"], "l2_bytes": r["l2"],
           "l2_policy": ("inputs larger than L2: %d-layer rotation, footprint >= 4x L2" % r["R"])
           if r["footprint"] >= 4 * r["l2"] else "profiling rotation of %d layers (footprint below 4x L2)" % r["R"],
           "parallelism": ("single GPU" if world == 1 else
                           "replicas" if shard_mode == "replicas" else "sequences sharded across ranks")}
    if r.get("layer"):
        cfg["hidden"] = r["hidden"]
    return cfg


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--shard", default="replicas", choices=["replicas", "sequences"],
                    help="replicas: every rank its own workload (weak scaling); sequences: the batch's "
                         "sequences split across ranks (strong scaling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="skip the verify+commit sub-record of the layer line")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch size")
    ap.add_argument("--gla-only", action="store_true",
                    help="for profiler runs: only the per-channel-gate (GLA) verify and commit record")
    ap.add_argument("--profile", action="store_true",
                    help="for profiler runs: no clock soak, no e2e leg, no CPU baseline, no side records")
    ap.add_argument("--layers", type=int, default=None,
                    help="for profiler runs: rotate this many layers instead of >= 4x L2 of them")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    rc = check_world(args, world)
    if rc is not None:
        sys.exit(rc)

    if args.impl == "reference":
        run_reference(args)
        return

    import torch
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
    if args.gla_only:
        rec = run_gla(args.steps, rank, world, local, torch, args.shard, l2_size(torch, local))
        if rank == 0:
            print(json.dumps(rec), flush=True)
        return
    sub = small = None
    if args.config == 4:
        r = run_layer(args.steps, args.warmup, rank, world, local, torch, dist, args.profile, args.layers, args.shard)
        if not (args.profile or args.no_sub):
            torch.cuda.empty_cache()
            sub = run_tree(3, args.steps, args.warmup, rank, world, local, torch, dist, False, None, None, args.shard)
            sub["gla"] = run_gla(args.steps, rank, world, local, torch, args.shard, sub["l2"])
            torch.cuda.empty_cache()
            # the single-sequence workloads: the 8-token chain and the 32-node tree
            small = {c: run_tree(c, args.steps, args.warmup, rank, world, local, torch, dist, False, None, None,
                                 "replicas", True, False) for c in (1, 2)}
    else:
        r = run_tree(args.config, args.steps, args.warmup, rank, world, local, torch, dist, args.profile,
                     args.batch, args.layers, args.shard)

    if rank == 0:
        cpu = None if args.no_cpu_baseline or args.profile or world > 1 else cpu_baseline(args.config)
        spec = r["spec"]
        line = {
            "metric": METRIC, "value": round(r["value"], 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms"], 4),
            "higher_is_better": True, "scaling": "strong" if args.shard == "sequences" and world > 1 else "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_record(r, spec, world, args.shard),
            "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r["e2e"],
            "gpu_launches": r["gpu_launches"], "clocks": r["clocks"], "replays": r.get("replays"),
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
            seq = r["sequential"]
            if seq:
                seq["tree_step_speedup"] = round(r["value"] / seq["value"], 2)
            line["sequential_decode"] = seq
        if sub is not None:
            rec = {"metric": METRIC, "value": round(sub["value"], 1), "unit": UNIT,
                   "ms_per_step": round(sub["ms"], 4), "config": config_record(sub, sub["spec"], world, args.shard),
                   "roofline": sub["roofline"], "replays": sub["replays"], "e2e": sub["e2e"],
                   "gpu_launches": sub["gpu_launches"], "clocks": sub["clocks"]}
            for key, name in (("baselines", "replay_baselines"), ("hybrid", "hybrid_verify"), ("prune", "prune_tree"),
                              ("gla", "gla_verify_commit")):
                if sub.get(key):
                    rec[name] = sub[key]
            line["tree_verify_commit"] = rec
            line["single_sequence"] = {
                s["spec"].name: {"value": round(s["value"], 1), "unit": UNIT, "ms_per_step": round(s["ms"], 4),
                                 "layers_rotated": s["R"], "roofline": s["roofline"], "replays": s["replays"],
                                 "gpu_launches": s["gpu_launches"]} for s in small.values()}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
