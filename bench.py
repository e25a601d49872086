#!/usr/bin/env python3
"""Decode-layer benchmark of the GB300 MoE decode library.

One step = one full decode layer (RMSNorm -> input projection 7168->12288 ->
out-projection 8192->7168 + residual -> RMSNorm -> router/top-8 over 384
experts -> routed + shared SwiGLU experts 7168->2048->7168 -> combine +
residual) on a batch of M tokens, through the library's decode_layer entry
point. Weights are seeded random tensors of the workload's shapes (about
34.5 GB in HBM); activations are seeded N(0,1) rows. The layer is applied
repeatedly to its own output, so routing (and the experts read) changes
every step; the dense weights alternate between two copies. Every step reads
1.1-25 GB, far more than the 129 MB L2.

Reported (one JSON line, rank 0):
  value        device-timed microseconds per step at --batch (CUDA events, inputs resident):
               the K steps captured once as a CUDA graph and replayed --repeats times, the
               median (min/max in the sweep; the stream-launched time of the same K steps is
               reported beside it as us_per_step_stream)
  e2e          same through the C ABI (stream-launched steps) with every step's input
               copied from pinned host memory and its output copied back inside the
               timed region; the copies run on a copy stream over two alternating
               device buffers, overlapping the neighbouring steps
  sweep        the same for every M in --sweep, with weight-stream GB/s (the
               unique bytes the step must read, incl. the actual distinct experts U)
  roofline     dominant kernel of the --batch step: algorithmic bytes / its
               event-timed duration, against the measured HBM copy bandwidth
  workloads    the workload's other configurations, each alone through its entry point
               (--configs): the 4096x4096 projection at one token, the input projection at
               M = 1..64, the out-projection with its residual at M = 1, 4, 16, 64, and the MoE
               layer (moe_layer) at M = 1, 8, 64; µs per call, GB/s and the fraction of the
               measured copy peak, with every kernel's event-timed GB/s beside it
  cpu_baseline the fp64 oracle on the host cores, on one token of the step, median of three
               runs (single_core: the same with one BLAS/OpenMP thread, in a child process)
With --impl reference the fp64 oracle is the timed arm.

Multi-GPU (torchrun, --gpus N): the decode layer does not shard across GPUs
here (replicas only); each rank runs the same workload on its own GPU and the
time is the maximum over ranks.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode layer µs/step and weight-stream HBM GB/s (% of GB300 peak), batch 1–64"
H, N_IN, K_OUT, E, TOPK, I = 7168, 12288, 8192, 384, 8, 2048
WORKLOAD = ("full decode layer step: RMSNorm -> input projection (K=7168, N=12288) -> out-projection "
            "(K=8192, N=7168) + residual -> RMSNorm -> MoE (router W_r[384,7168] fp32, sigmoid, top-8 "
            "renormalised; 384 routed + 1 shared SwiGLU experts 7168->2048->7168), bf16")
EXPERT_BYTES = 3 * I * H * 2
DENSE_BYTES = N_IN * H * 2 + H * K_OUT * 2 + E * H * 4 + 2 * H * 2


SHARD = 1


def set_shard(s: int) -> None:
    """Per-GPU shapes of an s-way tensor-parallel deployment of the layer (the
    pages' TP8 / TP16): the input projection split over its outputs (N_in / s),
    the out-projection over its inputs (K_out / s) and every expert over its
    intermediate size (I / s); hidden size, router (replicated) and top-k
    unchanged. The exchange steps of a TP group (all-reduces) have no one-GPU
    counterpart and are not run."""
    global SHARD, N_IN, K_OUT, I, EXPERT_BYTES, WORKLOAD
    SHARD = int(s)
    N_IN, K_OUT, I = 12288 // SHARD, 8192 // SHARD, 2048 // SHARD
    EXPERT_BYTES = 3 * I * H * 2
    set_experts(E)
    if SHARD > 1:
        WORKLOAD = (f"decode layer step at TP{SHARD} per-GPU shapes: RMSNorm -> input projection (K={H}, "
                    f"N={N_IN}) -> out-projection (K={K_OUT}, N={H}) + residual -> RMSNorm -> MoE (router "
                    f"W_r[{E},{H}] fp32 replicated, sigmoid, top-{TOPK} renormalised; {E} routed + 1 shared "
                    f"SwiGLU experts {H}->{I}->{H}), bf16; no all-reduce")


def set_experts(n: int) -> None:
    """Routed experts in the bank (384 for the workload; fewer only for small profiling captures)."""
    global E, DENSE_BYTES
    E = int(n)
    DENSE_BYTES = N_IN * H * 2 + H * K_OUT * 2 + E * H * 4 + 2 * H * 2


def step_bytes(M: int, U: float) -> float:
    """Unique bytes one step must move: weights read once + activations in/out."""
    act = M * H * 2 * 2 + M * N_IN * 2 * 2
    return DENSE_BYTES + (U + 1) * EXPERT_BYTES + act


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of a kernel, reported while its sources are unchanged (the
# sha256 of the listed files at capture time); null otherwise.
NCU_TRAFFIC = {
    # one-token MoE front launch: dram__bytes_read.sum + dram__bytes_write.sum of two launches of one
    # ncu capture on the 32-expert bank (read 529,558,528 / 529,543,168 B, write 3,401,216 /
    # 242,432 B), scaled to the 384-expert workload: at one token a launch reads what it reads
    # with 384 experts except the router, 352 x 7168 x 4 B more.
    ("moe_front", 1): {"bytes": (529558528 + 529543168) // 2 + (384 - 32) * 7168 * 4 + (3401216 + 242432) // 2,
                       "sources": ("moe_layers_gb300/csrc/route_shared.cu", "moe_layers_gb300/csrc/topk.cuh",
                                   "moe_layers_gb300/csrc/common.cuh", "moe_layers_gb300/csrc/internal.h",
                                   "moe_layers_gb300/csrc/api.cu"),
                       "sha256": "be162b5a3613baf933db184505311049afaa36e83adfa3a0f0da48ce9996eea6"},
}


def captured_traffic(tag: str, M: int):
    import hashlib
    rec = NCU_TRAFFIC.get((tag, M))
    if rec is None:
        return None
    h = hashlib.sha256()
    root = os.path.dirname(os.path.abspath(__file__))
    for f in rec["sources"]:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest() == rec["sha256"] else None


def kernel_bytes(tag: str, M: int, U: float, shared_in: str | None = None) -> float:
    """Algorithmic bytes of one launch of a kernel of the step. shared_in names
    where the one-token schedule runs the shared expert's gate/up ("router":
    inside the routing launch; "gate_up": problem 0 of the gate/up launch;
    "front": one launch of the routing and both gate/ups); its down projection
    then is part of the down launch. None: the shared expert
    has launches of its own (batch >= 2)."""
    b = {
        "in_proj": N_IN * H * 2 + M * H * 2 + M * N_IN * 2,
        "out_proj": H * K_OUT * 2 + M * K_OUT * 2 + 2 * M * H * 2,
        "router": E * H * 4 + M * H * 2,
        "gate_up": U * 2 * I * H * 2 + M * TOPK * (H + I) * 2,
        "down": U * H * I * 2 + M * TOPK * (I * 2 + H * 4),
        "shared_gate_up": 2 * I * H * 2 + M * (H + I) * 2,
        "shared_down": H * I * 2 + M * (I * 2 + H * 4),
    }
    if shared_in == "front":  # one launch: routing, the shared and the routed gate/up
        b["moe_front"] = b["router"] + b["gate_up"] + 2 * I * H * 2 + M * I * 2
        b["down"] += H * I * 2
    elif shared_in is not None:
        b[shared_in] += 2 * I * H * 2 + M * I * 2
        b["down"] += H * I * 2
    return b.get(tag, 0.0)


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, source="fallback")


# ---------------------------------------------------------------------------- distributed helpers
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def reduce_max(value: float, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[int(str(device).split(":")[1])])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.lines, self.proc, self.th = gpu, [], None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.th:
            self.th.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- our arm
def layer_copies() -> int:
    """Weight copies the bench rotates through. At full shapes a step reads
    1.1-25 GB, far above the 129 MB L2, and two dense copies suffice (the router
    and shared expert are re-read only after about 1 GB of other traffic). The
    sharded steps read 80-150 MB, so every weight, router and expert bank
    included, gets enough copies that a step's bytes come back only after four
    times L2 of traffic."""
    if SHARD == 1:
        return 2
    step_m1 = DENSE_BYTES + (TOPK + 1) * EXPERT_BYTES
    return max(2, -(-4 * 129_000_000 // step_m1))


def build_weights(dev: str, copies: int = 2, distinct: bool = False):
    """`copies` layers' weights. distinct: every layer has its own seeded
    values (tensor id + 100 l for layer l: its own projections, router and
    expert banks, about 34.5 GB each at full shapes); otherwise the copies hold
    the same values and only make every step stream its weights from HBM."""
    import torch
    import moe_layers_gb300 as ML
    import synth

    def fill_bf16(shape, tid, sigma):
        t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        synth.fill_bf16_dev(t.data_ptr(), t.numel(), 0, tid, 0, sigma)
        return t

    def moe_weights(l):
        Wg = fill_bf16((E, I, H), synth.W_G + 100 * l, 0.02)
        Wu = fill_bf16((E, I, H), synth.W_U + 100 * l, 0.02)
        Wd = fill_bf16((E, H, I), synth.W_D + 100 * l, 0.02)
        Ws = (fill_bf16((I, H), synth.W_G_S + 100 * l, 0.02), fill_bf16((I, H), synth.W_U_S + 100 * l, 0.02),
              fill_bf16((H, I), synth.W_D_S + 100 * l, 0.02))
        Wr = torch.empty((E, H), dtype=torch.float32, device=dev)
        synth.fill_f32_dev(Wr.data_ptr(), Wr.numel(), 0, synth.W_R + 100 * l, 0, 0.01)
        return Wg, Wu, Wd, Ws, Wr

    ones = torch.ones(H, dtype=torch.bfloat16, device=dev)
    layers = []
    moe = moe_weights(0)
    for c in range(copies):
        l = c if distinct else 0
        if c > 0 and (SHARD > 1 or distinct):
            # sharded steps are small: nothing may stay in L2 from step to step; distinct layers: their own values
            moe = moe_weights(l)
        Wg, Wu, Wd, Ws, Wr = moe
        W_in = fill_bf16((N_IN, H), synth.W_IN + 100 * l, 0.02)
        W_o = fill_bf16((H, K_OUT), synth.W_O + 100 * l, 0.02)
        layers.append(ML.LayerWeights(gamma1=ones, W_in=W_in, W_o=W_o, gamma2=ones, W_r=Wr, Wg=Wg, Wu=Wu, Wd=Wd,
                                      Wg_s=Ws[0], Wu_s=Ws[1], Wd_s=Ws[2], k=TOPK, k_out=K_OUT))
    torch.cuda.synchronize()
    return layers


def _graph_replays(step_fn, K: int, reps: int, dev, reset=None):
    """Capture step_fn(i, stream) for i < K once as a CUDA graph on a side
    stream and replay it `reps` times, each bracketed by CUDA events on the
    launching stream (reset() runs before every replay, untimed). Returns the
    microseconds per step of each replay."""
    import torch
    stream = torch.cuda.current_stream()
    gs = torch.cuda.Stream(device=dev)
    gs.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for i in range(K):
            step_fn(i, gs)
    if reset:
        reset()
    graph.replay()  # (untimed: first replay)
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        if reset:
            reset()
        torch.cuda.synchronize()
        barrier(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        graph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        barrier(dev)
        out.append(g0.elapsed_time(g1) * 1000.0 / K)
    del graph
    return out


def _spread(vals):
    return {"median": round(statistics.median(vals), 2), "min": round(min(vals), 2), "max": round(max(vals), 2),
            "n": len(vals)}


def _kernel_table(prof: dict, K: int, bytes_of, peak: float) -> dict:
    """Per-kernel event-timed averages of a profiled pass: launches per step,
    µs per launch, algorithmic GB/s and fraction of the measured copy peak."""
    kern = {}
    for tag, (n, ms) in prof.items():
        avg_us = ms * 1000.0 / max(n, 1)
        kb = bytes_of(tag)
        gbs = kb / (avg_us * 1e3) if kb and avg_us > 0 else None
        kern[tag] = {"launches_per_step": n / K, "avg_us": round(avg_us, 2),
                     "bytes": int(kb) if kb else None,
                     "GBps": round(gbs, 1) if gbs else None, "frac": round(gbs / peak, 4) if gbs else None}
    return kern


def run_layer_sweep(args, h, layers, cws, dev, peaks):
    """The decode layer (the headline workload) at every batch of the sweep."""
    import numpy as np
    import torch
    import moe_layers_gb300 as ML
    import synth

    stream = torch.cuda.current_stream()
    sweep = sorted(set([int(m) for m in args.sweep.split(",") if m] + [args.batch]))
    results = {}
    for M in sweep:
        ws = h.workspace(("bench", M), ML.decode_layer_workspace_size(h, layers[0], M), ("layer", M))
        if args.verify > 1:
            # speculative-verify batch: groups of `verify` related rows (one request's drafts)
            x0 = synth.correlated_rows(synth.X_BASE + 100, range(M), args.verify, H, 0, args.verify_noise)
        else:
            x0 = synth.bf16_rows(synth.X_BASE + 100, range(M), H, 0)
        host_in = torch.from_numpy(x0.view(np.int16)).view(torch.bfloat16).reshape(M, H).pin_memory()
        host_out = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
        hidden = host_in.to(dev)
        K = args.steps
        idx_all = torch.empty((K, M, TOPK), dtype=torch.int32, device=dev)

        def step(i, trace=None, stream=None):
            ML.decode_layer(h, layers[i % len(layers)], hidden, trace=trace, ws=ws, _cw=cws[i % len(layers)],
                            stream=stream)

        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        # Every timed pass (eager, graph, profiled, e2e) starts from the same
        # input rows, so all of them route the same K steps (the routing, hence
        # the distinct experts U and the bytes, drift as the hidden state evolves).
        hidden.copy_(host_in)
        # ---- timed: inputs resident, K steps launched from the host
        barrier(dev)
        torch.cuda.synchronize()
        launches0 = h.launch_count
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(K):
            step(i, trace={"idx": idx_all[i]})
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(dev)
        us_eager = ev0.elapsed_time(ev1) * 1000.0 / K
        launches = h.launch_count - launches0
        reps = [us_eager]
        if args.graph:
            # The same K steps captured once as a CUDA graph (no host work per
            # step) and replayed `repeats` times: the GPU-bound time.
            reps = _graph_replays(lambda i, s: step(i, trace={"idx": idx_all[i]}, stream=s), K, args.repeats, dev,
                                  reset=lambda: hidden.copy_(host_in))
        idx_host = idx_all.cpu().numpy()
        U = float(np.mean([len(np.unique(idx_host[i])) for i in range(K)]))
        us_max = reduce_max(statistics.median(reps), dev)
        us_eager = reduce_max(us_eager, dev)
        # ---- profiled pass: per-kernel event times (separate; events break PDL overlap)
        hidden.copy_(host_in)
        h.set_profiling(True)
        for i in range(K):
            step(i, trace={"idx": idx_all[i]})
        prof = h.profile_read()
        h.set_profiling(False)
        idx_host = idx_all.cpu().numpy()
        U_prof = float(np.mean([len(np.unique(idx_host[i])) for i in range(K)]))
        # ---- end to end: every step uploads its input rows from pinned host
        # memory and downloads its output rows, through the public API. Two
        # device buffers alternate and the copies run on a copy stream, so step
        # i+1's upload and step i's download overlap the neighbouring steps'
        # layers (as a serving loop would run them); the timed region covers
        # every copy. The inputs of the K steps are the evolving hidden state
        # the device-timed passes saw (recorded by an untimed pass), so that
        # e2e routes the same steps as value does.
        inputs_dev = torch.empty((K, M, H), dtype=torch.bfloat16, device=dev)
        hidden.copy_(host_in)
        for i in range(K):
            inputs_dev[i].copy_(hidden)
            step(i)
        inputs_host = inputs_dev.cpu().pin_memory()
        del inputs_dev
        cstream = torch.cuda.Stream(device=dev)
        bufs = [torch.empty_like(hidden) for _ in range(2)]
        outs = [host_out, torch.empty((M, H), dtype=torch.bfloat16).pin_memory()]
        h2d = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        torch.cuda.synchronize()
        barrier(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cstream.wait_stream(stream)
        with torch.cuda.stream(cstream):
            bufs[0].copy_(inputs_host[0], non_blocking=True)
            h2d[0].record(cstream)
        for i in range(K):
            b = i % 2
            stream.wait_event(h2d[b])
            ML.decode_layer(h, layers[i % len(layers)], bufs[b], ws=ws, _cw=cws[i % len(layers)], stream=stream)
            done[b].record(stream)
            with torch.cuda.stream(cstream):
                if i + 1 < K:  # (the other buffer's download, step i-1's, is already queued before this)
                    bufs[1 - b].copy_(inputs_host[i + 1], non_blocking=True)
                    h2d[1 - b].record(cstream)
                cstream.wait_event(done[b])
                outs[b].copy_(bufs[b], non_blocking=True)
        stream.wait_stream(cstream)
        e1.record(stream)
        torch.cuda.synchronize()
        us_e2e = reduce_max(e0.elapsed_time(e1) * 1000.0 / K, dev)
        b = step_bytes(M, U)
        # one and two tokens: the shared expert runs inside the MoE front (or gate/up) and down launches
        shared_in = None if "shared_gate_up" in prof else "front" if "moe_front" in prof else "gate_up"
        kern = _kernel_table(prof, K, lambda tag: kernel_bytes(tag, M, U_prof, shared_in), peaks["hbm_gbs"])
        results[M] = dict(M=M, us_per_step=round(us_max, 2), us_per_step_replays=_spread(reps),
                          us_per_step_stream=round(us_eager, 2), e2e_us=round(us_e2e, 2), U=round(U, 2),
                          step_bytes=int(b), weight_stream_GBps=round(b / (us_max * 1e3), 1),
                          hbm_frac=round(b / (us_max * 1e3) / peaks["hbm_gbs"], 4),
                          kernels_per_step=launches / K, gpu_launches=launches, kernels=kern)
    return sweep, results


def run_dense_config(args, h, dev, peaks, name, N, Kd, Ms, copies, residual, weights=None):
    """One projection alone (dec_linear or, with residual, dec_linear_residual),
    the workload's shape and N(0, 0.02) weights, at every batch in Ms. The
    weights rotate over `copies` tensors so that every call streams its matrix
    from HBM (copies x bytes >= 4 x L2). µs per call from CUDA-graph replays of
    K calls; per-kernel event times from a profiled pass."""
    import torch
    import moe_layers_gb300 as ML
    import synth
    Ws = list(weights or [])
    tid0 = synth.W_LINEAR + (40 if residual else 0)
    while len(Ws) < copies:
        t = torch.empty((N, Kd), dtype=torch.bfloat16, device=dev)
        synth.fill_bf16_dev(t.data_ptr(), t.numel(), 0, tid0 + len(Ws), 0, 0.02)
        Ws.append(t)
    K = args.steps
    out = {}
    for M in Ms:
        x = torch.empty((M, Kd), dtype=torch.bfloat16, device=dev)
        synth.fill_bf16_dev(x.data_ptr(), x.numel(), 0, synth.X_BASE + 300, 0, 1.0)
        r = None
        if residual:
            r = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            synth.fill_bf16_dev(r.data_ptr(), r.numel(), 0, synth.R_BASE + 300, 0, 1.0)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        nb = ML._load()
        import ctypes
        sz = ctypes.c_size_t()
        ML._check(nb.dec_linear_workspace_size(h.ptr, M, N, Kd, ctypes.byref(sz)), "dec_linear_workspace_size")
        ws = h.workspace(("bench_dense", name, M), sz.value, ("linear", name, M))

        def call(i, s=None):
            W = Ws[i % len(Ws)]
            if residual:
                ML.dec_linear_residual(h, x, W, r, out=y, stream=s, ws=ws)
            else:
                ML.dec_linear(h, x, W, y, stream=s, ws=ws)

        for i in range(args.warmup):
            call(i)
        torch.cuda.synchronize()
        l0 = h.launch_count
        reps = _graph_replays(call, K, args.repeats, dev)
        launches = (h.launch_count - l0) / K
        h.set_profiling(True)
        for i in range(K):
            call(i)
        prof = h.profile_read()
        h.set_profiling(False)
        variant = {ML.VARIANT_SMALL_M: "small_m", ML.VARIANT_SPLIT_K: "split_k"}.get(h.last_variant)
        nbytes = N * Kd * 2 + M * Kd * 2 + M * N * 2 + (M * N * 2 if residual else 0)
        us = statistics.median(reps)
        gbs = nbytes / (us * 1e3)
        out[M] = {"M": M, "us_per_call": _spread(reps), "bytes": nbytes, "GBps": round(gbs, 1),
                  "frac": round(gbs / peaks["hbm_gbs"], 4), "family": variant, "launches_per_call": launches,
                  "kernels": _kernel_table(prof, K, lambda tag: nbytes, peaks["hbm_gbs"])}
    return {"shape": {"N": N, "K": Kd}, "weight_copies": len(Ws), "batches": out}


def run_moe_config(args, h, dev, peaks, layer, Ms):
    """The MoE layer alone (moe_layer: router, top-8, 384 routed + 1 shared
    experts, combine; no RMSNorm, no residual) on fresh N(0, 1) rows every
    step, so the routing and the experts read change from step to step."""
    import numpy as np
    import torch
    import moe_layers_gb300 as ML
    import synth
    wts = ML.MoeWeights(W_r=layer.W_r, Wg=layer.Wg, Wu=layer.Wu, Wd=layer.Wd, Wg_s=layer.Wg_s, Wu_s=layer.Wu_s,
                        Wd_s=layer.Wd_s, k=TOPK)
    cw = wts.c_struct()
    K = args.steps
    res = {}
    for M in Ms:
        xs = torch.empty((K + args.warmup, M, H), dtype=torch.bfloat16, device=dev)
        synth.fill_bf16_dev(xs.data_ptr(), xs.numel(), 0, synth.X_BASE + 400 + M, 0, 1.0)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        idx_all = torch.empty((K, M, TOPK), dtype=torch.int32, device=dev)
        ws = h.workspace(("bench_moe", M), ML.moe_layer_workspace_size(h, wts, M), ("moe_layer", M))

        def call(i, s=None, warm=False):
            x = xs[K + i] if warm else xs[i]
            ML.moe_layer(h, wts, x, out=out, trace=None if warm else {"idx": idx_all[i]}, stream=s, ws=ws, _cw=cw)

        for i in range(args.warmup):
            call(i, warm=True)
        torch.cuda.synchronize()
        l0 = h.launch_count
        reps = _graph_replays(call, K, args.repeats, dev)
        launches = (h.launch_count - l0) / K
        idx_host = idx_all.cpu().numpy()
        U = float(np.mean([len(np.unique(idx_host[i])) for i in range(K)]))
        h.set_profiling(True)
        for i in range(K):
            call(i)
        prof = h.profile_read()
        h.set_profiling(False)
        nbytes = E * H * 4 + (U + 1) * EXPERT_BYTES + 2 * M * H * 2
        us = statistics.median(reps)
        gbs = nbytes / (us * 1e3)
        shared_in = None if "shared_gate_up" in prof else "front" if "moe_front" in prof else "gate_up"
        res[M] = {"M": M, "us_per_call": _spread(reps), "U": round(U, 2), "bytes": int(nbytes), "GBps": round(gbs, 1),
                  "frac": round(gbs / peaks["hbm_gbs"], 4), "launches_per_call": launches,
                  "kernels": _kernel_table(prof, K, lambda tag: kernel_bytes(tag, M, U, shared_in),
                                           peaks["hbm_gbs"])}
    return {"batches": res}


def run_ours(args, rank, local, world):
    import torch
    import moe_layers_gb300 as ML

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    ML.build()
    h = ML.Handle(local)
    h.set_shared_sms(args.shared_sms)
    if args.l2_ahead is not None:
        h.set_l2_ahead(args.l2_ahead)
    h.set_force_variant({"auto": ML.VARIANT_AUTO, "small_m": ML.VARIANT_SMALL_M,
                         "split_k": ML.VARIANT_SPLIT_K}[args.family])
    layers = build_weights(dev, args.layers if args.layers > 0 else layer_copies(), distinct=args.layers > 0)
    if args.prefetch_next:
        # Cross-layer prefetch: while layer l routes, the next layer's input
        # projection is pulled into L2 (up to the given bytes).
        for li, L in enumerate(layers):
            nxt = layers[(li + 1) % len(layers)].W_in
            L.prefetch_next = nxt
            L.prefetch_bytes = min(int(args.prefetch_next), nxt.numel() * 2) // 16 * 16
    cws = [L.c_struct() for L in layers]
    peaks = measured_peaks()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    sweep, results = run_layer_sweep(args, h, layers, cws, dev, peaks)
    # The workload's other configurations, each alone through its entry point.
    workloads = {}
    cfgs = [c for c in args.configs.split(",") if c] if SHARD == 1 and E == 384 else []
    for c in cfgs:
        if c == "proj4096":
            workloads[c] = run_dense_config(args, h, dev, peaks, c, 4096, 4096, [1], 16, False)
            workloads[c]["workload"] = "single decode projection: x[1,4096] W[4096,4096] bf16, y = x W^T"
        elif c == "in_proj":
            workloads[c] = run_dense_config(args, h, dev, peaks, c, N_IN, H, [1, 2, 4, 8, 16, 32, 64], 3, False,
                                            weights=[L.W_in for L in layers])
            workloads[c]["workload"] = "batch-swept input projection: K=7168, N=12288 bf16"
        elif c == "out_proj":
            workloads[c] = run_dense_config(args, h, dev, peaks, c, H, K_OUT, [1, 4, 16, 64], 4, True,
                                            weights=[L.W_o for L in layers])
            workloads[c]["workload"] = "out-projection fused with residual: K=8192, N=7168 bf16, out = r + x W^T"
        elif c == "moe":
            workloads[c] = run_moe_config(args, h, dev, peaks, layers[0], [1, 8, 64])
            workloads[c]["workload"] = ("MoE layer: router W_r[384,7168] fp32 sigmoid top-8 renormalised; 384 "
                                        "routed + 1 shared SwiGLU experts 7168->2048->7168 bf16")
        else:
            raise SystemExit(f"unknown config {c}")
    clk = clocks.stop()
    if h.check_device_error() != ML.DEC_OK:
        raise RuntimeError("device error word set during the benchmark")

    hl = results[args.batch]
    dom = max((t for t in hl["kernels"] if hl["kernels"][t]["GBps"]),  # (kernels with algorithmic bytes)
              key=lambda t: hl["kernels"][t]["avg_us"] * hl["kernels"][t]["launches_per_step"])
    dk = hl["kernels"][dom]
    achieved = dk["GBps"]
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4) if achieved else None,
                "traffic": captured_traffic(dom, args.batch),
                "peak_source": peaks["source"], "avg_us": dk["avg_us"], "bytes_per_launch": dk["bytes"]}
    out = {"metric": METRIC, "value": hl["us_per_step"], "unit": "us/step", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(hl["us_per_step"] / 1000.0, 5), "higher_is_better": False,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic: seeded random-init weights of the workload's shapes, seeded N(0,1) activations",
           "config": {"workload": WORKLOAD if E == 384 else WORKLOAD + f" (profiling variant: {E} routed experts)",
                      "weight_copies": len(layers),
                      "layers": (f"{len(layers)} distinct layers applied in sequence, each step one layer"
                                 if args.layers > 0 else "one layer's weights in rotating copies"),
                      "prefetch_next_bytes": int(args.prefetch_next),
                      "token_rows": ("independent" if args.verify <= 1 else
                                     f"speculative verify: groups of {args.verify} related rows, noise {args.verify_noise}"),
                      "batch": args.batch, "parallelism": "replicas" if world > 1 else "1 GPU",
                      "timing": f"CUDA-graph replays of the K steps, median of {args.repeats} (spread in the sweep)",
                      "l2": "inputs larger than L2: each step reads >= 1.1 GB (L2 129 MB); dense weights alternate "
                            "between 2 copies; routing changes every step",
                      "weight_stream_GBps": hl["weight_stream_GBps"], "hbm_frac": hl["hbm_frac"],
                      "distinct_experts_U": hl["U"], "shared_expert_sms": {0: "auto", -1: "overlap"}.get(args.shared_sms, args.shared_sms),
                      "sweep": [results[m] for m in sweep],
                      "kernels_at_batch": hl["kernels"]},
           "weight_stream_GBps": hl["weight_stream_GBps"], "hbm_frac": hl["hbm_frac"],
           "roofline": roofline,
           "e2e": {"value": hl["e2e_us"], "unit": "us/step", "h2d_bytes_per_step": args.batch * H * 2,
                   "d2h_bytes_per_step": args.batch * H * 2},
           "gpu_launches": hl["gpu_launches"], "clocks": clk}
    if workloads:
        out["workloads"] = workloads
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.batch, steps=3)
    if rank == 0:
        print(json.dumps(out), flush=True)
    h.close()


# ---------------------------------------------------------------------------- oracle arm
def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    env = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(env) if env else (os.cpu_count() or 1)


class _OracleSample:
    """One token of the decode-layer step, as the fp64 oracle computes it.
    Input bytes (weights, the token) are generated before any timing."""

    def __init__(self, M: int):
        import numpy as np
        import synth
        self.M = M
        self.W_in = synth.bf16(N_IN * H, 0, synth.W_IN, 0, 0.02).reshape(N_IN, H)
        self.W_o = synth.bf16(H * K_OUT, 0, synth.W_O, 0, 0.02).reshape(H, K_OUT)
        self.Wr = synth.f32(E * H, 0, synth.W_R, 0, 0.01).reshape(E, H)
        self.g = np.full(H, 0x3F80, dtype=np.uint16)
        self.x = synth.bf16_rows(synth.X_BASE + 100, [0], H, 0)
        self.shared = (synth.bf16(I * H, 0, synth.W_G_S, 0, 0.02).reshape(I, H),
                       synth.bf16(I * H, 0, synth.W_U_S, 0, 0.02).reshape(I, H),
                       synth.bf16(H * I, 0, synth.W_D_S, 0, 0.02).reshape(H, I))
        self.cache = {}

    def expert(self, e: int):
        import synth
        if e not in self.cache:
            n = I * H
            self.cache[e] = (synth.bf16(n, 0, synth.W_G, e * n, 0.02).reshape(I, H),
                             synth.bf16(n, 0, synth.W_U, e * n, 0.02).reshape(I, H),
                             synth.bf16(n, 0, synth.W_D, e * n, 0.02).reshape(H, I))
        return self.cache[e]

    def prepare(self):
        """Route the token once so that its experts' bytes exist before timing."""
        import oracle
        r = oracle.decode_layer(self.x, self.g, self.W_in, self.W_o, self.g, self.Wr, TOPK, self.expert, self.shared,
                                k_out=K_OUT)
        for e in r["idx"][0]:
            self.expert(int(e))

    def run(self) -> float:
        import oracle
        t0 = time.perf_counter()
        oracle.decode_layer(self.x, self.g, self.W_in, self.W_o, self.g, self.Wr, TOPK, self.expert, self.shared,
                            k_out=K_OUT)
        return time.perf_counter() - t0


def cpu_baseline(M: int, steps: int = 1) -> dict:
    s = _OracleSample(M)
    s.prepare()
    secs = [s.run() for _ in range(max(1, steps))]
    per_token_us = statistics.median(secs) * 1e6
    out = {"value": round(per_token_us * M, 1), "unit": "us/step", "cores": blas_threads(), "kind": "oracle",
           "sample": f"1 token of the M={M} decode-layer step (fp64 numpy oracle, weights widened inside), "
                     f"scaled by M; median of {len(secs)} run(s)"}
    one = oracle_one_thread(M)
    if one is not None:
        out["single_core"] = {"value": one, "unit": "us/step", "cores": 1}
    return out


def oracle_one_thread(M: int):
    """The same sample in a child process whose BLAS and OpenMP pools hold one
    thread (the pools are fixed when numpy loads); None if it fails."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-thread", str(M)], env=env,
                           capture_output=True, text=True, timeout=600)
        return round(float(json.loads(r.stdout.strip().splitlines()[-1])["us"]) * M, 1)
    except Exception:
        return None


def _oracle_one_thread_main(M: int) -> None:
    s = _OracleSample(M)
    s.prepare()
    print(json.dumps({"us": s.run() * 1e6}), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    s = _OracleSample(args.batch)
    s.prepare()
    for _ in range(args.warmup):
        s.run()
    secs = [s.run() for _ in range(args.steps)]
    us = sum(secs) / len(secs) * 1e6 * args.batch
    cb = {"value": round(us, 1), "unit": "us/step", "cores": blas_threads(), "kind": "oracle",
          "sample": f"1 token of the M={args.batch} decode-layer step per timed step, scaled by M"}
    print(json.dumps({"metric": METRIC, "value": round(us, 1), "unit": "us/step", "impl": "reference",
                      "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False, "scaling": "weak",
                      "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs as the GPU arm)",
                      "config": {"workload": WORKLOAD, "batch": args.batch, "parallelism": "host cores"},
                      "cpu_baseline": cb,
                      "e2e": {"value": round(us, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}), flush=True)


def main(argv=None):
    if argv is None and len(sys.argv) == 3 and sys.argv[1] == "--oracle-one-thread":
        _oracle_one_thread_main(int(sys.argv[2]))
        return
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=1, help="headline batch M (1..64)")
    ap.add_argument("--sweep", default="1,2,4,8,16,32,64")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--repeats", type=int, default=5, help="CUDA-graph replays per timed point (median reported)")
    ap.add_argument("--configs", default="proj4096,in_proj,out_proj,moe",
                    help="the workload's other configurations, each timed alone (comma list; empty for none): "
                         "proj4096 (4096x4096 projection, M=1), in_proj (7168->12288, M=1..64), out_proj "
                         "(8192->7168 + residual, M=1,4,16,64), moe (the MoE layer, M=1,8,64)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time the K steps as stream launches only (default: also capture them in a CUDA graph "
                         "and report the replay time as the value)")
    ap.add_argument("--shared-sms", type=int, default=0,
                    help="SMs for the shared expert: 0 automatic share (default), -1 every SM overlapped, n fixed")
    ap.add_argument("--family", choices=("auto", "small_m", "split_k"), default="auto",
                    help="kernel family (auto: by batch and size; small_m covers batch <= 4)")
    ap.add_argument("--l2-ahead", type=int, default=None,
                    help="bytes per CTA the small-matrix kernels keep requested into L2 ahead (default: library's)")
    ap.add_argument("--prefetch-next", type=int, default=0,
                    help="bytes of the next layer's input projection to pull into L2 during the routing (0: none)")
    ap.add_argument("--layers", type=int, default=0,
                    help="L distinct layers (their own seeded weights, routers and expert banks, ~34.5 GB each) "
                         "applied in sequence, one per step (0: one layer's weights in rotating copies)")
    ap.add_argument("--verify", type=int, default=1,
                    help="speculative-verify batch: groups of this many related token rows (1: independent rows)")
    ap.add_argument("--verify-noise", type=float, default=0.5,
                    help="per-token deviation from the group's row (rows of a group correlate at 1/(1+x^2))")
    ap.add_argument("--shard", type=int, choices=(1, 8, 16), default=1,
                    help="per-GPU shapes of a TP8 / TP16 deployment (1: the full layer)")
    ap.add_argument("--experts", type=int, default=E,
                    help="routed experts in the bank (default 384, the workload; smaller only for ncu captures)")
    args = ap.parse_args(argv)
    set_experts(args.experts)
    set_shard(args.shard)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 2:
        ap.error("--steps must be at least 2")
    if not 0 <= args.layers <= 6:
        ap.error("--layers must be 0..6 (each full-size layer holds about 34.5 GB)")
    rank, local, world = dist_env()
    if args.impl == "reference":
        if world > 1 and args.steps > 3:
            args.steps = min(args.steps, 20)
        if args.steps > 20:
            args.steps = 20
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl", device_id=torch.device(f"cuda:{local}"))
    try:
        run_ours(args, rank, local, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
