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
               the K steps captured once as a CUDA graph and replayed (the stream-launched
               time of the same K steps is reported beside it as us_per_step_stream)
  e2e          same through the C ABI (stream-launched steps) with every step's input
               copied from pinned host memory and its output copied back inside the
               timed region; the copies run on a copy stream over two alternating
               device buffers, overlapping the neighbouring steps
  sweep        the same for every M in --sweep, with weight-stream GB/s (the
               unique bytes the step must read, incl. the actual distinct experts U)
  roofline     dominant kernel of the --batch step: algorithmic bytes / its
               event-timed duration, against the measured HBM copy bandwidth
  cpu_baseline the fp64 oracle on the host cores, on one token of the step
               (single_core: the same with one BLAS/OpenMP thread, in a child process)
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
    # one-token MoE front launch, full workload: dram__bytes_read.sum + dram__bytes_write.sum,
    # mean of two launches of one ncu capture (read 539.64 / 539.64 MB, write 3.40 / 0.14 MB)
    ("moe_front", 1): {"bytes": (539637248 + 539639808) // 2 + (3399424 + 139776) // 2,
                       "sources": ("moe_layers_gb300/csrc/route_shared.cu", "moe_layers_gb300/csrc/topk.cuh",
                                   "moe_layers_gb300/csrc/common.cuh", "moe_layers_gb300/csrc/internal.h",
                                   "moe_layers_gb300/csrc/api.cu"),
                       "sha256": "7cf579a0bfede19da93d049016e68f13fc581dcc104bb370310bf7361821d986"},
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


def build_weights(dev: str, copies: int = 2):
    import torch
    import moe_layers_gb300 as ML
    import synth

    def fill_bf16(shape, tid, sigma):
        t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        synth.fill_bf16_dev(t.data_ptr(), t.numel(), 0, tid, 0, sigma)
        return t

    def moe_weights():
        Wg = fill_bf16((E, I, H), synth.W_G, 0.02)
        Wu = fill_bf16((E, I, H), synth.W_U, 0.02)
        Wd = fill_bf16((E, H, I), synth.W_D, 0.02)
        Ws = (fill_bf16((I, H), synth.W_G_S, 0.02), fill_bf16((I, H), synth.W_U_S, 0.02),
              fill_bf16((H, I), synth.W_D_S, 0.02))
        Wr = torch.empty((E, H), dtype=torch.float32, device=dev)
        synth.fill_f32_dev(Wr.data_ptr(), Wr.numel(), 0, synth.W_R, 0, 0.01)
        return Wg, Wu, Wd, Ws, Wr

    ones = torch.ones(H, dtype=torch.bfloat16, device=dev)
    layers = []
    moe = moe_weights()
    for c in range(copies):
        if c > 0 and SHARD > 1:
            moe = moe_weights()  # sharded steps are small: nothing may stay in L2 from step to step
        Wg, Wu, Wd, Ws, Wr = moe
        W_in = fill_bf16((N_IN, H), synth.W_IN, 0.02)
        W_o = fill_bf16((H, K_OUT), synth.W_O, 0.02)
        layers.append(ML.LayerWeights(gamma1=ones, W_in=W_in, W_o=W_o, gamma2=ones, W_r=Wr, Wg=Wg, Wu=Wu, Wd=Wd,
                                      Wg_s=Ws[0], Wu_s=Ws[1], Wd_s=Ws[2], k=TOPK, k_out=K_OUT))
    torch.cuda.synchronize()
    return layers


def run_ours(args, rank, local, world):
    import numpy as np
    import torch
    import moe_layers_gb300 as ML
    import synth

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    ML.build()
    h = ML.Handle(local)
    h.set_shared_sms(args.shared_sms)
    h.set_prefetch_shared(args.prefetch_shared)
    if args.l2_ahead is not None:
        h.set_l2_ahead(args.l2_ahead)
    h.set_one_token_shared(args.shared_in_routing)
    h.set_force_variant({"auto": ML.VARIANT_AUTO, "small_m": ML.VARIANT_SMALL_M,
                         "split_k": ML.VARIANT_SPLIT_K}[args.family])
    layers = build_weights(dev, layer_copies())
    if args.prefetch_next:
        # Cross-layer prefetch: while layer l routes, the next layer's input
        # projection is pulled into L2 (up to the given bytes).
        for li, L in enumerate(layers):
            nxt = layers[(li + 1) % len(layers)].W_in
            L.prefetch_next = nxt
            L.prefetch_bytes = min(int(args.prefetch_next), nxt.numel() * 2) // 16 * 16
    cws = [L.c_struct() for L in layers]
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    sweep = sorted(set([int(m) for m in args.sweep.split(",") if m] + [args.batch]))
    results = {}
    clocks = ClockSampler(local)
    clock_started = False

    for M in sweep:
        ws = h.workspace(("bench", M), ML.decode_layer_workspace_size(h, layers[0], M),
                         ("layer", M))
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

        def step(i, trace=None):
            ML.decode_layer(h, layers[i % len(layers)], hidden, trace=trace, ws=ws, _cw=cws[i % len(layers)])

        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        # Every timed pass (eager, graph, profiled) starts from the same input
        # rows, so all of them route the same K steps (the routing, hence the
        # distinct experts U and the bytes, drift as the hidden state evolves).
        hidden.copy_(host_in)
        # ---- timed: inputs resident, K steps
        if not clock_started:
            clocks.start()
            clock_started = True
            time.sleep(0.3)
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
        idx_host = idx_all.cpu().numpy()
        U = float(np.mean([len(np.unique(idx_host[i])) for i in range(K)]))
        us = us_eager
        if args.graph:
            # The same K steps captured once as a CUDA graph (one launch per step
            # sequence, no host work per step) and replayed: the GPU-bound time.
            gs = torch.cuda.Stream(device=dev)
            gs.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                for i in range(K):
                    ML.decode_layer(h, layers[i % len(layers)], hidden, trace={"idx": idx_all[i]}, ws=ws,
                                    _cw=cws[i % len(layers)],
                                    stream=gs)
            hidden.copy_(host_in)
            graph.replay()
            torch.cuda.synchronize()
            hidden.copy_(host_in)
            torch.cuda.synchronize()
            barrier(dev)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            graph.replay()
            g1.record(stream)
            torch.cuda.synchronize()
            barrier(dev)
            us = g0.elapsed_time(g1) * 1000.0 / K
            idx_host = idx_all.cpu().numpy()
            U = float(np.mean([len(np.unique(idx_host[i])) for i in range(K)]))
            del graph
        us_max = reduce_max(us, dev)
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
        # every copy.
        # The inputs of the K steps (the evolving hidden state the device-timed
        # passes saw, recorded by an untimed pass), so that e2e routes the
        # same steps as value does.
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
        kern = {}
        # batch 1: the shared expert runs inside the routing (or gate/up) and down launches
        shared_in = (None if "shared_gate_up" in prof else "front" if "moe_front" in prof else
                     "router" if args.shared_in_routing else "gate_up")
        for tag, (n, ms) in prof.items():
            avg_us = ms * 1000.0 / max(n, 1)
            kb = kernel_bytes(tag, M, U_prof, shared_in)
            kern[tag] = {"launches_per_step": n / K, "avg_us": round(avg_us, 2),
                         "GBps": round(kb / (avg_us * 1e3), 1) if kb and avg_us > 0 else None}
        results[M] = dict(M=M, us_per_step=round(us_max, 2), us_per_step_stream=round(us_eager, 2),
                          e2e_us=round(us_e2e, 2), U=round(U, 2),
                          step_bytes=int(b), weight_stream_GBps=round(b / (us_max * 1e3), 1),
                          hbm_frac=round(b / (us_max * 1e3) / peaks["hbm_gbs"], 4),
                          kernels_per_step=launches / K, gpu_launches=launches, kernels=kern)
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
                "peak_source": peaks["source"], "avg_us": dk["avg_us"]}
    out = {"metric": METRIC, "value": hl["us_per_step"], "unit": "us/step", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(hl["us_per_step"] / 1000.0, 5), "higher_is_better": False,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic: seeded random-init weights of the workload's shapes, seeded N(0,1) activations",
           "config": {"workload": WORKLOAD if E == 384 else WORKLOAD + f" (profiling variant: {E} routed experts)",
                      "weight_copies": len(layers),
                      "token_rows": ("independent" if args.verify <= 1 else
                                     f"speculative verify: groups of {args.verify} related rows, noise {args.verify_noise}"),
                      "batch": args.batch, "parallelism": "replicas" if world > 1 else "1 GPU",
                      "l2": "inputs larger than L2: each step reads >= 1.1 GB (L2 129 MB); dense weights alternate "
                            "between 2 copies; routing changes every step",
                      "weight_stream_GBps": hl["weight_stream_GBps"], "hbm_frac": hl["hbm_frac"],
                      "distinct_experts_U": hl["U"], "shared_expert_sms": {0: "auto", -1: "overlap"}.get(args.shared_sms, args.shared_sms),
                      "sweep": [{k: v for k, v in results[m].items() if k != "kernels"} for m in sweep],
                      "kernels_at_batch": hl["kernels"]},
           "weight_stream_GBps": hl["weight_stream_GBps"], "hbm_frac": hl["hbm_frac"],
           "roofline": roofline,
           "e2e": {"value": hl["e2e_us"], "unit": "us/step", "h2d_bytes_per_step": args.batch * H * 2,
                   "d2h_bytes_per_step": args.batch * H * 2},
           "gpu_launches": hl["gpu_launches"], "clocks": clk}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.batch, steps=1)
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
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time the K steps as stream launches only (default: also capture them in a CUDA graph "
                         "and report the replay time as the value)")
    ap.add_argument("--shared-sms", type=int, default=0,
                    help="SMs for the shared expert: 0 automatic share (default), -1 every SM overlapped, n fixed")
    ap.add_argument("--family", choices=("auto", "small_m", "split_k"), default="auto",
                    help="kernel family (auto: by batch and size; small_m covers batch <= 4)")
    ap.add_argument("--shared-in-routing", type=int, choices=(0, 1, 2), default=2,
                    help="batch 1: one launch of the routing and both gate/ups (2, default), the shared "
                         "expert's gate/up inside the routing launch (1) or the gate/up launch (0)")
    ap.add_argument("--l2-ahead", type=int, default=None,
                    help="bytes per CTA the small-matrix kernels keep requested into L2 ahead (default: library's)")
    ap.add_argument("--prefetch-shared", action="store_true",
                    help="at batch 1, pull the shared expert into L2 during the router phase (off: measured slower)")
    ap.add_argument("--prefetch-next", type=int, default=0,
                    help="bytes of the next layer's input projection to pull into L2 during the routing (0: none)")
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
