"""Shared helpers of the test suite: tolerance rule, device copies of seeded
inputs, and router-gap filtering of activation rows (through the oracle)."""
from __future__ import annotations

import math
from typing import Callable, List, Sequence

import numpy as np

import oracle
import synth

SEED = 0
TOL = 1e-2          # bf16 outputs: max |err| <= 1e-2 rms(oracle), beyond the output's own half-ulp
SCORE_TOL = 1e-4    # fp32 router scores, absolute
WEIGHT_TOL = 1e-5   # fp32 renormalised top-k weights, absolute
GAP = 1e-3          # minimum gap between consecutive top-(k+1) oracle scores


# ---------------------------------------------------------------------------- device copies
def dev_bf16(bits: np.ndarray, shape=None, device: str = "cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    if shape is not None:
        t = t.reshape(shape)
    return t.to(device)


def dev_f32(a: np.ndarray, device: str = "cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def host_bits(t) -> np.ndarray:
    """bf16 device tensor -> uint16 bit patterns on the host."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------- tolerance
def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def bf16_report(gpu_bits: np.ndarray, ref: np.ndarray) -> dict:
    """Compare bf16 GPU output with the fp64 oracle.

    literal  = max|gpu - ref| / rms(ref)
    floor    = max|bf16(ref) - ref| / rms(ref)  (what a correctly rounded output reaches)
    adjusted = max(|gpu - ref| - half_ulp_bf16(ref)) / rms(ref)  -> the pass criterion (<= 1e-2)
    """
    g = oracle.bf16_to_f64(gpu_bits).reshape(ref.shape)
    ref = np.asarray(ref, dtype=np.float64)
    rms = math.sqrt(float(np.mean(ref * ref))) or 1.0
    err = np.abs(g - ref)
    return dict(literal=float(err.max() / rms), floor=float(np.abs(oracle.round_bf16(ref) - ref).max() / rms),
                adjusted=float(np.max(err - half_ulp_bf16(ref)) / rms), rms=rms,
                nonfinite=int(np.count_nonzero(~np.isfinite(g))))


def ulp_bf16(ref: np.ndarray) -> np.ndarray:
    return 2.0 * half_ulp_bf16(ref)


def assert_bf16_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str = "", tol: float = TOL,
                      passthrough=None) -> dict:
    """Pass iff max(|gpu - ref| - half_ulp(ref) - passthrough) <= tol * rms(ref).

    passthrough (optional, elementwise) is a difference that enters the output
    unchanged through a residual add: for a layer output h1 + MoE, the
    measured |h1_gpu - h1_oracle| of the stored bf16 residual, which two
    correct roundings of h1 (fp32 vs fp64 sums) may leave one ulp apart."""
    r = bf16_report(gpu_bits, ref)
    if passthrough is not None:
        g = oracle.bf16_to_f64(gpu_bits).reshape(ref.shape)
        adj = np.abs(g - ref) - half_ulp_bf16(ref) - np.asarray(passthrough).reshape(ref.shape)
        r["adjusted"] = float(adj.max() / r["rms"])
    assert r["nonfinite"] == 0, f"{what}: non-finite outputs"
    assert r["adjusted"] <= tol, f"{what}: {r}"
    return r


# ---------------------------------------------------------------------------- router gap
def gap_ok(scores_row: np.ndarray, k: int, gap: float = GAP) -> bool:
    top = np.sort(scores_row)[::-1][: k + 1]
    return bool(np.all(-np.diff(top) >= gap))


def gap_rows(score_fn: Callable[[np.ndarray], np.ndarray], M: int, H: int, k: int, base: int, seed: int = SEED,
             sigma: float = 1.0, gap: float = GAP, max_attempts: int = 200):
    """Draw M activation rows (bf16 bits); row r uses attempt a = 0, 1, ...
    until the oracle's scores for it have consecutive top-(k+1) gaps >= gap.
    score_fn maps a batch of bf16-bit rows [n, H] to oracle scores [n, E].
    Returns (bits [M, H], attempts per row)."""
    bits = np.empty((M, H), dtype=np.uint16)
    attempts = [0] * M
    pending = list(range(M))
    while pending:
        cand = synth.bf16_rows(base, pending, H, seed, sigma, [attempts[r] for r in pending])
        sc = score_fn(cand)
        nxt = []
        for i, r in enumerate(pending):
            if gap_ok(sc[i], k, gap):
                bits[r] = cand[i]
            else:
                attempts[r] += 1
                if attempts[r] > max_attempts:
                    raise RuntimeError("gap rule: too many redraws")
                nxt.append(r)
        pending = nxt
    return bits, attempts


def gap_correlated_rows(score_fn: Callable[[np.ndarray], np.ndarray], M: int, H: int, k: int, base: int, group: int,
                        eps: float, seed: int = SEED, gap: float = GAP, max_attempts: int = 200):
    """As gap_rows, for a speculative-verify batch: groups of `group` related
    rows (synth.correlated_rows); a row that misses the gap rule redraws its
    own deviation (attempt counter), its group's shared row stays."""
    bits = np.empty((M, H), dtype=np.uint16)
    attempts = [0] * M
    pending = list(range(M))
    while pending:
        cand = synth.correlated_rows(base, pending, group, H, seed, eps, [attempts[r] for r in pending])
        sc = score_fn(cand)
        nxt = []
        for i, r in enumerate(pending):
            if gap_ok(sc[i], k, gap):
                bits[r] = cand[i]
            else:
                attempts[r] += 1
                if attempts[r] > max_attempts:
                    raise RuntimeError("gap rule: too many redraws")
                nxt.append(r)
        pending = nxt
    return bits, attempts


# ---------------------------------------------------------------------------- expert banks
class HostBank:
    """Host view of a seeded expert bank: regenerates expert e's weights on demand."""

    def __init__(self, E: int, H: int, I: int, seed: int = SEED, ids=(synth.W_G, synth.W_U, synth.W_D),
                 sigma: float = 0.02, cache: int = 16):
        """cache: experts whose bits are kept (a full-size expert is 88 MB), so
        that a second oracle pass over the same experts does not regenerate them."""
        self.E, self.H, self.I, self.seed, self.ids, self.sigma = E, H, I, seed, ids, sigma
        self._cache = {}
        self._cap = int(cache)

    def bits(self, e: int):
        if e not in self._cache:
            n = self.I * self.H
            g = synth.bf16(n, self.seed, self.ids[0], e * n, self.sigma).reshape(self.I, self.H)
            u = synth.bf16(n, self.seed, self.ids[1], e * n, self.sigma).reshape(self.I, self.H)
            d = synth.bf16(n, self.seed, self.ids[2], e * n, self.sigma).reshape(self.H, self.I)
            if len(self._cache) >= self._cap:
                self._cache.clear()
            self._cache[e] = (g, u, d)
        return self._cache[e]

    def __call__(self, e: int):
        return tuple(oracle.bf16_to_f64(b) for b in self.bits(int(e)))
