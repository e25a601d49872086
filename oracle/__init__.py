"""Plain fp64 CPU oracle of the MoE decode-layer hot path.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The
CUDA library never calls it and shares no code with it; the only thing both
sides share is the seeded input generator in ``synth/``.

Sources. The pages (the vLLM "Kimi K3" decode article in its Spanish and
Korean versions, and the aihirek.info summary "A vLLM ügynöki kódolással
gyorsította a Kimi K3-at") name the steps of the decode hot path but print no
formula, dtype or shape:

* Part 1 §1 "Ajustar las formas": the attention input projections run as a
  small-matrix kernel at batch 1-2 and as split-K kernels at larger batch;
* Part 1 §2 "Superposición de computación y comunicación": the attention
  output projection is fused with the residual that follows it (the
  all-reduce in between has no counterpart on one GPU);
* Part 1 §3 "Mejorar la programación de MoE": router scores, then the routed
  experts; the shared expert runs beside them;
* Part 1 §4 "Prefetching": small-batch decode is bound by weight reads.

The rules the pages leave open are taken from the workload definition and
the plainest reading, and each function below states the one it uses:
sigmoid router scores, top-8 by score (ties to the lower expert id),
weights renormalised over the eight; SwiGLU experts
``W_d (silu(W_g x) * (W_u x))``; pre-norm RMSNorm with eps 1e-6.

Every function computes its plain definition in float64 with no intermediate
rounding. Inputs stored as bf16 / fp32 are widened exactly. A library matmul
serves as the dot-product step; nothing is blocked, fused or reordered beyond
that.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
brute force on tiny inputs, exact integer cases, closed forms and invariants
(linearity, permutation of expert ids, the silu odd-part identity, scale
invariance of the norm, M-invariance of the layer).
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence, Tuple

import numpy as np

RMS_EPS = 1e-6


# ----------------------------------------------------------------------------- storage widening
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def as_f64(a) -> np.ndarray:
    """Widen a stored tensor exactly: uint16 arrays are bf16 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_to_f64(a)
    return a.astype(np.float64)


def round_bf16(a) -> np.ndarray:
    """Nearest-even rounding of float64 values to bfloat16, returned as float64.

    v = q * 2^(e-8) with q an integer of at most 8 significant bits, chosen by
    round-half-to-even (numpy rint) on the exactly scaled significand. Used
    only where the workload stores an activation as bf16 between operations.
    """
    v = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(v)                      # v = m 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                 # below 2^-126: bf16 subnormal spacing
    q = np.rint(np.ldexp(v, 8 - e))         # exact scaling, then round half to even
    return np.ldexp(q, e - 8)


# ----------------------------------------------------------------------------- dense steps
def linear(x, W) -> np.ndarray:
    """y = x W^T: the decode projection, nn.Linear layout W[N, K].

    Kimi K3 article, Part 1 §1 (attention input projections): the product is
    the same for the small-matrix and split-K kernels; only its evaluation
    differs. x[M, K], W[N, K] -> y[M, N].
    """
    x = as_f64(x)
    W = as_f64(W)
    if x.ndim != 2 or W.ndim != 2 or x.shape[1] != W.shape[1]:
        raise ValueError(f"linear: x{list(x.shape)} W{list(W.shape)}")
    return x @ W.T


def linear_residual(x, W, r) -> np.ndarray:
    """out = r + x W^T: out-projection fused with the residual add.

    Kimi K3 article, Part 1 §2: the attention output projection is fused with
    the residual computation that follows it.
    """
    return as_f64(r) + linear(x, W)


def rmsnorm(x, gamma, eps: float = RMS_EPS) -> np.ndarray:
    """a = x / sqrt(mean(x^2) + eps) * gamma, per row.

    Not named on the pages; the decode layer of the workload applies it before
    the attention input projection and before the MoE layer (pre-norm).
    """
    x = as_f64(x)
    g = as_f64(gamma)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


# ----------------------------------------------------------------------------- router
def sigmoid(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):  # exp(-z) = inf for z << 0 gives the exact limit 0
        return 1.0 / (1.0 + np.exp(-z))


def router_scores(x, Wr) -> Tuple[np.ndarray, np.ndarray]:
    """Router logits x W_r^T and sigmoid scores.

    Kimi K3 article, Part 1 §3 (router scores before the experts run). The
    pages give no formula; the workload fixes sigmoid scoring of fp32 router
    weights W_r[E, H]. Returns (logits[M, E], scores[M, E]).
    """
    logits = linear(x, Wr)
    return logits, sigmoid(logits)


def topk(scores, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Per token: the k largest scores, highest first, ties to the lower id.

    Weights are the selected scores divided by their sum (renormalised top-k),
    with no bias, grouping or extra scale: the workload's rule read plainly.
    Returns (idx int32 [M, k], w float64 [M, k]).
    """
    s = np.asarray(scores, dtype=np.float64)
    M, E = s.shape
    if not 1 <= k <= E:
        raise ValueError("topk: k out of range")
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float64)
    ids = np.arange(E)
    for t in range(M):
        order = np.lexsort((ids, -s[t]))  # primary: score descending; then id ascending
        sel = order[:k]
        idx[t] = sel
        w[t] = s[t, sel] / np.sum(s[t, sel])
    return idx, w


# ----------------------------------------------------------------------------- experts
def silu(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def swiglu_expert(x, Wg, Wu, Wd) -> np.ndarray:
    """One SwiGLU expert on rows x[c, H]: W_d (silu(W_g x) * (W_u x)).

    Kimi K3 article, Part 1 §3 (routed and shared experts); the expert form is
    the workload's (gate/up H -> I, down I -> H).
    """
    x = as_f64(x)
    g = linear(x, Wg)
    u = linear(x, Wu)
    return linear(silu(g) * u, Wd)


ExpertFn = Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray]]


def moe(x, idx, w, expert: ExpertFn, shared: Optional[Sequence] = None, residual=None,
        tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """MoE layer output for the given routing.

    out_t = [r_t +] sum_j w_tj E_{idx_tj}(x_t) [+ S(x_t)], where E_e is routed
    expert e (its weights from ``expert(e)``), S the shared expert (weight 1).
    Kimi K3 article, Part 1 §3: routed experts over the selected ids, shared
    expert alongside. ``tokens`` restricts the computation to some rows (the
    result then has one row per listed token).
    """
    x = as_f64(x)
    idx = np.asarray(idx)
    w = np.asarray(w, dtype=np.float64)
    rows = list(range(x.shape[0])) if tokens is None else [int(t) for t in tokens]
    out = np.zeros((len(rows), x.shape[1]), dtype=np.float64)
    pos = {t: i for i, t in enumerate(rows)}
    for e in sorted(set(int(v) for t in rows for v in idx[t])):
        sel = [(t, j) for t in rows for j in range(idx.shape[1]) if int(idx[t, j]) == e]
        Wg, Wu, Wd = expert(e)
        ye = swiglu_expert(x[[t for t, _ in sel]], Wg, Wu, Wd)
        for (t, j), y in zip(sel, ye):
            out[pos[t]] += w[t, j] * y
    if shared is not None:
        out += swiglu_expert(x[rows], *shared)
    if residual is not None:
        out += as_f64(residual)[rows]
    return out


# ----------------------------------------------------------------------------- MoE layer
def moe_layer(x, gamma, Wr, k: int, expert: ExpertFn, shared: Optional[Sequence] = None, residual=None,
              eps: float = RMS_EPS, tokens: Optional[Sequence[int]] = None, storage: str = "bf16"):
    """The MoE layer as one step: optional RMSNorm, router, top-k, experts.

    b = RMSNorm(x; gamma) (x itself when gamma is None); logits, scores =
    router(b); idx, w = top-k; out = [residual +] moe(b, idx, w) [+ S(b)].
    Kimi K3 article, Part 1 §3 (router scores, then the routed experts and the
    shared expert). With ``storage`` "bf16" (default) the normalised rows b,
    a stored activation, are rounded to bf16 before the router and the
    experts read them; "f64" rounds nothing.

    Returns a dict with b, logits, scores, idx, w and ``out`` (unrounded),
    and ``b_unrounded`` (b before its storage rounding); ``tokens`` limits all
    of it to some rows.
    """
    if storage not in ("bf16", "f64"):
        raise ValueError("storage must be 'bf16' or 'f64'")
    st = round_bf16 if storage == "bf16" else (lambda v: v)
    x = as_f64(x)
    rows = list(range(x.shape[0])) if tokens is None else [int(t) for t in tokens]
    x = x[rows]
    b_unrounded = rmsnorm(x, gamma, eps) if gamma is not None else x
    b = st(b_unrounded)
    logits, scores = router_scores(b, Wr)
    idx, w = topk(scores, k)
    out = moe(b, idx, w, expert, shared)
    if residual is not None:
        out = out + as_f64(residual)[rows]
    return dict(b=b, b_unrounded=b_unrounded, logits=logits, scores=scores, idx=idx, w=w, out=out)


# ----------------------------------------------------------------------------- decode layer
def decode_layer(h, gamma1, W_in, W_o, gamma2, Wr, k: int, expert: ExpertFn, shared: Optional[Sequence],
                 k_out: Optional[int] = None, eps: float = RMS_EPS, tokens: Optional[Sequence[int]] = None,
                 storage: str = "bf16"):
    """One decode layer: RMSNorm -> input projection -> out-projection + residual
    -> RMSNorm -> MoE (+ residual).

    The pages omit the attention core between the input projection and the
    out-projection; the plainest reading that keeps the data dependency is to
    feed the first ``k_out`` columns of the input projection (K of the
    out-projection) straight to the out-projection. The MoE block is pre-norm
    with its own residual: out = h1 + MoE(RMSNorm(h1)) (``moe_layer`` with
    gamma2 and the residual h1).

    ``storage``: the layer's activations are bf16 tensors, so with "bf16"
    (default) the output of each operation (a, y_in, h1, b) is rounded to bf16
    before the next operation reads it; each operation itself is exact fp64.
    This keeps the routing decision (an arg-max over scores) in the precision
    the layer defines. "f64" rounds nothing.

    Returns a dict with the intermediates (a, y_in, h1, b, logits, scores,
    idx, w), the output ``out`` (unrounded), and ``unrounded``: the values of
    a, y_in, h1 and b before their storage rounding (each the exact result of
    its operation on the stored inputs); ``tokens`` limits all of it to some
    rows.
    """
    if storage not in ("bf16", "f64"):
        raise ValueError("storage must be 'bf16' or 'f64'")
    st = round_bf16 if storage == "bf16" else (lambda v: v)
    h = as_f64(h)
    rows = list(range(h.shape[0])) if tokens is None else [int(t) for t in tokens]
    h = h[rows]
    W_o64 = as_f64(W_o)
    k_out = W_o64.shape[1] if k_out is None else k_out
    a_x = rmsnorm(h, gamma1, eps)
    a = st(a_x)
    y_x = linear(a, W_in)
    y_in = st(y_x)
    h1_x = linear_residual(y_in[:, :k_out], W_o64, h)
    h1 = st(h1_x)
    m = moe_layer(h1, gamma2, Wr, k, expert, shared, residual=h1, eps=eps, storage=storage)
    return dict(a=a, y_in=y_in, h1=h1, b=m["b"], logits=m["logits"], scores=m["scores"], idx=m["idx"], w=m["w"],
                out=m["out"], unrounded=dict(a=a_x, y_in=y_x, h1=h1_x, b=m["b_unrounded"]))
