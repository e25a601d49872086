"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each check below is written so that a plausible mistake in the oracle (a
transposed operand, a dropped term, a wrong sign or index, sigmoid in place
of silu, swapped gate/up, a reversed tie-break, a missing renormalisation)
fails at least one of them; ``test_mutations_are_caught`` plants each such
mistake in the oracle (on the CPU) and confirms that a pin fails.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LN3 = math.log(3.0)
LN9 = math.log(9.0)


def _val(s) -> float:
    """Parse the golden fixtures' tiny expression language: a/b, lnN, products."""
    s = str(s).strip()
    neg = s.startswith("-")
    if neg:
        s = s[1:]
    out = 1.0
    for part in s.split("*"):
        if part.startswith("ln"):
            out *= math.log(float(part[2:]))
        else:
            out *= float(Fraction(part))
    return -out if neg else out


def _arr(a):
    return np.array([[_val(v) for v in row] for row in a]) if isinstance(a[0], list) else np.array([_val(v) for v in a])


def _bf16_bits(values):
    """bf16 bit patterns of values that are exactly representable in bf16."""
    v = np.asarray(values, dtype=np.float32)
    bits = v.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


# ============================================================================ linear
def pin_linear_bruteforce(o):
    rng = np.random.default_rng(1)
    for M, K, N in [(1, 1, 1), (2, 5, 3), (3, 64, 16), (1, 17, 9)]:
        x = rng.standard_normal((M, K))
        W = rng.standard_normal((N, K))
        y = o.linear(x, W)
        assert y.shape == (M, N)
        for m in range(M):
            for n in range(N):
                ref = math.fsum(x[m, k] * W[n, k] for k in range(K))
                assert abs(y[m, n] - ref) <= 1e-12 * (1 + abs(ref))


def pin_linear_integer_exact(o):
    # Small integers times 2^-4 are exact in bf16; their products and sums are
    # exact in float64, so the result must equal the integer arithmetic bit for bit.
    rng = np.random.default_rng(2)
    M, K, N = 3, 48, 11
    xi = rng.integers(-8, 9, size=(M, K))
    wi = rng.integers(-8, 9, size=(N, K))
    x = _bf16_bits(xi / 16.0)
    W = _bf16_bits(wi / 16.0)
    y = o.linear(x, W)
    for m in range(M):
        for n in range(N):
            exact = Fraction(int(sum(int(xi[m, k]) * int(wi[n, k]) for k in range(K))), 256)
            assert Fraction(y[m, n]) == exact


def pin_linear_orientation(o):
    # A single nonzero weight at (n0, k0) must route input column k0 to output column n0.
    M, K, N = 2, 6, 6
    x = np.arange(1.0, 1.0 + M * K).reshape(M, K)
    W = np.zeros((N, K))
    W[4, 1] = 3.0
    y = o.linear(x, W)
    expect = np.zeros((M, N))
    expect[:, 4] = 3.0 * x[:, 1]
    assert np.array_equal(y, expect)


def pin_linear_linearity(o):
    rng = np.random.default_rng(3)
    a, b = rng.standard_normal((2, 4, 40))
    W1, W2 = rng.standard_normal((2, 7, 40))
    lhs = o.linear(a + b, W1)
    rhs = o.linear(a, W1) + o.linear(b, W1)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    lhs = o.linear(a, W1 + W2)
    rhs = o.linear(a, W1) + o.linear(a, W2)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


def pin_linear_residual(o):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 8))
    W = rng.standard_normal((5, 8))
    r = rng.standard_normal((3, 5))
    assert np.array_equal(o.linear_residual(x, np.zeros_like(W), r), r)
    assert np.allclose(o.linear_residual(x, W, np.zeros_like(r)), o.linear(x, W), rtol=0, atol=0)
    # residual enters with a plus sign and weight one
    assert np.allclose(o.linear_residual(x, W, r) - o.linear(x, W), r, rtol=1e-14, atol=1e-14)


# ============================================================================ rmsnorm
def pin_rmsnorm(o):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 33))
    g = np.ones(33)
    a = o.rmsnorm(x, g, eps=0.0)
    # with unit gain and eps = 0 every output row has mean square exactly one
    assert np.allclose(np.mean(a * a, axis=1), 1.0, rtol=1e-13)
    # scale invariance (c > 0) and sign equivariance
    assert np.allclose(o.rmsnorm(7.5 * x, g, eps=0.0), a, rtol=1e-13)
    assert np.allclose(o.rmsnorm(-x, g, eps=0.0), -a, rtol=1e-13)
    # a constant row c maps to the gain
    gam = 1.0 + 0.1 * rng.standard_normal(33)
    assert np.allclose(o.rmsnorm(np.full((1, 33), 2.5), gam, eps=0.0), gam[None, :], rtol=1e-14)
    # +-1 rows are fixed points with unit gain
    pm = np.array([[1.0, -1.0, 1.0, -1.0]])
    assert np.array_equal(o.rmsnorm(pm, np.ones(4), eps=0.0), pm)
    # eps enters under the square root, added to the mean square: for x = 0 the output is 0,
    # and for a row of ones with eps = 3 the scale is 1/sqrt(1 + 3) = 1/2
    assert np.allclose(o.rmsnorm(np.ones((1, 8)), np.ones(8), eps=3.0), 0.5, rtol=1e-15)


# ============================================================================ router
def _golden_router():
    with open(os.path.join(GOLDEN, "router_tiny.json")) as f:
        return json.load(f)


def pin_router_golden(o):
    gd = _golden_router()
    x = np.array([gd["x"]])
    Wr = _arr(gd["Wr"])
    logits, scores = o.router_scores(x, Wr)
    assert np.allclose(scores[0], _arr(gd["scores"]), rtol=0, atol=1e-14)
    for case in gd["cases"]:
        idx, w = o.topk(scores, case["k"])
        assert idx[0].tolist() == case["idx"]
        assert np.allclose(w[0], _arr(case["w"]), rtol=0, atol=1e-14)
    tc = gd["tie_case"]
    _, s2 = o.router_scores(x, _arr(tc["Wr"]))
    idx, w = o.topk(s2, tc["k"])
    assert idx[0].tolist() == tc["idx"]
    assert np.allclose(w[0], _arr(tc["w"]), rtol=0, atol=1e-14)


def pin_router_properties(o):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, 24))
    Wr = 0.3 * rng.standard_normal((16, 24))
    logits, scores = o.router_scores(x, Wr)
    assert np.all((scores > 0) & (scores < 1))
    # scores are a monotone function of logits: the same top-k either way
    idx_s, w = o.topk(scores, 4)
    idx_l = np.argsort(-logits, axis=1, kind="stable")[:, :4]
    assert np.array_equal(idx_s, idx_l)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)  # highest first
    # zero router: all scores 1/2, ids 0..k-1, equal weights
    _, s0 = o.router_scores(x, np.zeros_like(Wr))
    assert np.all(s0 == 0.5)
    i0, w0 = o.topk(s0, 8)
    assert np.array_equal(i0, np.tile(np.arange(8), (5, 1)))
    assert np.allclose(w0, 1.0 / 8, rtol=1e-15)
    # sigmoid symmetry
    z = np.linspace(-9, 9, 37)
    assert np.allclose(o.sigmoid(z) + o.sigmoid(-z), 1.0, rtol=1e-15)


# ============================================================================ experts
def _golden_swiglu():
    with open(os.path.join(GOLDEN, "swiglu_tiny.json")) as f:
        return json.load(f)


def pin_swiglu_golden(o):
    for c in _golden_swiglu()["cases"]:
        out = o.swiglu_expert(_arr(c["x"])[None, :], _arr(c["Wg"]), _arr(c["Wu"]), _arr(c["Wd"]))
        assert np.allclose(out[0], _arr(c["out"]), rtol=0, atol=1e-14)


def pin_swiglu_odd_part(o):
    # silu(z) - silu(-z) = z, so E(Wg) - E(-Wg) = Wd ((Wg x) * (Wu x)): a bilinear
    # quantity that a library matmul gives directly. It fails for sigmoid in place
    # of silu and for gate/up swapped.
    rng = np.random.default_rng(7)
    x = rng.standard_normal((3, 20))
    Wg, Wu = rng.standard_normal((2, 12, 20))
    Wd = rng.standard_normal((20, 12))
    diff = o.swiglu_expert(x, Wg, Wu, Wd) - o.swiglu_expert(x, -Wg, Wu, Wd)
    expect = ((x @ Wg.T) * (x @ Wu.T)) @ Wd.T
    assert np.allclose(diff, expect, rtol=1e-11, atol=1e-11)
    # linear in Wu and in Wd; zero gate gives zero
    e1 = o.swiglu_expert(x, Wg, Wu, Wd)
    assert np.allclose(o.swiglu_expert(x, Wg, 2.5 * Wu, Wd), 2.5 * e1, rtol=1e-12, atol=1e-12)
    assert np.allclose(o.swiglu_expert(x, Wg, Wu, -3.0 * Wd), -3.0 * e1, rtol=1e-12, atol=1e-12)
    assert np.array_equal(o.swiglu_expert(x, np.zeros_like(Wg), Wu, Wd), np.zeros((3, 20)))


def _bank(rng, E, H, I):
    Wg = rng.standard_normal((E, I, H)) * 0.3
    Wu = rng.standard_normal((E, I, H)) * 0.3
    Wd = rng.standard_normal((E, H, I)) * 0.3
    return Wg, Wu, Wd


def pin_moe_properties(o):
    rng = np.random.default_rng(8)
    M, H, I, E, k = 5, 16, 8, 10, 3
    x = rng.standard_normal((M, H))
    Wr = rng.standard_normal((E, H))
    Wg, Wu, Wd = _bank(rng, E, H, I)
    Ws = tuple(a[0] for a in _bank(rng, 1, H, I))
    ex = lambda e: (Wg[e], Wu[e], Wd[e])
    _, s = o.router_scores(x, Wr)
    idx, w = o.topk(s, k)
    base = o.moe(x, idx, w, ex, Ws)
    # brute force over (token, slot)
    for t in range(M):
        ref = sum(w[t, j] * o.swiglu_expert(x[t:t + 1], *ex(int(idx[t, j])))[0] for j in range(k))
        ref = ref + o.swiglu_expert(x[t:t + 1], *Ws)[0]
        assert np.allclose(base[t], ref, rtol=1e-12, atol=1e-12)
    # permuting expert ids (router rows and bank together) permutes idx, leaves the output
    perm = rng.permutation(E)
    inv = np.argsort(perm)
    _, sp = o.router_scores(x, Wr[perm])
    idxp, wp = o.topk(sp, k)
    assert np.array_equal(perm[idxp], idx)
    outp = o.moe(x, idxp, wp, lambda e: ex(int(perm[e])), Ws)
    assert np.allclose(outp, base, rtol=1e-12, atol=1e-12)
    # identical experts: the routed part equals that expert (weights sum to one)
    same = lambda e: ex(0)
    routed = o.moe(x, idx, w, same, None)
    assert np.allclose(routed, o.swiglu_expert(x, *ex(0)), rtol=1e-12, atol=1e-12)
    # k = 1: routed part is the argmax expert alone
    i1, w1 = o.topk(s, 1)
    assert np.all(w1 == 1.0)
    r1 = o.moe(x, i1, w1, ex, None)
    for t in range(M):
        assert int(i1[t, 0]) == int(np.argmax(s[t]))
        assert np.allclose(r1[t], o.swiglu_expert(x[t:t + 1], *ex(int(i1[t, 0])))[0], rtol=1e-12)
    # gates far below zero switch routed experts off: only the shared expert remains
    xp = np.abs(x) + 0.1  # positive rows, so a negative gate matrix gives gates <= -1.6e2
    _, sp_ = o.router_scores(xp, Wr)
    ip, wp_ = o.topk(sp_, k)
    off = lambda e: (-100.0 * np.ones_like(Wg[e]), Wu[e], Wd[e])
    out_off = o.moe(xp, ip, wp_, off, Ws)
    assert np.allclose(out_off, o.swiglu_expert(xp, *Ws), rtol=1e-12, atol=1e-12)
    # residual adds with weight one; token subset matches the full result
    r = rng.standard_normal((M, H))
    assert np.allclose(o.moe(x, idx, w, ex, Ws, residual=r) - base, r, rtol=1e-12, atol=1e-12)
    sub = o.moe(x, idx, w, ex, Ws, tokens=[4, 1])
    assert np.allclose(sub, base[[4, 1]], rtol=1e-13, atol=1e-13)


# ============================================================================ bf16 storage
def _exact_bf16(v: float) -> float:
    """Nearest-even bf16 value of v by exact rational arithmetic (independent of the oracle)."""
    if v == 0.0:
        return 0.0
    a = Fraction(abs(v))
    e = 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = a / Fraction(2) ** (e - 7)
    fl = math.floor(q)
    r = q - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    out = float(fl * Fraction(2) ** (e - 7))
    return -out if v < 0 else out


def pin_round_bf16(o):
    rng = np.random.default_rng(10)
    vals = np.concatenate([rng.standard_normal(2000), rng.standard_normal(300) * 1e-3, rng.standard_normal(300) * 1e4,
                           np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 2 ** -130, 0.0, 255.5])])
    got = o.round_bf16(vals)
    for v, g in zip(vals, got):
        assert g == _exact_bf16(float(v)), (v, g)
    # idempotent, and exact for representable values
    assert np.array_equal(o.round_bf16(got), got)


# ============================================================================ decode layer
def _tiny_layer(rng, H=16, N_in=24, K_out=12, E=12, k=3, I=8):
    W_in = rng.standard_normal((N_in, H)) * 0.4
    W_o = rng.standard_normal((H, K_out)) * 0.4
    Wr = rng.standard_normal((E, H))
    Wg, Wu, Wd = _bank(rng, E, H, I)
    Ws = tuple(a[0] for a in _bank(rng, 1, H, I))
    g1 = 1.0 + 0.1 * rng.standard_normal(H)
    g2 = 1.0 + 0.1 * rng.standard_normal(H)
    return dict(gamma1=g1, W_in=W_in, W_o=W_o, gamma2=g2, Wr=Wr, k=k,
                expert=lambda e: (Wg[e], Wu[e], Wd[e]), shared=Ws)


def pin_decode_layer(o):
    rng = np.random.default_rng(9)
    L = _tiny_layer(rng)
    h = rng.standard_normal((4, 16))
    # bf16 storage rounds each operation's output, and only that
    fb = o.decode_layer(h, **L)
    a = o.round_bf16(o.rmsnorm(h, L["gamma1"]))
    y = o.round_bf16(o.linear(a, L["W_in"]))
    h1 = o.round_bf16(h + o.linear(y[:, :12], L["W_o"]))
    b = o.round_bf16(o.rmsnorm(h1, L["gamma2"]))
    _, s = o.router_scores(b, L["Wr"])
    idx, w = o.topk(s, L["k"])
    assert np.array_equal(fb["idx"], idx)
    assert np.allclose(fb["out"], h1 + o.moe(b, idx, w, L["expert"], L["shared"]), rtol=1e-13, atol=1e-13)
    full = o.decode_layer(h, storage="f64", **L)
    # composition of the separately pinned stages
    a = o.rmsnorm(h, L["gamma1"])
    y = o.linear(a, L["W_in"])
    h1 = h + o.linear(y[:, :12], L["W_o"])
    b = o.rmsnorm(h1, L["gamma2"])
    _, s = o.router_scores(b, L["Wr"])
    idx, w = o.topk(s, L["k"])
    out = h1 + o.moe(b, idx, w, L["expert"], L["shared"])
    assert np.array_equal(full["idx"], idx)
    assert np.allclose(full["out"], out, rtol=1e-13, atol=1e-13)
    # M-invariance: each row of a batch equals the batch-of-one result on that row
    for t in range(4):
        one = o.decode_layer(h[t:t + 1], storage="f64", **L)
        assert np.array_equal(one["idx"][0], full["idx"][t])
        assert np.allclose(one["out"][0], full["out"][t], rtol=1e-12, atol=1e-12)
    sub = o.decode_layer(h, tokens=[3, 0], storage="f64", **L)
    assert np.allclose(sub["out"], full["out"][[3, 0]], rtol=1e-12, atol=1e-12)


def pin_moe_layer(o):
    rng = np.random.default_rng(11)
    E, H, I, k = 10, 16, 8, 3
    Wg, Wu, Wd = _bank(rng, E, H, I)
    Ws = tuple(a[0] for a in _bank(rng, 1, H, I))
    Wr = rng.standard_normal((E, H))
    ex = lambda e: (Wg[e], Wu[e], Wd[e])
    x = rng.standard_normal((5, H))
    r = rng.standard_normal((5, H))
    g = 1.0 + 0.1 * rng.standard_normal(H)
    # without gains the rows are read as they are
    plain = o.moe_layer(x, None, Wr, k, ex, Ws, storage="f64")
    assert np.array_equal(plain["b"], x)
    # the residual enters once, unchanged
    with_r = o.moe_layer(x, None, Wr, k, ex, Ws, residual=r, storage="f64")
    assert np.allclose(with_r["out"] - plain["out"], r, rtol=0, atol=1e-12)
    # with gains the rows are normalised first: invariant under a positive row scale (eps 0)
    a = o.moe_layer(x, g, Wr, k, ex, Ws, eps=0.0, storage="f64")
    b = o.moe_layer(x * np.array([[0.5], [2.0], [3.0], [0.25], [7.0]]), g, Wr, k, ex, Ws, eps=0.0, storage="f64")
    assert np.array_equal(a["idx"], b["idx"])
    assert np.allclose(a["out"], b["out"], rtol=1e-9, atol=1e-9)
    assert not np.allclose(a["out"], plain["out"], rtol=1e-3, atol=1e-3)
    # identical experts: the renormalised weights sum to one, so the routed part is that expert
    same = lambda e: (Wg[0], Wu[0], Wd[0])
    one = o.moe_layer(x, None, Wr, k, same, None, storage="f64")
    assert np.allclose(one["out"], o.swiglu_expert(x, Wg[0], Wu[0], Wd[0]), rtol=1e-12, atol=1e-12)
    # bf16 storage rounds the normalised rows once; the unrounded value is kept beside them
    st = o.moe_layer(x, g, Wr, k, ex, Ws, eps=0.0)
    assert np.array_equal(st["b"], o.round_bf16(st["b_unrounded"]))
    assert np.array_equal(st["b_unrounded"], a["b"])
    # the decode layer's stored activations and their unrounded values
    L = _tiny_layer(rng)
    d = o.decode_layer(rng.standard_normal((3, 16)), **L)
    for key in ("a", "y_in", "h1", "b"):
        assert np.array_equal(d[key], o.round_bf16(d["unrounded"][key])), key


PINS = [pin_linear_bruteforce, pin_linear_integer_exact, pin_linear_orientation, pin_linear_linearity,
        pin_linear_residual, pin_rmsnorm, pin_router_golden, pin_router_properties, pin_swiglu_golden,
        pin_swiglu_odd_part, pin_moe_properties, pin_round_bf16, pin_decode_layer, pin_moe_layer]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle)


# ============================================================================ planted mistakes
def _mut_linear_transposed(mp):
    orig = oracle.linear
    mp.setattr(oracle, "linear", lambda x, W: orig(x, oracle.as_f64(W).T) if oracle.as_f64(W).shape[0] == oracle.as_f64(W).shape[1] else orig(x, W))


def _mut_linear_dropped_term(mp):
    orig = oracle.linear
    mp.setattr(oracle, "linear", lambda x, W: orig(oracle.as_f64(x)[:, :-1], oracle.as_f64(W)[:, :-1]) if oracle.as_f64(x).shape[1] > 1 else orig(x, W))


def _mut_residual_sign(mp):
    mp.setattr(oracle, "linear_residual", lambda x, W, r: oracle.linear(x, W) - oracle.as_f64(r))


def _mut_rms_sum(mp):
    mp.setattr(oracle, "rmsnorm", lambda x, g, eps=oracle.RMS_EPS: oracle.as_f64(x) / np.sqrt(np.sum(oracle.as_f64(x) ** 2, axis=-1, keepdims=True) + eps) * oracle.as_f64(g))


def _mut_rms_eps_outside(mp):
    mp.setattr(oracle, "rmsnorm", lambda x, g, eps=oracle.RMS_EPS: oracle.as_f64(x) / (np.sqrt(np.mean(oracle.as_f64(x) ** 2, axis=-1, keepdims=True)) + eps) * oracle.as_f64(g))


def _mut_sigmoid_sign(mp):
    mp.setattr(oracle, "sigmoid", lambda z: 1.0 / (1.0 + np.exp(np.asarray(z, dtype=np.float64))))


def _mut_softmax_scores(mp):
    def rs(x, Wr):
        lg = oracle.linear(x, Wr)
        e = np.exp(lg - lg.max(axis=1, keepdims=True))
        return lg, e / e.sum(axis=1, keepdims=True)
    mp.setattr(oracle, "router_scores", rs)


def _mut_tie_high_id(mp):
    def tk(scores, k):
        s = np.asarray(scores, dtype=np.float64)
        idx = np.array([np.lexsort((-np.arange(s.shape[1]), -row))[:k] for row in s], dtype=np.int32)
        w = np.take_along_axis(s, idx, 1)
        return idx, w / w.sum(axis=1, keepdims=True)
    mp.setattr(oracle, "topk", tk)


def _mut_no_renorm(mp):
    orig = oracle.topk
    def tk(scores, k):
        idx, _ = orig(scores, k)
        return idx, np.take_along_axis(np.asarray(scores, dtype=np.float64), idx.astype(np.int64), 1)
    mp.setattr(oracle, "topk", tk)


def _mut_silu_as_sigmoid(mp):
    mp.setattr(oracle, "silu", lambda z: oracle.sigmoid(z))


def _mut_gate_up_swapped(mp):
    mp.setattr(oracle, "swiglu_expert", lambda x, Wg, Wu, Wd: oracle.linear(oracle.silu(oracle.linear(x, Wu)) * oracle.linear(x, Wg), Wd))


def _mut_moe_unweighted(mp):
    orig = oracle.moe
    mp.setattr(oracle, "moe", lambda x, idx, w, expert, shared=None, residual=None, tokens=None:
               orig(x, idx, np.ones_like(np.asarray(w, dtype=np.float64)), expert, shared, residual, tokens))


def _mut_moe_no_shared(mp):
    orig = oracle.moe
    mp.setattr(oracle, "moe", lambda x, idx, w, expert, shared=None, residual=None, tokens=None:
               orig(x, idx, w, expert, None, residual, tokens))


def _mut_layer_no_moe_residual(mp):
    orig = oracle.decode_layer
    def dl(*a, **kw):
        d = orig(*a, **kw)
        d["out"] = d["out"] - d["h1"]
        return d
    mp.setattr(oracle, "decode_layer", dl)


def _mut_moe_layer_always_normalises(mp):
    orig = oracle.moe_layer
    mp.setattr(oracle, "moe_layer", lambda x, gamma, *a, **kw: orig(
        x, np.ones(np.asarray(x).shape[1]) if gamma is None else gamma, *a, **kw))


def _mut_round_half_up(mp):
    mp.setattr(oracle, "round_bf16", lambda a: (lambda v, e: np.ldexp(np.floor(np.ldexp(v, 8 - e) + 0.5), e - 8))(
        np.asarray(a, dtype=np.float64), np.maximum(np.frexp(np.asarray(a, dtype=np.float64))[1], -125)))


MUTATIONS = [_mut_round_half_up, _mut_linear_transposed, _mut_linear_dropped_term, _mut_residual_sign, _mut_rms_sum,
             _mut_rms_eps_outside, _mut_sigmoid_sign, _mut_softmax_scores, _mut_tie_high_id, _mut_no_renorm,
             _mut_silu_as_sigmoid, _mut_gate_up_swapped, _mut_moe_unweighted, _mut_moe_no_shared,
             _mut_layer_no_moe_residual, _mut_moe_layer_always_normalises]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=[m.__name__[5:] for m in MUTATIONS])
def test_mutations_are_caught(mutate, monkeypatch):
    mutate(monkeypatch)
    failed = []
    for pin in PINS:
        try:
            pin(oracle)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutate.__name__}"
