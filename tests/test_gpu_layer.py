"""GPU parity of the whole decode layer (decode_layer) against the oracle:
indices bit-exact (router inputs drawn with a 1e-3 top-(k+1) gap), h1 and the
layer output within the bf16 tolerance."""
import numpy as np
import pytest

import oracle
import synth
from _util import (SCORE_TOL, SEED, WEIGHT_TOL, HostBank, assert_bf16_close, dev_bf16, dev_f32, gap_correlated_rows,
                   gap_rows, host_bits, ulp_bf16)
from conftest import E_FULL, H_FULL, I_FULL, K_FULL, K_OUT_FULL, N_IN_FULL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import torch
    import moe_layers_gb300 as M
    assert torch.cuda.is_available()
    M.build()
    with M.Handle(0) as hd:
        yield hd


def _bits(a):
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


class Layer:
    """Host (bits) and device copies of one decode layer's dense weights."""

    def __init__(self, H, N_in, K_out, E, I, k, base, gamma_noise=True, sigma=0.02, sr=0.01):
        self.H, self.N_in, self.K_out, self.E, self.I, self.k = H, N_in, K_out, E, I, k
        if gamma_noise:
            g1 = oracle.round_bf16(1.0 + oracle.bf16_to_f64(synth.bf16(H, SEED, base, 0, 0.1)))
            g2 = oracle.round_bf16(1.0 + oracle.bf16_to_f64(synth.bf16(H, SEED, base + 1, 0, 0.1)))
        else:
            g1 = g2 = np.ones(H)
        self.g1, self.g2 = _bits(g1), _bits(g2)
        self.W_in = synth.bf16(N_in * H, SEED, base + 2, 0, sigma).reshape(N_in, H)
        self.W_o = synth.bf16(H * K_out, SEED, base + 3, 0, sigma).reshape(H, K_out)
        self.Wr = synth.f32(E * H, SEED, base + 4, 0, sr).reshape(E, H)
        self.W_in64 = oracle.bf16_to_f64(self.W_in)
        self.W_o64 = oracle.bf16_to_f64(self.W_o)

    def scores(self, rows):
        a = oracle.round_bf16(oracle.rmsnorm(rows, self.g1))
        y = oracle.round_bf16(oracle.linear(a, self.W_in64))
        h1 = oracle.round_bf16(oracle.linear_residual(y[:, :self.K_out], self.W_o64, rows))
        b = oracle.round_bf16(oracle.rmsnorm(h1, self.g2))
        return oracle.router_scores(b, self.Wr)[1]

    def oracle(self, hbits, expert, shared, tokens=None):
        return oracle.decode_layer(hbits, self.g1, self.W_in64, self.W_o64, self.g2, self.Wr, self.k, expert,
                                   shared, k_out=self.K_out, tokens=tokens)

    def device(self, Wg, Wu, Wd, shared):
        import moe_layers_gb300 as ML
        return ML.LayerWeights(gamma1=dev_bf16(self.g1, (self.H,)), W_in=dev_bf16(self.W_in, self.W_in.shape),
                               W_o=dev_bf16(self.W_o, self.W_o.shape), gamma2=dev_bf16(self.g2, (self.H,)),
                               W_r=dev_f32(self.Wr), Wg=Wg, Wu=Wu, Wd=Wd,
                               Wg_s=None if shared is None else shared[0],
                               Wu_s=None if shared is None else shared[1],
                               Wd_s=None if shared is None else shared[2], k=self.k, k_out=self.K_out)


def _run(h, L, dev_w, hbits):
    import moe_layers_gb300 as ML
    M = hbits.shape[0]
    hid = dev_bf16(hbits, hbits.shape)
    tr = ML.decode_layer(h, dev_w, hid, trace=True)
    return hid, tr


@pytest.mark.parametrize("M,shared", [(1, True), (2, False), (3, True), (16, True), (64, True)])
def test_layer_small(h, M, shared):
    H, N_in, K_out, E, I, k = 256, 520, 384, 32, 128, 4
    L = Layer(H, N_in, K_out, E, I, k, base=6000 + M)
    n = E * I * H
    g = synth.bf16(n, SEED, 6100, 0, 0.05).reshape(E, I, H)
    u = synth.bf16(n, SEED, 6101, 0, 0.05).reshape(E, I, H)
    d = synth.bf16(n, SEED, 6102, 0, 0.05).reshape(E, H, I)
    sh = None
    if shared:
        sh = (synth.bf16(I * H, SEED, 6103, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 6104, 0, 0.05).reshape(I, H),
              synth.bf16(H * I, SEED, 6105, 0, 0.05).reshape(H, I))
    hbits, _ = gap_rows(L.scores, M, H, k, base=6200 + M)
    dev_w = L.device(dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                     None if sh is None else tuple(dev_bf16(a, a.shape) for a in sh))
    hid, tr = _run(h, L, dev_w, hbits)
    ex = lambda e: (g[e], u[e], d[e])
    ref = L.oracle(hbits, ex, sh)
    _check_layer(tr, hid, ref, slice(None), f"layer M={M}", L, ex, sh)


@pytest.mark.parametrize("front", [True, False])
@pytest.mark.parametrize("H,E,k,shared", [(1152, 37, 5, True), (1152, 37, 5, False), (256, 9, 8, True),
                                          (2048, 300, 8, True)])
def test_layer_one_token_shapes(h, H, E, k, shared, front):
    """One token: the fused RMSNorm / router / top-k / routing-table launch on
    a router row split into a full and a ragged chunk (H = 1152), with a
    number of experts that leaves a partial row group, k = 8 (the fused down
    projection + combine) over only 9 experts, and 300 experts; the MoE front
    launch (routing, shared and routed gate/up), and with the front switched
    off the routing launch followed by the grouped gate/up with the shared
    expert as problem 0."""
    N_in, K_out, I = 264, 256, 128
    L = Layer(H, N_in, K_out, E, I, k, base=6500 + E)
    n = E * I * H
    g = synth.bf16(n, SEED, 6510, 0, 0.05).reshape(E, I, H)
    u = synth.bf16(n, SEED, 6511, 0, 0.05).reshape(E, I, H)
    d = synth.bf16(n, SEED, 6512, 0, 0.05).reshape(E, H, I)
    sh = None
    if shared:
        sh = (synth.bf16(I * H, SEED, 6513, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 6514, 0, 0.05).reshape(I, H),
              synth.bf16(H * I, SEED, 6515, 0, 0.05).reshape(H, I))
    dev_w = L.device(dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                     None if sh is None else tuple(dev_bf16(a, a.shape) for a in sh))
    h.test_set_moe_front(front)
    for rep in range(3):  # the hand-off and queue counters must be left at zero by every call
        hbits, _ = gap_rows(L.scores, 1, H, k, base=6600 + 10 * E + rep)
        try:
            hid, tr = _run(h, L, dev_w, hbits)
        finally:
            h.test_set_moe_front(True)
        ex = lambda e: (g[e], u[e], d[e])
        ref = L.oracle(hbits, ex, sh)
        _check_layer(tr, hid, ref, slice(None), f"layer one token H={H} E={E} rep={rep}", L, ex, sh)


def test_layer_batch_rows_match_single_tokens(h):
    """M-invariance across the kernel families: the same 8 token rows as one
    batch (split-K family), as four batches of two (the few-token MoE front)
    and one by one (the one-token MoE front) give bit-identical top-k indices
    and outputs within the bf16 rule of each other (and of the oracle)."""
    H, N_in, K_out, E, I, k = 512, 520, 384, 40, 256, 8
    L = Layer(H, N_in, K_out, E, I, k, base=7600)
    n = E * I * H
    g = synth.bf16(n, SEED, 7610, 0, 0.05).reshape(E, I, H)
    u = synth.bf16(n, SEED, 7611, 0, 0.05).reshape(E, I, H)
    d = synth.bf16(n, SEED, 7612, 0, 0.05).reshape(E, H, I)
    sh = (synth.bf16(I * H, SEED, 7613, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 7614, 0, 0.05).reshape(I, H),
          synth.bf16(H * I, SEED, 7615, 0, 0.05).reshape(H, I))
    dev_w = L.device(dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                     tuple(dev_bf16(a, a.shape) for a in sh))
    hbits, _ = gap_rows(L.scores, 8, H, k, base=7700)
    ref = L.oracle(hbits, lambda e: (g[e], u[e], d[e]), sh)
    hid8, tr8 = _run(h, L, dev_w, hbits)
    out8, idx8, h1_8 = host_bits(hid8), tr8["idx"].cpu().numpy(), oracle.bf16_to_f64(host_bits(tr8["h1"]))
    for size in (2, 1):
        for r0 in range(0, 8, size):
            rows = slice(r0, r0 + size)
            hid, tr = _run(h, L, dev_w, hbits[rows])
            what = f"rows {r0}..{r0 + size - 1} as a batch of {size}"
            assert np.array_equal(tr["idx"].cpu().numpy(), idx8[rows]), what + ": top-k against the batch of 8"
            got = oracle.bf16_to_f64(host_bits(hid))
            # (each side may round its residual h1 one ulp apart: at most that much passes through)
            h1s = oracle.bf16_to_f64(host_bits(tr["h1"]))
            dh1 = np.minimum(np.abs(h1s - h1_8[rows]), ulp_bf16(h1_8[rows]))
            assert_bf16_close(host_bits(hid), oracle.bf16_to_f64(out8[rows]), what + " against the batch of 8",
                              tol=2e-2, passthrough=dh1)
            assert_bf16_close(host_bits(hid), ref["out"][rows], what + " against the oracle",
                              passthrough=np.minimum(np.abs(h1s - ref["h1"][rows]), ulp_bf16(ref["h1"][rows])))
            assert np.isfinite(got).all()


def _check_router_stage(L, tr, rows, what):
    """Router scores and weights on the layer's own input: the oracle's RMSNorm
    and router applied to the h1 the GPU produced. h1 is a bf16 activation
    that may differ from the oracle's h1 in last bits (checked above), and a
    last-bit change of the router input moves a logit by |W_r| * ulp, far
    beyond the router's own tolerance over 7168 terms; on the same input the
    router's fp32 error bound applies."""
    h1g = host_bits(tr["h1"])[rows]
    b = oracle.round_bf16(oracle.rmsnorm(h1g, L.g2))
    _, s_ref = oracle.router_scores(b, L.Wr)
    i_ref, w_ref = oracle.topk(s_ref, L.k)
    assert np.array_equal(tr["idx"].cpu().numpy()[rows], i_ref), what + ": top-k on the layer's h1"
    assert np.max(np.abs(tr["scores"].cpu().numpy()[rows] - s_ref)) <= SCORE_TOL, what + ": scores"
    assert np.max(np.abs(tr["w"].cpu().numpy()[rows] - w_ref)) <= WEIGHT_TOL, what + ": weights"


@pytest.mark.slow
def test_layer_one_token_two_router_units(h):
    """One token with more router units (40 row groups x 8 column chunks = 320)
    than the routing launch has CTAs on a 152-SM GPU (304): the first CTAs own
    two units, the second loaded after the norm. The 2 GB bank is placed by the
    device filler and regenerated per selected expert for the oracle."""
    import torch
    H, E, I, k, N_in, K_out = 8192, 320, 128, 8, 264, 256
    L = Layer(H, N_in, K_out, E, I, k, base=6700)
    n = E * I * H
    Wg = torch.empty((E, I, H), dtype=torch.bfloat16, device="cuda")
    Wu = torch.empty_like(Wg)
    Wd = torch.empty((E, H, I), dtype=torch.bfloat16, device="cuda")
    for t, tid in ((Wg, synth.W_G), (Wu, synth.W_U), (Wd, synth.W_D)):
        synth.fill_bf16_dev(t.data_ptr(), n, 0, tid, 0, 0.02)
    sh_bits = (synth.bf16(I * H, SEED, 6710, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 6711, 0, 0.05).reshape(I, H),
               synth.bf16(H * I, SEED, 6712, 0, 0.05).reshape(H, I))
    dev_w = L.device(Wg, Wu, Wd, tuple(dev_bf16(a, a.shape) for a in sh_bits))
    bank = HostBank(E, H, I)
    for rep in range(2):
        hbits, _ = gap_rows(L.scores, 1, H, k, base=6720 + rep)
        hid, tr = _run(h, L, dev_w, hbits)
        ref = L.oracle(hbits, bank, sh_bits)
        _check_layer(tr, hid, ref, slice(None), f"layer one token two units rep={rep}", L, bank, sh_bits)
    del Wg, Wu, Wd
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,group", [(2, 2), (16, 8), (64, 8)])
def test_layer_speculative_verify_batch(h, M, group):
    """A speculative-verify batch: groups of related token rows (one request's
    drafts) route largely to the same experts, so the split-K family's expert
    tiles carry several tokens and U is well below the independent-token case."""
    H, N_in, K_out, E, I, k = 256, 264, 256, 128, 128, 8
    L = Layer(H, N_in, K_out, E, I, k, base=6950 + M)
    n = E * I * H
    g = synth.bf16(n, SEED, 6960, 0, 0.05).reshape(E, I, H)
    u = synth.bf16(n, SEED, 6961, 0, 0.05).reshape(E, I, H)
    d = synth.bf16(n, SEED, 6962, 0, 0.05).reshape(E, H, I)
    sh = (synth.bf16(I * H, SEED, 6963, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 6964, 0, 0.05).reshape(I, H),
          synth.bf16(H * I, SEED, 6965, 0, 0.05).reshape(H, I))
    dev_w = L.device(dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                     tuple(dev_bf16(a, a.shape) for a in sh))
    hbits, _ = gap_correlated_rows(L.scores, M, H, k, base=7000 + M, group=group, eps=0.3)
    hid, tr = _run(h, L, dev_w, hbits)
    ex = lambda e: (g[e], u[e], d[e])
    ref = L.oracle(hbits, ex, sh)
    _check_layer(tr, hid, ref, slice(None), f"layer verify batch M={M} group={group}", L, ex, sh)
    idx = tr["idx"].cpu().numpy()
    U = len(np.unique(idx))
    if M >= 16:  # related rows share experts: well below the independent-token expectation
        assert U < 0.8 * E * (1 - (1 - k / E) ** M), U


@pytest.mark.parametrize("front", [True, False])
@pytest.mark.parametrize("M", [2, 3, 4])
@pytest.mark.parametrize("I,shared", [(128, True), (256, False), (256, True), (384, True), (512, False)])
def test_layer_few_tokens(h, M, I, shared, front):
    """Two to four tokens on the small-matrix family (forced): one routing
    launch (second RMSNorm, router, per-token top-k, a routing table with one
    problem per (token, expert) entry, and the shared expert's gate/up), the
    entries' gate/up (with a shared expert and the front on: inside that
    launch, the MoE front; otherwise a launch of its own), down over the
    shared expert's M rows plus the entries, then the combine. At two tokens
    with I > 256 the down, the combine and the residual are one kernel
    (I = 384: a ragged thread count; I = 512 without a shared expert)."""
    import moe_layers_gb300 as ML
    H, N_in, K_out, E, k = 1152, 264, 256, 40, 8
    L = Layer(H, N_in, K_out, E, I, k, base=6800 + I + M)
    n = E * I * H
    g = synth.bf16(n, SEED, 6810, 0, 0.05).reshape(E, I, H)
    u = synth.bf16(n, SEED, 6811, 0, 0.05).reshape(E, I, H)
    d = synth.bf16(n, SEED, 6812, 0, 0.05).reshape(E, H, I)
    sh = None
    if shared:
        sh = (synth.bf16(I * H, SEED, 6813, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 6814, 0, 0.05).reshape(I, H),
              synth.bf16(H * I, SEED, 6815, 0, 0.05).reshape(H, I))
    dev_w = L.device(dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                     None if sh is None else tuple(dev_bf16(a, a.shape) for a in sh))
    h.set_force_variant(ML.VARIANT_SMALL_M)
    h.test_set_moe_front(front)
    try:
        for rep in range(2):  # the counters must be back at zero after every call
            hbits, _ = gap_rows(L.scores, M, H, k, base=6900 + 10 * M + I + rep)
            hid, tr = _run(h, L, dev_w, hbits)
            assert h.last_expert_variant == ML.VARIANT_SMALL_M
            ex = lambda e: (g[e], u[e], d[e])
            ref = L.oracle(hbits, ex, sh)
            _check_layer(tr, hid, ref, slice(None), f"layer few tokens M={M} I={I} front={front} rep={rep}", L, ex, sh)
    finally:
        h.set_force_variant(ML.VARIANT_AUTO)
        h.test_set_moe_front(True)


@pytest.mark.parametrize("M,family", [(1, "auto"), (2, "auto"), (4, "auto"), (4, "split_k")])
def test_layer_front_with_sms_held_by_another_stream(h, M, family):
    """The MoE front's CTAs wait for the routing that one of them publishes.
    Here a kernel on another stream holds half the SMs for 150 ms, so only
    half of the front's CTAs can be resident at once, and the routing wait is
    limited to 30 ms: the routing must complete with the CTAs that are
    running (router units go to whichever CTAs take them), so the layer
    returns DEC_OK with the oracle's result instead of a timeout. (A front
    whose router units belonged to fixed CTAs would wait for CTAs that cannot
    start until the other kernel ends, and time out.) At four tokens these small
    experts take the few-token front; with the split-K family forced, the
    engine's launches run with half the SMs held: the CTA that finishes a
    split tile waits a bounded time for the other pieces, then leaves the tile
    to the last piece's CTA, so it completes as well."""
    import time
    import torch
    import moe_layers_gb300 as ML
    H, N_in, K_out, E, I, k = 1152, 264, 256, 40, 256, 8
    L = Layer(H, N_in, K_out, E, I, k, base=7800 + M)
    n = E * I * H
    g = synth.bf16(n, SEED, 7810, 0, 0.05).reshape(E, I, H)
    u = synth.bf16(n, SEED, 7811, 0, 0.05).reshape(E, I, H)
    d = synth.bf16(n, SEED, 7812, 0, 0.05).reshape(E, H, I)
    sh = (synth.bf16(I * H, SEED, 7813, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 7814, 0, 0.05).reshape(I, H),
          synth.bf16(H * I, SEED, 7815, 0, 0.05).reshape(H, I))
    dev_w = L.device(dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                     tuple(dev_bf16(a, a.shape) for a in sh))
    hbits, _ = gap_rows(L.scores, M, H, k, base=7900 + M)
    ex = lambda e: (g[e], u[e], d[e])
    ref = L.oracle(hbits, ex, sh)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    hid = dev_bf16(hbits, hbits.shape)
    torch.cuda.synchronize()
    side, main = torch.cuda.Stream(), torch.cuda.Stream()
    h.set_wait_limit_ns(30_000_000)
    if family == "split_k":
        h.set_force_variant(ML.VARIANT_SPLIT_K)
    try:
        ML.test_occupy_sms(h, sms // 2, 150_000_000, stream=side)
        time.sleep(0.002)  # the holding kernel is resident before the layer is launched
        launches0 = h.launch_count
        with torch.cuda.stream(main):
            tr = ML.decode_layer(h, dev_w, hid, trace=True, stream=main)
        # the MoE front schedule: four launches at one and two tokens, five at four (down and combine
        # apart); the split-K family: twelve (the first RMSNorm is a launch of its own there)
        assert h.launch_count - launches0 == (12 if family == "split_k" else 4 if M <= 2 else 5)
        torch.cuda.synchronize()
    finally:
        h.set_wait_limit_ns(500_000_000)
        h.set_force_variant(ML.VARIANT_AUTO)
    assert h.check_device_error() == ML.DEC_OK
    _check_layer(tr, hid, ref, slice(None), f"layer M={M} beside a kernel holding {sms // 2} SMs", L, ex, sh)


def _check_layer(tr, hid, ref, rows, what, L=None, expert=None, shared=None):
    """Layer output checks, on the rows `rows` of the GPU's buffers (ref holds
    the oracle's rows for them):
    - top-k indices bit-exact against the oracle's layer;
    - h1 (a stored bf16 activation) by the bf16 rule against the oracle's h1
      before its storage rounding (the exact out-projection + residual of the
      oracle's stored inputs), so that the rule's half-ulp allowance covers the
      one rounding each side makes: against the oracle's rounded h1 a correct
      rounding of a sum near a midpoint would count a whole ulp;
    - the output end to end by the bf16 rule, where the h1 difference that
      passes unchanged through the residual add is allowed up to one bf16 ulp
      of the oracle's h1 per element: h1 is rounded to bf16 once on each side
      (fp32 sums on the GPU, fp64 in the oracle), and two correct roundings of
      nearly equal sums can land one ulp apart;
    - with L and expert given, the MoE stage on the GPU's own h1 by the plain
      bf16 rule, nothing passed through: out against h1_gpu + the oracle's
      RMSNorm, router, top-k and experts applied to that h1, and the router's
      scores and weights on it (_check_router_stage)."""
    assert np.array_equal(tr["idx"].cpu().numpy()[rows], ref["idx"]), what + ": top-k indices"
    h1g = oracle.bf16_to_f64(host_bits(tr["h1"])[rows])
    dh1 = np.minimum(np.abs(h1g - ref["h1"]), ulp_bf16(ref["h1"]))
    assert_bf16_close(host_bits(tr["h1"])[rows], ref["unrounded"]["h1"], what + " h1")
    assert_bf16_close(host_bits(hid)[rows], ref["out"], what + " out", passthrough=dh1)
    if L is not None:
        _check_router_stage(L, tr, rows, what)
        if expert is not None:
            b = oracle.round_bf16(oracle.rmsnorm(h1g, L.g2))
            _, s = oracle.router_scores(b, L.Wr)
            idx, w = oracle.topk(s, L.k)
            stage = h1g + oracle.moe(b, idx, w, expert, shared)
            assert_bf16_close(host_bits(hid)[rows], stage, what + " out from the GPU's h1 (MoE stage)")


def sample_rows(M: int, n: int = 16):
    """Every row of a batch of up to n rows, else n rows spread over the batch
    (first and last included)."""
    if M <= n:
        return list(range(M))
    return sorted(set(int(round(v)) for v in np.linspace(0, M - 1, n)))


@pytest.fixture(scope="module")
def full_layer():
    return Layer(H_FULL, N_IN_FULL, K_OUT_FULL, E_FULL, I_FULL, K_FULL, base=synth.W_IN * 0 + 7000,
                 gamma_noise=False)


@pytest.mark.parametrize("M,front", [(1, True), (1, False), (2, True), (2, False), (4, True), (8, True), (16, True),
                                     (32, True), (64, True)])
def test_layer_full_size(h, full_bank, full_layer, M, front):
    """The full-size layer; at one and two tokens also with the MoE front
    switched off (the routing launch, then the grouped kernels). Output rows are compared
    with the oracle on every row up to 16 tokens and on 16 rows spread over
    the batch above; the top-k indices on every row."""
    Wg, Wu, Wd, sh = full_bank
    L = full_layer
    hbits, _ = gap_rows(L.scores, M, H_FULL, K_FULL, base=synth.X_BASE + 30)
    h.test_set_moe_front(front)
    try:
        hid, tr = _run(h, L, L.device(Wg, Wu, Wd, sh), hbits)
    finally:
        h.test_set_moe_front(True)
    bank = HostBank(E_FULL, H_FULL, I_FULL, cache=160)
    shared = tuple(oracle.bf16_to_f64(synth.bf16(I_FULL * H_FULL, SEED, tid, 0, 0.02)).reshape(shape)
                   for tid, shape in ((synth.W_G_S, (I_FULL, H_FULL)), (synth.W_U_S, (I_FULL, H_FULL)),
                                      (synth.W_D_S, (H_FULL, I_FULL))))
    tokens = sample_rows(M)
    ref = L.oracle(hbits, bank, shared, tokens=tokens)
    _check_layer(tr, hid, ref, tokens, f"layer full M={M}", L, bank, shared)
    # indices of all tokens: bit-exact against the oracle's router on every row
    s_all = L.scores(hbits)
    i_all, _ = oracle.topk(s_all, K_FULL)
    assert np.array_equal(tr["idx"].cpu().numpy(), i_all)


# ---------------------------------------------------------------------------- TP-shard shapes
@pytest.fixture(scope="module", params=[8, 16], ids=["tp8", "tp16"])
def tp_layer(request):
    """Per-GPU shapes of the layer in an s-way tensor-parallel deployment: the
    input projection split over its outputs, the out-projection over its
    inputs and every expert over its intermediate size; 384 experts, the
    router replicated. The bank is placed by the device filler."""
    import torch
    sh = request.param
    H, E, k = H_FULL, E_FULL, K_FULL
    N_in, K_out, I = N_IN_FULL // sh, K_OUT_FULL // sh, I_FULL // sh
    L = Layer(H, N_in, K_out, E, I, k, base=7100 + sh, gamma_noise=True)
    n = E * I * H
    Wg = torch.empty((E, I, H), dtype=torch.bfloat16, device="cuda")
    Wu = torch.empty_like(Wg)
    Wd = torch.empty((E, H, I), dtype=torch.bfloat16, device="cuda")
    ids = (synth.W_G, synth.W_U, synth.W_D)
    for t, tid in zip((Wg, Wu, Wd), ids):
        synth.fill_bf16_dev(t.data_ptr(), n, 0, tid, 0, 0.02)
    sh_bits = tuple(synth.bf16(I * H, SEED, 7150 + q, 0, 0.02).reshape(shape)
                    for q, shape in enumerate(((I, H), (I, H), (H, I))))
    dev_w = L.device(Wg, Wu, Wd, tuple(dev_bf16(a, a.shape) for a in sh_bits))
    yield sh, L, dev_w, HostBank(E, H, I, cache=300), sh_bits
    del Wg, Wu, Wd, dev_w
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("M", [1, 2, 4, 64])
def test_layer_tp_shapes(h, tp_layer, M):
    sh, L, dev_w, bank, sh_bits = tp_layer
    hbits, _ = gap_rows(L.scores, M, L.H, L.k, base=synth.X_BASE + 60 + sh)
    hid, tr = _run(h, L, dev_w, hbits)
    tokens = sample_rows(M)
    ref = L.oracle(hbits, bank, sh_bits, tokens=tokens)
    _check_layer(tr, hid, ref, tokens, f"layer TP{sh} M={M}", L, bank, sh_bits)
    s_all = L.scores(hbits)
    i_all, _ = oracle.topk(s_all, L.k)
    assert np.array_equal(tr["idx"].cpu().numpy(), i_all)


# ---------------------------------------------------------------------------- several distinct layers in sequence
def _chain_gap_rows(layers, M, H, k, base, gaps=(1e-3, 2.5e-3, 2.5e-3), max_attempts=4000):
    """Token rows whose routing has a top-(k+1) score gap in every layer of
    the chain, as the oracle computes it (layer l's input is layer l-1's
    output stored as bf16): 1e-3 in the first layer, whose input is drawn,
    and 2.5e-3 in the later ones, whose inputs on the GPU carry the earlier
    layers' roundings (measured: after two layers they can move a score by
    more than half of 1e-3). About 2% of rows pass all three."""
    from _util import gap_ok
    bits = np.empty((M, H), dtype=np.uint16)
    for r in range(M):
        for attempt in range(max_attempts + 1):
            row = synth.bf16_rows(base, [r], H, SEED, 1.0, [attempt])
            x, ok = row, True
            for (L, ex, sh), gap in zip(layers, gaps):
                s = L.scores(x)
                if not gap_ok(s[0], L.k, gap):
                    ok = False
                    break
                o = L.oracle(x, ex, sh)
                x = _bits(oracle.round_bf16(o["out"]))
            if ok:
                bits[r] = row[0]
                break
        else:
            raise RuntimeError("gap rule: too many redraws")
    return bits


@pytest.mark.parametrize("M", [1, 2, 8])
def test_layers_in_sequence_with_cross_layer_prefetch(h, M):
    """Three distinct layers (their own seeded weights, routers and expert
    banks) applied in sequence, layer l's output (bf16) being layer l+1's
    input, each layer's prefetch_next region set to the next layer's input
    projection (the last to the first) and, in a second run, to nothing:
    - the outputs of the two runs are bit-identical (the prefetch moves data
      into L2 only);
    - every layer's output and top-k indices pass the layer rule against the
      oracle applied to that layer's GPU input;
    - every layer's top-k indices are bit-exact against the oracle's own
      chain (its rows drawn with a wider score gap in the later layers, see
      _chain_gap_rows; the router is the workload's N(0, 0.01), at which one
      last-bit difference of a normalised row stays within the 1e-4 score
      tolerance);
    - the chain's final output is within 3 x 1e-2 rms of the oracle's chain
      (each of the three layers may contribute up to the one-layer budget)."""
    import torch
    import moe_layers_gb300 as ML
    H, N_in, K_out, E, I, k = 1152, 1040, 1024, 40, 256, 8
    layers = []
    for l in range(3):
        L = Layer(H, N_in, K_out, E, I, k, base=9200 + 20 * l)
        n = E * I * H
        g = synth.bf16(n, SEED, 9210 + 20 * l, 0, 0.05).reshape(E, I, H)
        u = synth.bf16(n, SEED, 9211 + 20 * l, 0, 0.05).reshape(E, I, H)
        d = synth.bf16(n, SEED, 9212 + 20 * l, 0, 0.05).reshape(E, H, I)
        sh = (synth.bf16(I * H, SEED, 9213 + 20 * l, 0, 0.05).reshape(I, H),
              synth.bf16(I * H, SEED, 9214 + 20 * l, 0, 0.05).reshape(I, H),
              synth.bf16(H * I, SEED, 9215 + 20 * l, 0, 0.05).reshape(H, I))
        ex = (lambda g, u, d: (lambda e: (g[e], u[e], d[e])))(g, u, d)
        dev_w = L.device(dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                         tuple(dev_bf16(a, a.shape) for a in sh))
        layers.append((L, ex, sh, dev_w))
    hbits = _chain_gap_rows([(L, ex, sh) for L, ex, sh, _ in layers], M, H, k, base=9300 + M)
    outs = {}
    for pf in (True, False):
        for l, (_, _, _, dev_w) in enumerate(layers):
            nxt = layers[(l + 1) % 3][3].W_in
            dev_w.prefetch_next = nxt if pf else None
            dev_w.prefetch_bytes = nxt.numel() * 2 if pf else 0
        hid = dev_bf16(hbits, hbits.shape)
        ins, trs = [], []
        for l, (_, _, _, dev_w) in enumerate(layers):
            ins.append(host_bits(hid))
            trs.append(ML.decode_layer(h, dev_w, hid, trace=True))
        torch.cuda.synchronize()
        outs[pf] = (host_bits(hid), ins, [{k_: v.clone() for k_, v in t.items()} for t in trs])
    assert h.check_device_error() == ML.DEC_OK
    assert np.array_equal(outs[True][0], outs[False][0]), "cross-layer prefetch changed the result"
    final, ins, trs = outs[True]
    x, last = hbits, None
    for l, (L, ex, sh, _) in enumerate(layers):
        # this layer on the GPU's own input to it
        ref = L.oracle(ins[l], ex, sh)
        got = ins[l + 1] if l + 1 < 3 else final
        hid_l = dev_bf16(got, got.shape)
        _check_layer(trs[l], hid_l, ref, slice(None), f"chain M={M} layer {l}", L, ex, sh)
        # the oracle's own chain
        oc = L.oracle(x, ex, sh)
        assert np.array_equal(trs[l]["idx"].cpu().numpy(), oc["idx"]), f"chain M={M} layer {l}: top-k"
        x, last = _bits(oracle.round_bf16(oc["out"])), oc["out"]
    assert_bf16_close(final, last, f"chain M={M}: final output against the oracle's chain", tol=3e-2)
