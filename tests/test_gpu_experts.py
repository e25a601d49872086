"""GPU parity of the MoE expert layer (moe_experts): routed SwiGLU experts
over the selected ids, the shared expert on the side stream, weighted combine
and optional residual, against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import synth
from _util import SEED, HostBank, assert_bf16_close, dev_bf16, dev_f32, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import torch
    import moe_layers_gb300 as M
    assert torch.cuda.is_available()
    M.build()
    with M.Handle(0) as hd:
        yield hd


def _routing(M, E, k, rng, skew=False):
    if skew:  # every token picks the same experts: one expert sees all M tokens
        ids = np.tile(rng.permutation(E)[:k], (M, 1))
    else:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(M)])
    w = rng.random((M, k)) + 0.1
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids.astype(np.int32), w


def _small_bank(E, H, I, base):
    n = E * I * H
    g = synth.bf16(n, SEED, base, 0, 0.05)
    u = synth.bf16(n, SEED, base + 1, 0, 0.05)
    d = synth.bf16(n, SEED, base + 2, 0, 0.05)
    return g.reshape(E, I, H), u.reshape(E, I, H), d.reshape(E, H, I)


@pytest.mark.parametrize("family", ["auto", "split_k"])
@pytest.mark.parametrize("M,E,H,I,k,shared,resid,skew", [
    (1, 24, 384, 256, 8, True, True, False),
    (1, 24, 384, 256, 8, False, False, False),
    (1, 16, 256, 128, 4, True, False, False),
    (3, 16, 256, 256, 4, False, True, False),
    (17, 32, 384, 128, 8, True, True, False),
    (64, 24, 256, 128, 8, True, False, False),
    (64, 40, 128, 256, 16, True, True, True),
    (20, 8, 512, 384, 2, False, False, True),
])
def test_experts_small(h, M, E, H, I, k, shared, resid, skew, family):
    import moe_layers_gb300 as ML
    if family == "split_k" and M > 1:
        pytest.skip("above one token the split-K family is the automatic choice")
    h.set_force_variant(ML.VARIANT_SPLIT_K if family == "split_k" else ML.VARIANT_AUTO)
    rng = np.random.default_rng(M * 131 + E)
    g, u, d = _small_bank(E, H, I, 4000 + E + H)
    x = synth.bf16(M * H, SEED, 4100 + M, 0, 1.0).reshape(M, H)
    idx, w = _routing(M, E, k, rng, skew)
    sh = None
    if shared:
        sg = synth.bf16(I * H, SEED, 4200, 0, 0.05).reshape(I, H)
        su = synth.bf16(I * H, SEED, 4201, 0, 0.05).reshape(I, H)
        sd = synth.bf16(H * I, SEED, 4202, 0, 0.05).reshape(H, I)
        sh = (sg, su, sd)
    r = synth.bf16(M * H, SEED, 4300 + M, 0, 1.0).reshape(M, H) if resid else None
    import torch
    out = ML.moe_experts(h, dev_bf16(x, (M, H)), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                         dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                         shared=None if sh is None else tuple(dev_bf16(a, a.shape) for a in sh),
                         residual=None if r is None else dev_bf16(r, (M, H)))
    h.set_force_variant(ML.VARIANT_AUTO)
    assert h.last_expert_variant == (ML.VARIANT_SMALL_M if (M == 1 and family == "auto") else ML.VARIANT_SPLIT_K)
    ref = oracle.moe(x, idx, w, lambda e: (g[e], u[e], d[e]), sh, r)
    assert_bf16_close(host_bits(out), ref, f"moe M={M} E={E} {family}")
    assert h.check_device_error() == ML.DEC_OK


@pytest.mark.parametrize("M,E,H,I,k", [(8, 16, 1024, 512, 4), (64, 24, 768, 256, 8)])
def test_split_tile_finish_paths_give_the_same_bits(h, M, E, H, I, k):
    """The split-K kernel's three ways of finishing a tile split between CTAs
    (the first piece's CTA from shared memory; the CTA that completes the count;
    the same with the pieces read from L2) add the same fp32 partials in the
    same k order: the grouped experts' outputs agree bit for bit."""
    import torch
    import moe_layers_gb300 as ML
    rng = np.random.default_rng(M * 7 + E)
    g, u, d = _small_bank(E, H, I, 4600 + E)
    x = synth.bf16(M * H, SEED, 4700 + M, 0, 1.0).reshape(M, H)
    idx, w = _routing(M, E, k, rng, False)
    sh = tuple(synth.bf16(n, SEED, 4800 + i, 0, 0.05).reshape(shape)
               for i, (n, shape) in enumerate([(I * H, (I, H)), (I * H, (I, H)), (H * I, (H, I))]))
    r = synth.bf16(M * H, SEED, 4900 + M, 0, 1.0).reshape(M, H)
    outs = []
    try:
        for mode in (0, 1, 2):
            h.test_set_engine_finish(mode)
            out = ML.moe_experts(h, dev_bf16(x, (M, H)), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                                 dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                                 shared=tuple(dev_bf16(a, a.shape) for a in sh), residual=dev_bf16(r, (M, H)))
            assert h.last_expert_variant == ML.VARIANT_SPLIT_K
            outs.append(host_bits(out))
    finally:
        h.test_set_engine_finish(0)
    assert_bf16_close(outs[0], oracle.moe(x, idx, w, lambda e: (g[e], u[e], d[e]), sh, r), f"moe M={M}")
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2]), "finish paths differ"
    assert h.check_device_error() == ML.DEC_OK


# ---------------------------------------------------------------------------- workload size
from conftest import E_FULL, H_FULL, I_FULL, K_FULL


@pytest.mark.parametrize("family", ["auto", "split_k"])
@pytest.mark.parametrize("k,ids", [(4, [3, 3, 7, 3]), (8, [5, 1, 5, 2, 5, 9, 1, 0])])
def test_experts_one_token_repeated_ids(h, family, k, ids):
    """A token may list an expert more than once (the top-k never does, a
    caller of the expert layer may): the result is still the sum over its
    entries. At one token each entry is its own problem."""
    import moe_layers_gb300 as ML
    import torch
    E, H, I = 12, 256, 128
    h.set_force_variant(ML.VARIANT_SPLIT_K if family == "split_k" else ML.VARIANT_AUTO)
    g, u, d = _small_bank(E, H, I, 4500 + k)
    x = synth.bf16(H, SEED, 4510 + k, 0, 1.0).reshape(1, H)
    idx = np.array([ids], dtype=np.int32)
    w = np.random.default_rng(k).random((1, k)).astype(np.float32) + 0.1
    w /= w.sum()
    sh = (synth.bf16(I * H, SEED, 4520, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 4521, 0, 0.05).reshape(I, H),
          synth.bf16(H * I, SEED, 4522, 0, 0.05).reshape(H, I))
    r = synth.bf16(H, SEED, 4530, 0, 1.0).reshape(1, H)
    out = ML.moe_experts(h, dev_bf16(x, (1, H)), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                         dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape),
                         shared=tuple(dev_bf16(a, a.shape) for a in sh), residual=dev_bf16(r, (1, H)))
    h.set_force_variant(ML.VARIANT_AUTO)
    ref = oracle.moe(x, idx, w, lambda e: (g[e], u[e], d[e]), sh, r)
    assert_bf16_close(host_bits(out), ref, f"moe repeated ids k={k} {family}")
    assert h.check_device_error() == ML.DEC_OK


@pytest.mark.parametrize("M,family", [(1, "auto"), (1, "split_k"), (8, "auto"), (64, "auto")])
def test_experts_full_size(h, full_bank, M, family):
    import torch
    import moe_layers_gb300 as ML
    h.set_force_variant(ML.VARIANT_SPLIT_K if family == "split_k" else ML.VARIANT_AUTO)
    Wg, Wu, Wd, sh = full_bank
    rng = np.random.default_rng(5000 + M)
    idx, w = _routing(M, E_FULL, K_FULL, rng)
    x = synth.bf16_rows(synth.X_BASE + 20, range(M), H_FULL, SEED)
    out = ML.moe_experts(h, dev_bf16(x, (M, H_FULL)), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                         Wg, Wu, Wd, shared=sh)
    h.set_force_variant(ML.VARIANT_AUTO)
    bank = HostBank(E_FULL, H_FULL, I_FULL)
    shared = tuple(oracle.bf16_to_f64(synth.bf16(I_FULL * H_FULL, SEED, tid, 0, 0.02)).reshape(shape)
                   for tid, shape in ((synth.W_G_S, (I_FULL, H_FULL)), (synth.W_U_S, (I_FULL, H_FULL)),
                                      (synth.W_D_S, (H_FULL, I_FULL))))
    # every token up to 16, else 16 tokens spread over the batch; each is a full output row
    tokens = list(range(M)) if M <= 16 else sorted(set(int(round(v)) for v in np.linspace(0, M - 1, 16)))
    ref = oracle.moe(x, idx, w, bank, shared, tokens=tokens)
    got = host_bits(out)[tokens]
    assert_bf16_close(got, ref, f"moe full M={M}")
