"""GPU parity of router scoring and top-k (moe_route_topk) against the oracle:
scores within 1e-4 absolute, indices bit-exact on inputs whose top-(k+1)
oracle scores are at least 1e-3 apart, weights within 1e-5."""
import numpy as np
import pytest

import oracle
import synth
from _util import GAP, SCORE_TOL, SEED, WEIGHT_TOL, dev_bf16, dev_f32, gap_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import torch
    import moe_layers_gb300 as M
    assert torch.cuda.is_available()
    M.build()
    with M.Handle(0) as hd:
        yield hd


def _check(h, xbits, Wr, k):
    import moe_layers_gb300 as ML
    M, H = xbits.shape
    idx, w, sc = ML.moe_route_topk(h, dev_bf16(xbits, (M, H)), dev_f32(Wr), k)
    _, s_ref = oracle.router_scores(xbits, Wr)
    i_ref, w_ref = oracle.topk(s_ref, k)
    assert np.max(np.abs(sc.cpu().numpy() - s_ref)) <= SCORE_TOL
    assert np.array_equal(idx.cpu().numpy(), i_ref)
    assert np.max(np.abs(w.cpu().numpy() - w_ref)) <= WEIGHT_TOL
    return idx


@pytest.mark.parametrize("M,H,E,k", [(1, 256, 64, 4), (5, 512, 128, 8), (17, 2056, 384, 8), (64, 1024, 40, 16),
                                     (3, 64, 16, 1), (1, 1032, 37, 5), (1, 2056, 1024, 4), (1, 1024, 40, 16), (1, 64, 16, 1),
                                     (1, 3072, 9, 9)])
def test_router_small(h, M, H, E, k):
    Wr = synth.f32(E * H, SEED, 3000 + E, 0, 0.8 / np.sqrt(H)).reshape(E, H)  # logits ~ N(0, 0.8^2)
    score = lambda rows: oracle.router_scores(rows, Wr)[1]
    xbits, _ = gap_rows(score, M, H, k, base=3100 + H, gap=GAP)
    _check(h, xbits, Wr, k)


@pytest.fixture(scope="module")
def wr_full():
    return synth.f32(384 * 7168, SEED, synth.W_R, 0, 0.01).reshape(384, 7168)


@pytest.mark.parametrize("M", [1, 8, 64])
def test_router_full(h, wr_full, M):
    score = lambda rows: oracle.router_scores(rows, wr_full)[1]
    xbits, attempts = gap_rows(score, M, 7168, 8, base=synth.X_BASE + 7, gap=GAP)
    _check(h, xbits, wr_full, 8)


def test_router_ties_go_to_lower_ids(h):
    import moe_layers_gb300 as ML
    M, H, E, k = 4, 128, 32, 8
    x = synth.bf16(M * H, SEED, 3200, 0, 1.0).reshape(M, H)
    Wr = np.zeros((E, H), dtype=np.float32)
    idx, w, sc = ML.moe_route_topk(h, dev_bf16(x, (M, H)), dev_f32(Wr), k)
    assert np.all(sc.cpu().numpy() == 0.5)
    assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(k, dtype=np.int32), (M, 1)))
    assert np.all(w.cpu().numpy() == np.float32(1.0 / k))


def test_router_one_token_repeated(h):
    """One token runs as one launch whose last CTA takes the top-k; its
    hand-off counter must be back at zero after every call."""
    H, E, k = 1032, 100, 6
    Wr = synth.f32(E * H, SEED, 3300, 0, 0.8 / np.sqrt(H)).reshape(E, H)
    score = lambda rows: oracle.router_scores(rows, Wr)[1]
    for rep in range(4):
        xbits, _ = gap_rows(score, 1, H, k, base=3400 + rep, gap=GAP)
        _check(h, xbits, Wr, k)


def test_router_ties_one_token(h):
    import moe_layers_gb300 as ML
    H, E, k = 128, 40, 8
    x = synth.bf16(H, SEED, 3201, 0, 1.0).reshape(1, H)
    Wr = np.zeros((E, H), dtype=np.float32)
    idx, w, sc = ML.moe_route_topk(h, dev_bf16(x, (1, H)), dev_f32(Wr), k)
    assert np.all(sc.cpu().numpy() == 0.5)
    assert np.array_equal(idx.cpu().numpy(), np.arange(k, dtype=np.int32)[None, :])
    assert np.all(w.cpu().numpy() == np.float32(1.0 / k))
