"""GPU checks of the schedule settings: every setting of the handle changes
how the layer is launched, never what it computes (each run is checked against
the oracle), the profiling records report every launch, and the settings and
the L2 prefetch entry point validate their arguments."""
import numpy as np
import pytest

import synth
from _util import SEED, dev_bf16, gap_rows
from test_gpu_layer import Layer, _check_layer, _run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import torch
    import moe_layers_gb300 as M
    assert torch.cuda.is_available()
    M.build()
    with M.Handle(0) as hd:
        yield hd


@pytest.fixture(scope="module")
def small_layer():
    H, N_in, K_out, E, I, k = 256, 264, 256, 32, 128, 8
    L = Layer(H, N_in, K_out, E, I, k, base=8000)
    n = E * I * H
    g = synth.bf16(n, SEED, 8010, 0, 0.05).reshape(E, I, H)
    u = synth.bf16(n, SEED, 8011, 0, 0.05).reshape(E, I, H)
    d = synth.bf16(n, SEED, 8012, 0, 0.05).reshape(E, H, I)
    sh = (synth.bf16(I * H, SEED, 8013, 0, 0.05).reshape(I, H), synth.bf16(I * H, SEED, 8014, 0, 0.05).reshape(I, H),
          synth.bf16(H * I, SEED, 8015, 0, 0.05).reshape(H, I))
    dev = (dev_bf16(g, g.shape), dev_bf16(u, u.shape), dev_bf16(d, d.shape), tuple(dev_bf16(a, a.shape) for a in sh))
    return L, (g, u, d, sh), dev


def _defaults(h):
    import moe_layers_gb300 as ML
    h.set_force_variant(ML.VARIANT_AUTO)
    h.set_shared_sms(0)
    h.set_pdl(True)
    h.set_l2_ahead(49152)
    h.test_set_moe_front(True)


SETTINGS = {
    "default": {},
    "no_pdl": {"pdl": False},
    "no_l2_ahead": {"l2_ahead": 0},
    "big_l2_ahead": {"l2_ahead": 1 << 20},
    "no_moe_front": {"moe_front": False},
    "shared_overlap": {"shared_sms": -1},
    "shared_fixed_4": {"shared_sms": 4},
    "prefetch_next": {"prefetch_next": True},
    "split_k_family": {"force": "split_k"},
    "small_m_family": {"force": "small_m"},
}


@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("name", list(SETTINGS))
def test_layer_settings_change_schedule_not_result(h, small_layer, M, name):
    import moe_layers_gb300 as ML
    L, (g, u, d, sh), (gd, ud, dd, shd) = small_layer
    cfg = SETTINGS[name]
    dev_w = L.device(gd, ud, dd, shd)
    if cfg.get("prefetch_next"):
        dev_w.prefetch_next = gd  # any device region: the pull into L2 must not change the result
        dev_w.prefetch_bytes = 1 << 20
    _defaults(h)
    try:
        if "pdl" in cfg:
            h.set_pdl(cfg["pdl"])
        if "l2_ahead" in cfg:
            h.set_l2_ahead(cfg["l2_ahead"])
        if "moe_front" in cfg:
            h.test_set_moe_front(cfg["moe_front"])
        if "shared_sms" in cfg:
            h.set_shared_sms(cfg["shared_sms"])
        if cfg.get("force") == "split_k":
            h.set_force_variant(ML.VARIANT_SPLIT_K)
        if cfg.get("force") == "small_m":
            if M > 4:
                pytest.skip("the small-matrix family covers up to four tokens")
            h.set_force_variant(ML.VARIANT_SMALL_M)
        for rep in range(2):
            hbits, _ = gap_rows(L.scores, M, L.H, L.k, base=8100 + 10 * M + rep)
            hid, tr = _run(h, L, dev_w, hbits)
            ex = lambda e: (g[e], u[e], d[e])
            ref = L.oracle(hbits, ex, sh)
            _check_layer(tr, hid, ref, slice(None), f"layer {name} M={M} rep={rep}", L, ex, sh)
        assert h.check_device_error() == ML.DEC_OK
    finally:
        _defaults(h)


def test_profiling_reports_every_launch(h, small_layer):
    L, _, (gd, ud, dd, shd) = small_layer
    dev_w = L.device(gd, ud, dd, shd)
    expect = {
        # one token: the MoE front launch (routing, shared and routed gate/up), then down + combine
        1: {"in_proj", "out_proj", "moe_front", "down"},
        # three tokens on small matrices: small-matrix input projection with the RMSNorm inside,
        # and, with experts this small, the few-token MoE front, down, combine
        3: {"in_proj", "out_proj", "moe_front", "down", "combine"},
        8: {"rmsnorm1", "in_proj", "out_proj", "rmsnorm2", "router", "topk", "route_table", "gate_up", "down",
            "shared_gate_up", "shared_down", "combine"},
    }
    for M, tags in expect.items():
        hbits, _ = gap_rows(L.scores, M, L.H, L.k, base=8200 + M)
        h.profile_read()  # drop older records
        n0 = h.launch_count
        h.set_profiling(True)
        try:
            steps = 3
            for _ in range(steps):
                _run(h, L, dev_w, hbits)
            prof = h.profile_read()
        finally:
            h.set_profiling(False)
        assert set(prof) == tags, f"M={M}: {sorted(prof)}"
        assert all(n == steps for n, _ in prof.values()), prof
        assert all(ms > 0 for _, ms in prof.values()), prof
        assert h.launch_count - n0 == steps * len(tags)


def test_prefetch_l2_and_setting_arguments(h):
    import torch
    import moe_layers_gb300 as ML
    t = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    ML.dec_prefetch_l2(h, t)
    ML.dec_prefetch_l2(h, t, nbytes=4096)
    torch.cuda.synchronize()
    bad = [
        lambda: ML.dec_prefetch_l2(h, t, nbytes=100),     # not a multiple of 16
        lambda: ML.dec_prefetch_l2(h, t[1:], nbytes=16),  # not 16-byte aligned
        lambda: h.set_l2_ahead(-1),
        lambda: h.set_l2_ahead((16 << 20) + 1),
        lambda: h.set_shared_sms(-2),
        lambda: h.set_shared_sms(10 ** 6),
    ]
    for i, f in enumerate(bad):
        with pytest.raises(ML.DecodeError):
            f()
    assert h.check_device_error() == ML.DEC_OK
