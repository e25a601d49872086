"""GPU parity of the projections (dec_linear, dec_linear_residual) and
RMSNorm against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from _util import SEED, assert_bf16_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


@pytest.fixture(scope="module")
def h(torch_cuda):
    import moe_layers_gb300 as M
    M.build()
    with M.Handle(0) as hd:
        yield hd


def _mats(M, N, K, tid, sx=1.0, sw=0.02):
    x = synth.bf16(M * K, SEED, synth.W_LINEAR + tid, 0, sx).reshape(M, K)
    W = synth.bf16(N * K, SEED, synth.W_LINEAR + tid + 1, 0, sw).reshape(N, K)
    return x, W


SMALL = [(1, 200, 72), (2, 300, 136), (1, 7, 8), (2, 1, 4096), (3, 257, 520), (4, 130, 64), (5, 128, 1000),
         (16, 384, 704), (17, 129, 136), (33, 640, 1032), (48, 256, 512), (64, 520, 704), (64, 1, 64),
         # narrow rows (K <= 1024: 16 to 128 threads per row), incl. the TP8 / TP16 out-projection shapes
         (1, 7168, 1024), (1, 3001, 512), (2, 1000, 256), (4, 333, 1024), (3, 77, 128), (1, 7168, 512)]


@pytest.mark.parametrize("M,N,K", SMALL)
@pytest.mark.parametrize("variant", ["small_m", "split_k"])
def test_linear_small_shapes(h, M, N, K, variant):
    import moe_layers_gb300 as ML
    if variant == "small_m" and M > 4:
        pytest.skip("small-matrix kernel covers M <= 4")
    v = ML.VARIANT_SMALL_M if variant == "small_m" else ML.VARIANT_SPLIT_K
    h.set_force_variant(v)
    try:
        x, W = _mats(M, N, K, 2 * (M * 1000 + K % 97))
        y = ML.dec_linear(h, dev_bf16(x, (M, K)), dev_bf16(W, (N, K)))
        assert h.last_variant == v
        assert_bf16_close(host_bits(y), oracle.linear(x, W), f"linear {variant} M={M} N={N} K={K}")
    finally:
        h.set_force_variant(ML.VARIANT_AUTO)


@pytest.mark.parametrize("M", [1, 2, 3, 8, 64])
def test_linear_integer_exact_bit_for_bit(h, M):
    # Small integers times 2^-4: every product and partial sum is exact in fp32,
    # so the kernels must return the correctly rounded exact value, bit for bit.
    import moe_layers_gb300 as ML
    N, K = 384, 512
    rng = np.random.default_rng(M)
    xi = rng.integers(-8, 9, size=(M, K))
    wi = rng.integers(-8, 9, size=(N, K))
    to_bits = lambda a: (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x, W = to_bits(xi / 16.0), to_bits(wi / 16.0)
    exact = oracle.linear(x, W)
    want = (oracle.round_bf16(exact).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    for v in ([ML.VARIANT_SMALL_M] if M <= 4 else []) + [ML.VARIANT_SPLIT_K]:
        h.set_force_variant(v)
        try:
            y = ML.dec_linear(h, dev_bf16(x, (M, K)), dev_bf16(W, (N, K)))
            assert np.array_equal(host_bits(y), want), f"variant {v}"
        finally:
            h.set_force_variant(ML.VARIANT_AUTO)


@pytest.mark.parametrize("M", [1, 2, 4, 64])
@pytest.mark.parametrize("N,K", [(520, 704), (1001, 4096), (1000, 8192)])
def test_linear_residual_and_alias(h, M, N, K):
    """Residual add, also in place. On the split-K kernel (M > 2) the shapes
    split every 128-row tile into pieces over several CTAs, so the tile is
    finished by the reduction of its pieces, with the residual rows staged in
    shared memory (N a multiple of 8) or read from global memory (N = 1001)."""
    import moe_layers_gb300 as ML
    x, W = _mats(M, N, K, 700 + M + N)
    r = synth.bf16(M * N, SEED, synth.R_BASE + M, 0, 1.0).reshape(M, N)
    ref = oracle.linear_residual(x, W, r)
    out = ML.dec_linear_residual(h, dev_bf16(x, (M, K)), dev_bf16(W, (N, K)), dev_bf16(r, (M, N)))
    assert_bf16_close(host_bits(out), ref, "residual")
    rr = dev_bf16(r, (M, N))
    ML.dec_linear_residual(h, dev_bf16(x, (M, K)), dev_bf16(W, (N, K)), rr, out=rr)  # out aliases r
    assert_bf16_close(host_bits(rr), ref, "residual in place")


@pytest.mark.parametrize("M", [1, 2, 5, 64])
def test_linear_strided_activation(h, M):
    # x is the leading K columns of a wider [M, ld] activation (the out-projection reads y_in[:, :K_out]).
    import moe_layers_gb300 as ML
    N, K, ld = 256, 512, 776
    wide = synth.bf16(M * ld, SEED, 900 + M, 0, 1.0).reshape(M, ld)
    W = synth.bf16(N * K, SEED, 901, 0, 0.02).reshape(N, K)
    xd = dev_bf16(wide, (M, ld))[:, :K]
    y = ML.dec_linear(h, xd, dev_bf16(W, (N, K)))
    assert_bf16_close(host_bits(y), oracle.linear(wide[:, :K], W), "strided x")


# ---------------------------------------------------------------------------- workload sizes
@pytest.fixture(scope="module")
def w_in():
    return synth.bf16(12288 * 7168, SEED, synth.W_IN, 0, 0.02).reshape(12288, 7168)


def test_single_decode_projection_4096(h):
    import moe_layers_gb300 as ML
    x = synth.bf16(4096, SEED, synth.row_tensor_id(synth.X_BASE, 0), 0, 1.0).reshape(1, 4096)
    W = synth.bf16(4096 * 4096, SEED, synth.W_LINEAR, 0, 0.02).reshape(4096, 4096)
    y = ML.dec_linear(h, dev_bf16(x, (1, 4096)), dev_bf16(W, (4096, 4096)))
    assert h.last_variant == ML.VARIANT_SMALL_M
    assert_bf16_close(host_bits(y), oracle.linear(x, W), "4096x4096 M=1")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
def test_input_projection_batch_sweep(h, w_in, M):
    import moe_layers_gb300 as ML
    x = synth.bf16_rows(synth.X_BASE, range(M), 7168, SEED)
    Wd = dev_bf16(w_in, (12288, 7168))
    y = ML.dec_linear(h, dev_bf16(x, (M, 7168)), Wd)
    # automatic choice: the small-matrix kernel up to two tokens (a 176 MB matrix), split-K above
    assert h.last_variant == (ML.VARIANT_SMALL_M if M <= 2 else ML.VARIANT_SPLIT_K)
    assert_bf16_close(host_bits(y), oracle.linear(x, w_in), f"in-proj M={M}")


@pytest.mark.parametrize("N,K", [(3001, 7168), (4096, 4096), (1000, 1024)])
def test_mixed_precision_fma_matches_widened(h, N, K):
    """The two-token small-matrix kernel multiplies bf16 operands with fp32
    fused multiply-adds (fma.rn.f32.bf16); the one-token kernel widens them to
    fp32 first. The product of two bf16 values is exact in fp32 and the
    per-row reduction order is the same, so two copies of a token must give
    the one-token output bit for bit. The narrow kernel (K <= 1024) takes the
    mixed form at every batch, so there the two calls are compared with the
    oracle only."""
    import moe_layers_gb300 as ML
    x1, W = _mats(1, N, K, 820 + K % 97)
    x2 = np.concatenate([x1, x1], axis=0)
    Wd = dev_bf16(W, (N, K))
    h.set_force_variant(ML.VARIANT_SMALL_M)
    try:
        y1 = host_bits(ML.dec_linear(h, dev_bf16(x1, (1, K)), Wd))
        y2 = host_bits(ML.dec_linear(h, dev_bf16(x2, (2, K)), Wd))
    finally:
        h.set_force_variant(ML.VARIANT_AUTO)
    ref = oracle.linear(x1, W)
    assert_bf16_close(y1, ref, f"M=1 N={N} K={K}")
    assert_bf16_close(y2[1:], ref, f"M=2 N={N} K={K}")
    assert np.array_equal(y2[0], y2[1]), "the two copies of the token differ"
    if K > 1024:
        assert np.array_equal(y1[0], y2[0]), "mixed-precision FMA differs from the widened form"


@pytest.mark.parametrize("M,N,K,resid", [(16, 1000, 8192, True), (64, 520, 4096, False), (4, 1001, 4096, True),
                                          (3, 128, 8192, True)])
def test_split_tile_finish_paths_give_the_same_bits(h, M, N, K, resid):
    """The split-K kernel's three ways of finishing a tile split between CTAs
    add the same fp32 partials in the same k order, so the outputs agree bit
    for bit: the first piece's CTA from shared memory (default), the CTA that
    completes the count (mode 1), and the same with the pieces read from L2
    (mode 2). The shapes split tiles over two to many CTAs, with the residual
    staged in shared memory (N a multiple of 8) or read from global memory."""
    import moe_layers_gb300 as ML
    x, W = _mats(M, N, K, 960 + M + N)
    r = synth.bf16(M * N, SEED, 970 + M, 0, 1.0).reshape(M, N) if resid else None
    with pytest.raises(ML.DecodeError):
        h.test_set_engine_finish(3)
    outs = []
    h.set_force_variant(ML.VARIANT_SPLIT_K)
    try:
        for mode in (0, 1, 2):
            h.test_set_engine_finish(mode)
            if resid:
                y = ML.dec_linear_residual(h, dev_bf16(x, (M, K)), dev_bf16(W, (N, K)), dev_bf16(r, (M, N)))
            else:
                y = ML.dec_linear(h, dev_bf16(x, (M, K)), dev_bf16(W, (N, K)))
            outs.append(host_bits(y))
    finally:
        h.test_set_engine_finish(0)
        h.set_force_variant(ML.VARIANT_AUTO)
    ref = oracle.linear_residual(x, W, r) if resid else oracle.linear(x, W)
    assert_bf16_close(outs[0], ref, f"split-K M={M} N={N} K={K}")
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2]), "finish paths differ"


def test_automatic_choice_by_size(h):
    """Up to four tokens a matrix of at most 48 MB stays on the small-matrix
    kernel (the split-K kernel's per-launch cost outweighs its rate there)."""
    import moe_layers_gb300 as ML
    for (M, N, K, want) in [(3, 1536, 7168, ML.VARIANT_SMALL_M), (4, 7168, 1024, ML.VARIANT_SMALL_M),
                            (3, 7168, 8192, ML.VARIANT_SPLIT_K), (5, 1536, 7168, ML.VARIANT_SPLIT_K)]:
        x = synth.bf16(M * K, SEED, 950 + M, 0, 1.0).reshape(M, K)
        W = synth.bf16(N * K, SEED, 951, 0, 0.02).reshape(N, K)
        y = ML.dec_linear(h, dev_bf16(x, (M, K)), dev_bf16(W, (N, K)))
        assert h.last_variant == want, (M, N, K)
        assert_bf16_close(host_bits(y), oracle.linear(x, W), f"auto M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_out_projection_residual_full(h, M):
    import moe_layers_gb300 as ML
    W = synth.bf16(7168 * 8192, SEED, synth.W_O, 0, 0.02).reshape(7168, 8192)
    x = synth.bf16_rows(synth.X_BASE + 1, range(M), 8192, SEED)
    r = synth.bf16_rows(synth.R_BASE, range(M), 7168, SEED)
    out = ML.dec_linear_residual(h, dev_bf16(x, (M, 8192)), dev_bf16(W, (7168, 8192)), dev_bf16(r, (M, 7168)))
    assert_bf16_close(host_bits(out), oracle.linear_residual(x, W, r), f"out-proj M={M}")


# ---------------------------------------------------------------------------- rmsnorm
@pytest.mark.parametrize("M,H", [(1, 7168), (3, 256), (64, 7168), (2, 8)])
def test_rmsnorm(h, M, H):
    import moe_layers_gb300 as ML
    x = synth.bf16(M * H, SEED, 950 + M, 0, 1.0).reshape(M, H)
    g = synth.bf16(H, SEED, 951, 0, 0.1)
    gam = oracle.round_bf16(1.0 + oracle.bf16_to_f64(g))
    gbits = (gam.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y = ML.dec_rmsnorm(h, dev_bf16(x, (M, H)), dev_bf16(gbits, (H,)))
    assert_bf16_close(host_bits(y), oracle.rmsnorm(x, gbits), "rmsnorm")
    xd = dev_bf16(x, (M, H))
    ML.dec_rmsnorm(h, xd, dev_bf16(gbits, (H,)), y=xd)  # in place
    assert_bf16_close(host_bits(xd), oracle.rmsnorm(x, gbits), "rmsnorm in place")


# ---------------------------------------------------------------------------- ordering and failure paths
@pytest.mark.parametrize("M", [1, 8])
def test_dependent_launch_reads_activations_after_the_wait(h, M, torch_cuda):
    # A slow producer writes x 200 us after it starts; the projection is launched
    # programmatically dependent on it and may start early, streaming weights.
    # If any activation read were hoisted above the dependency wait, the result
    # would use the stale (zero) x.
    import moe_layers_gb300 as ML
    torch = torch_cuda
    N, K = 4096, 4096
    x, W = _mats(M, N, K, 1200 + M)
    ref = oracle.linear(x, W)
    Wd = dev_bf16(W, (N, K))
    src = dev_bf16(x, (M, K))
    h.set_pdl(True)
    for _ in range(3):
        dst = torch.zeros_like(src)
        ML.test_delayed_copy(h, dst, src, 200_000)
        y = ML.dec_linear(h, dst, Wd)
        assert_bf16_close(host_bits(y), ref, "pdl ordering")


def test_wait_timeout_surfaces_as_status(h, torch_cuda):
    import moe_layers_gb300 as ML
    assert h.check_device_error() == ML.DEC_OK
    h.set_wait_limit_ns(2_000_000)
    try:
        ML.test_wait_timeout(h)
        assert h.check_device_error() == ML.DEC_ERR_TIMEOUT
        assert h.check_device_error() == ML.DEC_OK  # cleared
    finally:
        h.set_wait_limit_ns(500_000_000)
    # the context is still usable
    x, W = _mats(3, 256, 512, 1300)
    y = ML.dec_linear(h, dev_bf16(x, (3, 512)), dev_bf16(W, (256, 512)))
    assert_bf16_close(host_bits(y), oracle.linear(x, W), "after timeout")


@pytest.mark.parametrize("tokens", [1, 2])
def test_routing_wait_timeout_surfaces_as_status(h, torch_cuda, tokens):
    """The MoE front's CTAs wait for the routing flag with a bounded wait: on a
    problem whose hand-off never completes (nothing sets the flag) every CTA
    gives up after the limit, the error word reads DEC_ERR_TIMEOUT, and the
    context stays usable."""
    import moe_layers_gb300 as ML
    assert h.check_device_error() == ML.DEC_OK
    h.set_wait_limit_ns(2_000_000)
    try:
        ML.test_routing_wait_timeout(h, tokens)
        assert h.check_device_error() == ML.DEC_ERR_TIMEOUT
        assert h.check_device_error() == ML.DEC_OK  # cleared
    finally:
        h.set_wait_limit_ns(500_000_000)
    with pytest.raises(ML.DecodeError):
        ML.test_routing_wait_timeout(h, 3)
    x, W = _mats(2, 256, 512, 1310)
    y = ML.dec_linear(h, dev_bf16(x, (2, 512)), dev_bf16(W, (256, 512)))
    assert_bf16_close(host_bits(y), oracle.linear(x, W), "after the routing timeout")


def test_bad_arguments_launch_nothing(h, torch_cuda):
    import moe_layers_gb300 as ML
    torch = torch_cuda
    x = torch.zeros((65, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ML.DecodeError) as e:
        ML.dec_linear(h, x, W)  # M > 64
    assert e.value.status == ML.DEC_ERR_INVALID_ARG
    x = torch.zeros((2, 60), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((8, 60), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ML.DecodeError):
        ML.dec_linear(h, x, W)  # K % 8 != 0
    x = torch.zeros((2, 65), dtype=torch.bfloat16, device="cuda")[:, 1:]
    W = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ML.DecodeError):
        ML.dec_linear(h, x, W)  # misaligned x
    assert h.check_device_error() == ML.DEC_OK
