"""The projection entry point that allocates nothing (dec_linear_noalloc).

It serves callers that cannot give the library any device memory: a plugin
inside a runtime whose memory pool owns the GPU, or a latency-critical caller
that must not call cudaMalloc. Its scratch is a static array inside the
library, shared by all calls, so this checks two calls in a row against the
workspace-based entry point (dec_linear / dec_linear_residual, the same
split-K kernel), with the tolerance used by every bf16 test here. This file
sorts last so that a stop-at-first-failure run has run everything else first;
it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import SEED, assert_bf16_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def test_no_alloc_entry_point_matches_workspace_entry_point():
    import torch
    import moe_layers_gb300 as ML
    assert torch.cuda.is_available()
    ML.build()
    with ML.Handle(0) as h:
        # two calls in a row, second with a residual; both shapes are split-K shapes under the
        # automatic choice (batch 8; batch 3 with a 67 MB matrix)
        cases = [(8, 1000, 520, False), (3, 4096, 8192, True)]
        for i, (M, N, K, resid) in enumerate(cases):
            x = synth.bf16(M * K, SEED, 9100 + i, 0, 1.0).reshape(M, K)
            W = synth.bf16(N * K, SEED, 9110 + i, 0, 0.02).reshape(N, K)
            xd, Wd = dev_bf16(x, (M, K)), dev_bf16(W, (N, K))
            if resid:
                r = synth.bf16(M * N, SEED, 9120 + i, 0, 1.0).reshape(M, N)
                rd = dev_bf16(r, (M, N))
                want = ML.dec_linear_residual(h, xd, Wd, rd)
                got = ML.dec_linear_noalloc(h, xd, Wd, r=rd)
                exact = oracle.linear_residual(x, W, r)
            else:
                want = ML.dec_linear(h, xd, Wd)
                got = ML.dec_linear_noalloc(h, xd, Wd)
                exact = oracle.linear(x, W)
            torch.cuda.synchronize()
            assert h.last_variant == ML.VARIANT_SPLIT_K
            gb, wb = host_bits(got), host_bits(want)
            assert_bf16_close(gb, oracle.bf16_to_f64(wb), f"no-alloc vs workspace entry point, call {i + 1}")
            assert_bf16_close(gb, exact, f"no-alloc vs oracle, call {i + 1}")
        assert h.check_device_error() == ML.DEC_OK


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    import torch
    import moe_layers_gb300 as ML
    ML.build()
    with ML.Handle(0) as h:
        x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
        W = torch.zeros((131073, 64), dtype=torch.bfloat16, device="cuda")  # N above the 131072-row limit
        with pytest.raises(ML.DecodeError) as e:
            ML.dec_linear_noalloc(h, x, W)
        assert e.value.status == ML.DEC_ERR_UNSUPPORTED
        # M above 64 breaks the shape rules every projection entry point shares
        x65 = torch.zeros((65, 64), dtype=torch.bfloat16, device="cuda")
        W1 = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(ML.DecodeError) as e:
            ML.dec_linear_noalloc(h, x65, W1)
        assert e.value.status == ML.DEC_ERR_INVALID_ARG
