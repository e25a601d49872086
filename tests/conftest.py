import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size case (seconds to a minute)")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without a GPU is an error, not a skip: the CPU
    # suite deselects them with -m "not gpu".
    pass


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


# ---------------------------------------------------------------------------- workload-size weights (GPU tests)
E_FULL, H_FULL, I_FULL, K_FULL = 384, 7168, 2048, 8
N_IN_FULL, K_OUT_FULL = 12288, 8192


@pytest.fixture(scope="session")
def full_bank():
    """The 384-expert bank (about 34 GB) and the shared expert, placed in HBM by
    the seeded device filler (same bits as the host filler)."""
    import torch
    import synth
    n = E_FULL * I_FULL * H_FULL
    Wg = torch.empty((E_FULL, I_FULL, H_FULL), dtype=torch.bfloat16, device="cuda")
    Wu = torch.empty_like(Wg)
    Wd = torch.empty((E_FULL, H_FULL, I_FULL), dtype=torch.bfloat16, device="cuda")
    for t, tid in ((Wg, synth.W_G), (Wu, synth.W_U), (Wd, synth.W_D)):
        synth.fill_bf16_dev(t.data_ptr(), n, 0, tid, 0, 0.02)
    sh = []
    for tid, shape in ((synth.W_G_S, (I_FULL, H_FULL)), (synth.W_U_S, (I_FULL, H_FULL)),
                       (synth.W_D_S, (H_FULL, I_FULL))):
        t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        synth.fill_bf16_dev(t.data_ptr(), t.numel(), 0, tid, 0, 0.02)
        sh.append(t)
    torch.cuda.synchronize()
    yield Wg, Wu, Wd, tuple(sh)
    del Wg, Wu, Wd, sh
    torch.cuda.empty_cache()
