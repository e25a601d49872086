"""Host logic of bench.py's roofline accounting (no GPU): the algorithmic
bytes credited to each launch of a one-token layer step add up to the step's
unique bytes under every schedule of the shared expert, at the full and the
tensor-parallel shard shapes, and the traffic record is reported only while
its sources are unchanged."""
import importlib

import pytest


@pytest.fixture()
def bench():
    import bench as b
    b = importlib.reload(b)  # (module-level shapes: start from the full workload)
    yield b
    importlib.reload(b)


# the launches of a one-token step under each schedule, by profiling tag
SCHEDULES = {
    "front": ("in_proj", "out_proj", "moe_front", "down"),
    "router": ("in_proj", "out_proj", "router", "gate_up", "down"),
    "gate_up": ("in_proj", "out_proj", "router", "gate_up", "down"),
}


@pytest.mark.parametrize("shard", [1, 8, 16])
@pytest.mark.parametrize("shared_in", list(SCHEDULES))
def test_one_token_launch_bytes_add_up_to_the_step(bench, shard, shared_in):
    if shard > 1:
        bench.set_shard(shard)
    U = float(bench.TOPK)
    total = sum(bench.kernel_bytes(tag, 1, U, shared_in) for tag in SCHEDULES[shared_in])
    step = bench.step_bytes(1, U)
    # every weight byte once; the launches also credit the intermediate
    # activations they read and write, which the step's unique bytes leave out
    # (0.4% at the shard shapes)
    weights = bench.DENSE_BYTES + (U + 1) * bench.EXPERT_BYTES
    assert total >= weights
    assert abs(total - step) <= 1e-2 * step, (total, step)


def test_front_credits_every_moe_weight_byte_once(bench):
    U = float(bench.TOPK)
    front = bench.kernel_bytes("moe_front", 1, U, "front")
    down = bench.kernel_bytes("down", 1, U, "front")
    router_w = bench.E * bench.H * 4
    gate_up_w = (U + 1) * 2 * bench.I * bench.H * 2  # routed and shared gate/up
    down_w = (U + 1) * bench.H * bench.I * 2
    assert front - router_w - gate_up_w == pytest.approx(0, abs=1e6)
    assert down - down_w == pytest.approx(0, abs=1e6)


def test_traffic_record_follows_its_sources(bench, tmp_path, monkeypatch):
    tag, M = next(iter(bench.NCU_TRAFFIC))
    rec = bench.NCU_TRAFFIC[(tag, M)]
    assert bench.captured_traffic(tag, M) in (rec["bytes"], None)  # (null once a source has changed)
    assert bench.captured_traffic("no_such_kernel", 1) is None
    monkeypatch.setitem(bench.NCU_TRAFFIC, (tag, M), dict(rec, sha256="0" * 64))
    assert bench.captured_traffic(tag, M) is None  # any change to the sources voids it
