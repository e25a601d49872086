"""The seeded input generator: determinism, addressing, distribution, rounding."""
import math
from fractions import Fraction

import numpy as np
import pytest

import synth


def test_deterministic_and_keyed():
    a = synth.bf16(10000, 0, 7)
    assert np.array_equal(a, synth.bf16(10000, 0, 7))
    assert not np.array_equal(a, synth.bf16(10000, 0, 8))
    assert not np.array_equal(a, synth.bf16(10000, 1, 7))


def test_offset_addressing():
    full = synth.bf16(5000, 3, 11, 0, 0.02)
    part = synth.bf16(1000, 3, 11, 2500, 0.02)
    assert np.array_equal(full[2500:3500], part)
    f = synth.f32(3000, 3, 12, 0, 0.01)
    assert np.array_equal(f[1000:2000], synth.f32(1000, 3, 12, 1000, 0.01))


def test_thread_count_does_not_change_values():
    import ctypes
    lib = synth._host_lib()
    n = 300000
    outs = []
    for nt in (1, 3, 8):
        o = np.empty(n, dtype=np.uint16)
        lib.synth_fill_bf16(o.ctypes.data, n, 5, 9, 17, ctypes.c_double(1.0), nt)
        outs.append(o)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_normal_moments():
    z = synth.normals(1 << 20, 0, 3)
    n = z.size
    assert abs(z.mean()) < 5 / math.sqrt(n)
    assert abs(z.var() - 1.0) < 5 * math.sqrt(2.0 / n)
    # Irwin-Hall(12): kurtosis 3 - 6/(5*12) = 2.9, support within +-6
    kurt = np.mean(z ** 4) / z.var() ** 2
    assert abs(kurt - 2.9) < 0.02
    assert np.max(np.abs(z)) <= 6.0
    # values are exact multiples of 2^-17
    assert np.all(np.round(z * 2 ** 17) == z * 2 ** 17)


def test_scaled_bf16_distribution():
    bits = synth.bf16(1 << 18, 0, 4, 0, 0.02)
    v = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(v.std() - 0.02) < 0.0005
    assert abs(v.mean()) < 0.0005


def _ref_round(v: float, mbits: int) -> int:
    """Nearest-even rounding of v to sign/8-bit-exponent/mbits format, by exact rationals."""
    if v == 0:
        return 0
    sign = 1 if v < 0 else 0
    a = Fraction(abs(v))
    e = math.floor(math.log2(abs(v)))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = a / Fraction(2) ** (e - mbits)
    fl = math.floor(q)
    r = q - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    if fl >= 2 ** (mbits + 1):
        fl //= 2
        e += 1
    if fl < 2 ** mbits:  # subnormal
        return (sign << (8 + mbits)) | fl
    return (sign << (8 + mbits)) | ((e + 127) << mbits) | (fl - 2 ** mbits)


def test_rounding_matches_exact_rationals():
    rng = np.random.default_rng(0)
    vals = list(rng.standard_normal(3000) * 0.05) + list(rng.standard_normal(500) * 1e3)
    # ties: exact midpoints between bf16 neighbours, both parities
    for base in (1.0, 1.0078125, 0.5, 3.0):
        vals += [base + 2 ** -8 * (1 if base < 2 else 2), -(base + 2 ** -8)]
    vals += [2 ** -130, 3 * 2 ** -140, 1.0 - 2 ** -30]
    for v in vals:
        assert synth.round_bits(v, 7) == _ref_round(v, 7), v
        assert synth.round_bits(v, 23) == _ref_round(v, 23), v
        # binary32 also against numpy's IEEE conversion
        if abs(v) > 2 ** -120:
            assert synth.round_bits(v, 23) == int(np.float32(v).view(np.uint32)), v


def test_splitmix_stream_definition():
    # Output n of SplitMix64 from state s: mix(s + (n+1) * golden gamma), arithmetic mod 2^64.
    M = (1 << 64) - 1
    def mix(z):
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
        return z ^ (z >> 31)
    for key in (0, 1, 0xDEADBEEF12345678, M):
        for n in (0, 1, 2, 1000, 1 << 40):
            assert synth.stream_u64(key, n) == mix((key + (n + 1) * 0x9E3779B97F4A7C15) & M)


def test_correlated_rows_groups():
    """Rows of a group share their base row: correlated within a group,
    independent across groups, deterministic, and bf16 of the stated sum."""
    import numpy as np
    H = 4096
    r = synth.correlated_rows(1000, range(16), 8, H, 0, 0.5)
    assert r.shape == (16, H) and r.dtype == np.uint16
    assert np.array_equal(r, synth.correlated_rows(1000, range(16), 8, H, 0, 0.5))
    f = (r.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    c = np.corrcoef(f)
    within = [c[i, j] for i in range(16) for j in range(16) if i != j and i // 8 == j // 8]
    across = [c[i, j] for i in range(16) for j in range(16) if i // 8 != j // 8]
    assert min(within) > 0.75 and max(abs(x) for x in across) < 0.1  # 1 / (1 + 0.25) = 0.8
    b = (synth.bf16(H, 0, synth.row_tensor_id(1000, 0, 0), 0, 1.0).astype(np.uint32) << 16).view(np.float32)
    n = (synth.bf16(H, 0, synth.row_tensor_id(1001, 3, 0), 0, 1.0).astype(np.uint32) << 16).view(np.float32)
    want = (b + np.float32(0.5) * n).astype(np.float32)
    got = (r[3].astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-30)  # within half a bf16 ulp
