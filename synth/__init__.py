"""Seeded synthetic inputs for the MoE decode path (test and benchmark data).

Every tensor is defined by (seed, tensor id, element index) through the
counter-based stream in ``synth_arith.h``; the host filler (C, used for the
oracle's copies) and the device filler (CUDA, used to place the 30+ GB expert
bank in HBM quickly) compile the same arithmetic and agree bit for bit.

This module holds none of the decode path's arithmetic. It is shared by the
oracle side and the CUDA side only as a source of input bytes.

Input recipe (the workloads' shapes and distributions):

* activations x, h, residual r: N(0, 1) rounded to bf16;
* projection and expert weights: N(0, 0.02) rounded to bf16, nn.Linear
  layout ``[out_features, in_features]``; expert banks ``[E, I, H]`` for gate
  and up, ``[E, H, I]`` for down, one tensor id per bank;
* router weights: N(0, 0.01) rounded to fp32, ``[E, H]``;
* RMSNorm gains: ones (the graded layer), or 1 + N(0, 0.1) in unit tests.

"N(0, s)" is s times the Irwin-Hall(12) draw: mean 0, variance 1, tails cut
at six standard deviations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libsynth_host.so")
_DEV_SO = os.path.join(_HERE, "libsynth_dev.so")
_lock = threading.Lock()
_host = None
_dev = None

# Tensor ids of the decode-layer workload. Per-step activation sets use
# row_tensor_id(X_BASE + set, row, attempt).
W_IN, W_O, W_R, W_G, W_U, W_D, W_G_S, W_U_S, W_D_S, GAMMA1, GAMMA2 = range(1, 12)
X_BASE = 1000
R_BASE = 5000
W_LINEAR = 20  # single-projection workloads: W_LINEAR + k for the k-th matrix


def row_tensor_id(base: int, row: int, attempt: int = 0) -> int:
    """Tensor id of one activation row (rows are redrawn independently)."""
    return (int(base) << 40) | (int(attempt) << 20) | int(row)


def _newer(target: str, *sources: str) -> bool:
    return os.path.exists(target) and all(os.path.getmtime(target) >= os.path.getmtime(s) for s in sources)


def build_host() -> str:
    src = os.path.join(_HERE, "synth_host.c")
    hdr = os.path.join(_HERE, "synth_arith.h")
    if not _newer(_HOST_SO, src, hdr):
        tmp = _HOST_SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-ffp-contract=off", "-pthread",
                               src, "-o", tmp])
        os.replace(tmp, _HOST_SO)
    return _HOST_SO


def build_dev(arch: str = "103a") -> str:
    src = os.path.join(_HERE, "synth_dev.cu")
    hdr = os.path.join(_HERE, "synth_arith.h")
    if not _newer(_DEV_SO, src, hdr):
        tmp = _DEV_SO + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC,-ffp-contract=off", "-fmad=false",
                               f"-gencode=arch=compute_{arch},code=sm_{arch}", src, "-o", tmp])
        os.replace(tmp, _DEV_SO)
    return _DEV_SO


def _host_lib():
    global _host
    with _lock:
        if _host is None:
            lib = ctypes.CDLL(build_host())
            u64, dbl, i32 = ctypes.c_uint64, ctypes.c_double, ctypes.c_int
            lib.synth_fill_bf16.argtypes = [ctypes.c_void_p, u64, u64, u64, u64, dbl, i32]
            lib.synth_fill_f32.argtypes = [ctypes.c_void_p, u64, u64, u64, u64, dbl, i32]
            lib.synth_normals_f64.argtypes = [ctypes.c_void_p, u64, u64, u64, u64]
            lib.synth_round_bits.argtypes = [dbl, i32]
            lib.synth_round_bits.restype = ctypes.c_uint32
            lib.synth_stream_u64.argtypes = [u64, u64]
            lib.synth_stream_u64.restype = u64
            _host = lib
    return _host


def _dev_lib():
    global _dev
    with _lock:
        if _dev is None:
            lib = ctypes.CDLL(build_dev())
            u64, dbl = ctypes.c_uint64, ctypes.c_double
            for name in ("synth_fill_bf16_dev", "synth_fill_f32_dev"):
                f = getattr(lib, name)
                f.argtypes = [ctypes.c_void_p, u64, u64, u64, u64, dbl, ctypes.c_void_p]
                f.restype = ctypes.c_int
            _dev = lib
    return _dev


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def bf16(n: int, seed: int, tensor_id: int, offset: int = 0, sigma: float = 1.0) -> np.ndarray:
    """n bf16 values (as uint16 bit patterns) of sigma * N(0,1)."""
    out = np.empty(int(n), dtype=np.uint16)
    _host_lib().synth_fill_bf16(out.ctypes.data, int(n), int(seed), int(tensor_id), int(offset), float(sigma),
                                _threads())
    return out


def f32(n: int, seed: int, tensor_id: int, offset: int = 0, sigma: float = 1.0) -> np.ndarray:
    """n fp32 values of sigma * N(0,1)."""
    out = np.empty(int(n), dtype=np.uint32)
    _host_lib().synth_fill_f32(out.ctypes.data, int(n), int(seed), int(tensor_id), int(offset), float(sigma),
                               _threads())
    return out.view(np.float32)


def normals(n: int, seed: int, tensor_id: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float64)
    _host_lib().synth_normals_f64(out.ctypes.data, int(n), int(seed), int(tensor_id), int(offset))
    return out


def round_bits(v: float, mbits: int) -> int:
    return int(_host_lib().synth_round_bits(float(v), int(mbits)))


def stream_u64(key: int, n: int) -> int:
    return int(_host_lib().synth_stream_u64(int(key), int(n)))


def bf16_rows(base: int, rows, cols: int, seed: int, sigma: float = 1.0, attempts=None) -> np.ndarray:
    """Activation matrix whose row r is drawn from row_tensor_id(base, rows[r], attempts[r])."""
    rows = list(rows)
    attempts = [0] * len(rows) if attempts is None else list(attempts)
    out = np.empty((len(rows), cols), dtype=np.uint16)
    for i, (r, a) in enumerate(zip(rows, attempts)):
        out[i] = bf16(cols, seed, row_tensor_id(base, r, a), 0, sigma)
    return out


def correlated_rows(base: int, rows, group: int, cols: int, seed: int, eps: float, attempts=None) -> np.ndarray:
    """Activation rows in groups of `group` related rows (the draft tokens of
    one request in a speculative-verify batch): row r is
    bf16(b + eps * n_r), b the group's N(0, 1) row (row_tensor_id(base, r // group)),
    n_r an N(0, 1) row of its own (row_tensor_id(base + 1, r, attempt)), rounded
    to nearest-even bf16. Two rows of one group have correlation 1 / (1 + eps^2)."""
    rows = list(rows)
    attempts = [0] * len(rows) if attempts is None else list(attempts)
    out = np.empty((len(rows), cols), dtype=np.uint16)
    for i, (r, a) in enumerate(zip(rows, attempts)):
        b = _bits_to_f32(bf16(cols, seed, row_tensor_id(base, r // group, 0), 0, 1.0))
        n = _bits_to_f32(bf16(cols, seed, row_tensor_id(base + 1, r, a), 0, 1.0))
        out[i] = _f32_to_bf16_bits(b + np.float32(eps) * n)
    return out


def _bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def fill_bf16_dev(ptr: int, n: int, seed: int, tensor_id: int, offset: int = 0, sigma: float = 1.0,
                  stream: int = 0) -> None:
    """Fill n bf16 elements at device address ptr (same bits as bf16())."""
    rc = _dev_lib().synth_fill_bf16_dev(ctypes.c_void_p(ptr), int(n), int(seed), int(tensor_id), int(offset),
                                        float(sigma), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_bf16_dev failed: cuda error {rc}")


def fill_f32_dev(ptr: int, n: int, seed: int, tensor_id: int, offset: int = 0, sigma: float = 1.0,
                 stream: int = 0) -> None:
    rc = _dev_lib().synth_fill_f32_dev(ctypes.c_void_p(ptr), int(n), int(seed), int(tensor_id), int(offset),
                                       float(sigma), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_f32_dev failed: cuda error {rc}")
