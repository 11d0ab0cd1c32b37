"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark.

This module prepares inputs only: fp32 weights and activations drawn from a
counter-based generator, and the packing of weights into the Q4 / Q6 / CQ
block layouts.  None of the method's arithmetic lives here (no activation
quantisation, no dot products, no transform, no soft-cap or argmax); the
oracle and the CUDA kernels each implement that on their own.

The C source (``datagen.c``) states the generator and the layouts.  It is
compiled with gcc on first use into ``_build/`` beside this file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "datagen.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libdatagen.so")
_lock = threading.Lock()
_lib = None

GEN_CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]

# stream ids of the recipes below
STREAM_W = 0
STREAM_X = 1
STREAM_CODEBOOK = 2
STREAM_ROWSCALE = 3
STREAM_INDEX = 4


def build(force: bool = False) -> str:
    """Compile ``libdatagen.so`` (gcc) if it is missing or older than its source."""
    with _lock:
        if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
            os.makedirs(_BUILD, exist_ok=True)
            tmp = _SO + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", *GEN_CFLAGS, "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.dg_u64.argtypes = [u64, u64, u64]
        lib.dg_u64.restype = u64
        lib.dg_uniform.argtypes = [u64, u64, u64]
        lib.dg_uniform.restype = dbl
        lib.dg_normal.argtypes = [u64, u64, u64]
        lib.dg_normal.restype = dbl
        lib.dg_normal_f32.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
        lib.dg_uniform_f32.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
        lib.dg_f32_to_f16.argtypes = [vp, i64, vp]
        lib.dg_pack_q4_codes.argtypes = [vp, i64, i64, vp]
        lib.dg_pack_q6_codes.argtypes = [vp, i64, i64, vp, vp]
        lib.dg_pack_q2_codes.argtypes = [vp, i64, i64, vp]
        lib.dg_quantize_matrix.argtypes = [ctypes.c_int, vp, i64, i64, vp, vp, vp, vp]
        lib.dg_make_quantized.argtypes = [ctypes.c_int, u64, u64, i64, i64, dbl, vp, vp, vp, vp, ctypes.c_int]
        lib.dg_make_quantized.restype = ctypes.c_int
        lib.dg_weights_f32.argtypes = [u64, u64, i64, i64, i64, dbl, vp]
        lib.dg_make_cq_indices.argtypes = [u64, u64, i64, i64, vp]
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


# ---------------------------------------------------------------- primitives
def u64(seed: int, stream: int, i: int) -> int:
    return int(_load().dg_u64(seed, stream, i))


def uniform(seed: int, stream: int, i: int) -> float:
    return float(_load().dg_uniform(seed, stream, i))


def normal(seed: int, stream: int, i: int) -> float:
    return float(_load().dg_normal(seed, stream, i))


def normal_f32(seed: int, stream: int, n: int, offset: int = 0, mean: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().dg_normal_f32(seed, stream, offset, n, mean, sigma, _p(out))
    return out


def uniform_f32(seed: int, stream: int, n: int, offset: int = 0, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().dg_uniform_f32(seed, stream, offset, n, lo, hi, _p(out))
    return out


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().dg_f32_to_f16(_p(a), a.size, _p(out))
    return out


# ---------------------------------------------------------------- packers
def pack_q4_codes(q: np.ndarray) -> np.ndarray:
    """Pack codes (uint8 [n][k], values 0..15) into the Q4 byte layout [n][k/2]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    n, k = q.shape
    assert k % 32 == 0
    codes = np.empty((n, k // 2), dtype=np.uint8)
    _load().dg_pack_q4_codes(_p(q), n, k, _p(codes))
    return codes


def pack_q6_codes(q: np.ndarray):
    """Pack codes (uint8 [n][k], values 0..63) into the Q6 lo [n][k/2] and hi [n][k/4] planes."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    n, k = q.shape
    assert k % 32 == 0
    lo = np.empty((n, k // 2), dtype=np.uint8)
    hi = np.empty((n, k // 4), dtype=np.uint8)
    _load().dg_pack_q6_codes(_p(q), n, k, _p(lo), _p(hi))
    return lo, hi


def pack_q2_codes(q: np.ndarray) -> np.ndarray:
    """Pack codes (uint8 [n][k], values 0..3) into the Q2 byte layout [n][k/4]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    n, k = q.shape
    assert k % 32 == 0
    codes = np.empty((n, k // 4), dtype=np.uint8)
    _load().dg_pack_q2_codes(_p(q), n, k, _p(codes))
    return codes


def _alloc_planes(bits: int, n: int, k: int):
    if bits == 2:
        return np.empty((n, k // 4), np.uint8), None, np.empty((n, k // 32), np.uint16), None
    lo = np.empty((n, k // 2), dtype=np.uint8)
    hi = np.empty((n, k // 4), dtype=np.uint8) if bits == 6 else None
    return lo, hi, np.empty((n, k // 32), dtype=np.uint16), np.empty((n, k // 32), dtype=np.uint16)


def quantize_matrix(bits: int, w: np.ndarray) -> dict:
    """Block-quantise a caller-supplied fp32 matrix [n][k] to the Q4 / Q6 layout."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    assert bits in (2, 4, 6) and k % 32 == 0
    lo, hi, scale, mn = _alloc_planes(bits, n, k)
    _load().dg_quantize_matrix(bits, _p(w), n, k, _p(lo), _p(hi) if hi is not None else None, _p(scale),
                               _p(mn) if mn is not None else None)
    return {"bits": bits, "n": n, "k": k, "lo": lo, "hi": hi, "scale": scale, "min": mn}


def make_quantized(bits: int, seed: int, n: int, k: int, sigma: float = 0.02, stream: int = STREAM_W,
                   nthreads: int | None = None) -> dict:
    """Seeded matrix W[r][c] = f32(sigma * normal(seed, stream, r*k + c)), block-quantised."""
    assert bits in (2, 4, 6) and k % 32 == 0
    lo, hi, scale, mn = _alloc_planes(bits, n, k)
    rc = _load().dg_make_quantized(bits, seed, stream, n, k, sigma, _p(lo), _p(hi) if hi is not None else None,
                                   _p(scale), _p(mn) if mn is not None else None, nthreads or _threads())
    assert rc == 0
    return {"bits": bits, "n": n, "k": k, "lo": lo, "hi": hi, "scale": scale, "min": mn}


def weights_f32(seed: int, n_rows: int, k: int, row0: int = 0, sigma: float = 0.02, stream: int = STREAM_W) -> np.ndarray:
    """The unquantised fp32 weights behind :func:`make_quantized` for rows [row0, row0+n_rows)."""
    out = np.empty((n_rows, k), dtype=np.float32)
    _load().dg_weights_f32(seed, stream, row0, n_rows, k, sigma, _p(out))
    return out


def make_cq(seed: int, n: int, k: int, stream_base: int = 0) -> dict:
    """CQ matrix: 4-bit indices U{0..15}, 16-entry f16 codebook N(0, 0.05), f16 row scales 0.5 + U(0,1)."""
    assert k % 2 == 0
    idx = np.empty((n, k // 2), dtype=np.uint8)
    _load().dg_make_cq_indices(seed, STREAM_INDEX + stream_base, n, k, _p(idx))
    codebook = f32_to_f16_bits(normal_f32(seed, STREAM_CODEBOOK + stream_base, 16, sigma=0.05))
    row_scale = f32_to_f16_bits(uniform_f32(seed, STREAM_ROWSCALE + stream_base, n, lo=0.5, hi=1.5))
    return {"n": n, "k": k, "idx": idx, "codebook": codebook, "row_scale": row_scale}
