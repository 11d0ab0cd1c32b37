"""CPU oracle for the quantized-weight GEMV library.  TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct statement of what the hot path computes, in
fp64 except where the method fixes fp32 (the activation scale and the int8
decision).  It is written in C (``oracle.c``, compiled with gcc on first use)
and shares no code with the CUDA library.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package; the library itself never does.

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against something other than itself (closed forms, brute force on tiny
inputs, textbook matrices, exhaustive enumeration, library routines).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc if it is missing or older than its source."""
    with _lock:
        if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
            os.makedirs(_BUILD, exist_ok=True)
            tmp = _SO + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", *ORACLE_CFLAGS, "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        i64, vp, dbl, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
        lib.or_half_to_double.argtypes = [ctypes.c_uint16]
        lib.or_half_to_double.restype = dbl
        lib.or_quantize_act.argtypes = [vp, i64, vp, vp, vp]
        lib.or_q4_code.argtypes = [vp, i64]
        lib.or_q4_code.restype = c_int
        lib.or_q6_code.argtypes = [vp, vp, i64]
        lib.or_q6_code.restype = c_int
        lib.or_q2_code.argtypes = [vp, i64]
        lib.or_q2_code.restype = c_int
        lib.or_codes.argtypes = [c_int, vp, vp, i64, i64, i64, vp]
        lib.or_dequant_rows.argtypes = [c_int, vp, vp, vp, vp, i64, i64, i64, vp]
        lib.or_blockdots.argtypes = [c_int, vp, vp, i64, i64, vp, vp]
        lib.or_gemv.argtypes = [c_int, vp, vp, vp, vp, i64, vp, i64, i64, vp, vp, vp, vp]
        lib.or_gemv_rows.argtypes = [c_int, vp, vp, vp, vp, i64, vp, vp, i64, vp, vp, vp, vp]
        lib.or_softcap.argtypes = [dbl, dbl]
        lib.or_softcap.restype = dbl
        lib.or_softcap_vec.argtypes = [vp, i64, dbl, vp]
        lib.or_argmax_f64.argtypes = [vp, i64]
        lib.or_argmax_f64.restype = i64
        lib.or_argmax_f32.argtypes = [vp, i64]
        lib.or_argmax_f32.restype = i64
        lib.or_wht.argtypes = [vp, i64, vp]
        lib.or_cq_matvec.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp, vp, vp]
        lib.or_logsumexp.argtypes = [vp, i64]
        lib.or_logsumexp.restype = dbl
        lib.or_select.argtypes = [vp, i64, vp, i64, vp]
        lib.or_select.restype = i64
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits: int) -> float:
    return float(_load().or_half_to_double(int(bits)))


def quantize_act(x: np.ndarray):
    """Per-block int8 activation quantisation: returns (xq int8 [k], s fp32 [k/32], S int32 [k/32])."""
    x = _c(x, np.float32)
    k = x.size
    assert k % 32 == 0
    xq = np.empty(k, np.int8)
    s = np.empty(k // 32, np.float32)
    S = np.empty(k // 32, np.int32)
    _load().or_quantize_act(_p(x), k, _p(xq), _p(s), _p(S))
    return xq, s, S


def _planes(w: dict):
    lo = _c(w["lo"], np.uint8)
    hi = _c(w["hi"], np.uint8) if w["bits"] == 6 else None
    mn = _c(w["min"], np.uint16) if w["bits"] != 2 else None  # Q2: zero point 2, no min plane
    return lo, hi, _c(w["scale"], np.uint16), mn


def codes(w: dict, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Integer codes [nrows][k] decoded from the packed planes."""
    lo, hi, _, _ = _planes(w)
    k = w["k"]
    nrows = w["n"] - row0 if nrows is None else nrows
    out = np.empty((nrows, k), np.int32)
    _load().or_codes(w["bits"], _p(lo), _p(hi), k, row0, nrows, _p(out))
    return out


def dequant(w: dict, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Dequantised weights scale*code + min, fp64 [nrows][k]."""
    lo, hi, sc, mn = _planes(w)
    k = w["k"]
    nrows = w["n"] - row0 if nrows is None else nrows
    out = np.empty((nrows, k), np.float64)
    _load().or_dequant_rows(w["bits"], _p(lo), _p(hi), _p(sc), _p(mn), k, row0, nrows, _p(out))
    return out


def blockdots(w: dict, xq: np.ndarray) -> np.ndarray:
    """Exact integer block dots D [n][k/32] of the codes with int8 xq."""
    lo, hi, _, _ = _planes(w)
    n, k = w["n"], w["k"]
    xq = _c(xq, np.int8)
    out = np.empty((n, k // 32), np.int32)
    _load().or_blockdots(w["bits"], _p(lo), _p(hi), n, k, _p(xq), _p(out))
    return out


def gemv(w: dict, x: np.ndarray, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """y (fp64) for rows [row0, row0+nrows): fp64 dequantised weights dotted with the int8-dequantised x."""
    lo, hi, sc, mn = _planes(w)
    k = w["k"]
    x = _c(x, np.float32)
    assert x.size == k
    nrows = w["n"] - row0 if nrows is None else nrows
    y = np.empty(nrows, np.float64)
    xq = np.empty(k, np.int8)
    s = np.empty(k // 32, np.float32)
    S = np.empty(k // 32, np.int32)
    _load().or_gemv(w["bits"], _p(lo), _p(hi), _p(sc), _p(mn), k, _p(x), row0, nrows, _p(y), _p(xq), _p(s), _p(S))
    return y


def gemv_rows(w: dict, x: np.ndarray, rows) -> np.ndarray:
    """y (fp64) at an explicit list of rows."""
    lo, hi, sc, mn = _planes(w)
    k = w["k"]
    x = _c(x, np.float32)
    rows = _c(rows, np.int64)
    y = np.empty(rows.size, np.float64)
    xq = np.empty(k, np.int8)
    s = np.empty(k // 32, np.float32)
    S = np.empty(k // 32, np.int32)
    _load().or_gemv_rows(w["bits"], _p(lo), _p(hi), _p(sc), _p(mn), k, _p(x), _p(rows), rows.size, _p(y), _p(xq),
                         _p(s), _p(S))
    return y


def gemv_batched(w: dict, X: np.ndarray) -> np.ndarray:
    """Y [B][n] (fp64): each activation column quantised and dotted on its own."""
    X = np.atleast_2d(_c(X, np.float32))
    return np.stack([gemv(w, X[b]) for b in range(X.shape[0])])


def gemv_chain(mats, src, inputs, gemv_fn=None):
    """Outputs (fp64, one per GEMV) of GEMVs run in order, each on an earlier one's output.

    Decode runs its projections back to back: what one matrix-vector product writes
    is the vector the next one quantises and reads (genie-ai-runtime, "The decode
    arc": the activation is quantised per matmul; Gemma WebGPU Engine, "Roadmap":
    a layer's ordered dispatches, each reading the buffer the previous one wrote).
    GEMV j reads
      src[j] >= 0 : the output of GEMV src[j] (src[j] < j), handed over as the fp32
                    vector a kernel writes, i.e. the fp64 result rounded to fp32;
      src[j] <  0 : the external fp32 vector inputs[-src[j] - 1].
    Each GEMV is ``gemv`` above (int8-quantised input, exact block dots, fp64 sum);
    ``gemv_fn`` may replace it by the same function evaluated over row slices in
    parallel, for large matrices.
    """
    gemv_fn = gemv if gemv_fn is None else gemv_fn
    outs = []
    for j, w in enumerate(mats):
        if src[j] >= 0:
            assert src[j] < j, "a GEMV reads only the outputs of earlier ones"
            x = outs[src[j]].astype(np.float32)
        else:
            x = np.asarray(inputs[-src[j] - 1], np.float32)
        outs.append(gemv_fn(w, x))
    return outs


def softcap(z, c: float) -> np.ndarray:
    z = _c(np.atleast_1d(z), np.float64)
    out = np.empty_like(z)
    _load().or_softcap_vec(_p(z), z.size, float(c), _p(out))
    return out


def argmax(v: np.ndarray) -> int:
    """Lowest index of the maximum; NaN never wins."""
    if v.dtype == np.float32:
        v = _c(v, np.float32)
        return int(_load().or_argmax_f32(_p(v), v.size))
    v = _c(v, np.float64)
    return int(_load().or_argmax_f64(_p(v), v.size))


def vocab_softcap_argmax(w: dict, x: np.ndarray, c: float):
    """(logits fp64 [n], argmax) of the soft-capped projection."""
    z = gemv(w, x)
    logits = softcap(z, c)
    return logits, argmax(logits)


def wht(x: np.ndarray) -> np.ndarray:
    """Normalised Walsh-Hadamard transform of one group (explicit O(g^2) sum)."""
    x = _c(x, np.float64)
    g = x.size
    assert g > 0 and g & (g - 1) == 0
    u = np.empty(g, np.float64)
    _load().or_wht(_p(x), g, _p(u))
    return u


def cq_matvec(m: dict, x: np.ndarray, group: int, row_start: int = 0, row_count: int | None = None) -> np.ndarray:
    """y (fp64) over rows [row_start, row_start+row_count) of a CQ matrix."""
    k = m["k"]
    x = _c(x, np.float32)
    assert x.size == k and k % group == 0
    row_count = m["n"] - row_start if row_count is None else row_count
    y = np.empty(row_count, np.float64)
    xw = np.empty(k, np.float64)
    uw = np.empty(k, np.float64)
    _load().or_cq_matvec(_p(_c(m["idx"], np.uint8)), _p(_c(m["codebook"], np.uint16)),
                         _p(_c(m["row_scale"], np.uint16)), k, group, row_start, row_count, _p(x), _p(y), _p(xw),
                         _p(uw))
    return y


def logsumexp(v) -> float:
    """log(sum(exp(v))) in fp64, NaN skipped."""
    v = _c(np.atleast_1d(v), np.float64)
    return float(_load().or_logsumexp(_p(v), v.size))


def select(v, allowed=None):
    """(id, logprob): the allowed id of the largest value (lowest id on ties) and
    v[id] - logsumexp(v); allowed=None means every id.  id = -1 if none qualifies."""
    v = _c(np.atleast_1d(v), np.float64)
    lp = ctypes.c_double(0.0)
    if allowed is None:
        idx = _load().or_select(_p(v), v.size, None, 0, ctypes.byref(lp))
    else:
        a = _c(np.atleast_1d(allowed), np.int32)
        idx = _load().or_select(_p(v), v.size, _p(a), a.size, ctypes.byref(lp))
    return int(idx), float(lp.value)


def normwise_error(y, ref) -> float:
    """max_i |y_i - ref_i| / max(|ref_i|, rms(ref)): the fp32-output error measure."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), rms)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(y - ref) / den))
