"""Python binding of ``libqgemv.so``, the quantized-weight GEMV library for GB300.

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream; tensors
are passed to the C ABI (``include/qgemv.h``) as raw device pointers.  The
functions carry the C names.  A missing library raises instead of falling back
to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB as LIB_PATH

QG_OK = 0
QG_ERR_INVALID_ARG = -1
QG_ERR_ALIGNMENT = -2
QG_ERR_UNSUPPORTED = -3
QG_ERR_WORKSPACE = -4
QG_ERR_CUDA = -5

QG_FLAG_PDL = 0x1
QG_FLAG_PLAIN = 0x2
QG_FLAG_CHAIN_PERSISTENT = 0x4
QG_CHAIN_CTL_BYTES = 256
QG_CHAIN_MAX_PHASE_K = 32768

# every exported function and its ctypes signature (restype, argtypes)
_u8p = _u16p = _f32p = _i8p = _i32p = _vp = ctypes.c_void_p
_i, _u, _f, _sz = ctypes.c_int, ctypes.c_uint, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "qg_status_string": (ctypes.c_char_p, [_i]),
    "qg_version": (_i, []),
    "qg_device_error": (_i, [ctypes.POINTER(ctypes.c_uint32)]),
    "qgemv_q4": (_i, [_u8p, _u16p, _u16p, _i, _i, _f32p, _f32p, _u, _vp]),
    "qgemv_q6": (_i, [_u8p, _u8p, _u16p, _u16p, _i, _i, _f32p, _f32p, _u, _vp]),
    "qgemv_q2": (_i, [_u8p, _u16p, _i, _i, _f32p, _f32p, _u, _vp]),
    "qg_batched_workspace_bytes": (_sz, [_i, _i, _i]),
    "qgemv_batched": (_i, [_i, _u8p, _u8p, _u16p, _u16p, _i, _i, _i, _f32p, _f32p, _vp, _sz, _u, _vp]),
    "cq_fwht_matvec": (_i, [_u8p, _u16p, _u16p, _i, _i, _i, _i, _i, _f32p, _f32p, _u, _vp]),
    "qg_vocab_workspace_bytes": (_sz, []),
    "vocab_softcap_argmax": (_i, [_i, _u8p, _u8p, _u16p, _u16p, _i, _i, _f32p, _f, _f32p, _i32p, _vp, _sz, _u, _vp]),
    "qg_select_workspace_bytes": (_sz, []),
    "qg_logits_select": (_i, [_f32p, _i, _i32p, _i, _i32p, _f32p, _vp, _sz, _u, _vp]),
    "qg_vocab_select_workspace_bytes": (_sz, []),
    "vocab_softcap_select": (_i, [_i, _u8p, _u8p, _u16p, _u16p, _i, _i, _f32p, _f, _i32p, _i, _f32p, _i32p, _f32p, _vp,
                                  _sz, _u, _vp]),
    "qg_grouped_workspace_bytes": (_sz, [_vp, _i]),
    "qgemv_grouped": (_i, [_i, _vp, _i, _vp, _sz, _u, _vp]),
    "qgemv_grouped_noalloc": (_i, [_i, _vp, _i, _u, _vp]),
    "qg_chain_workspace_bytes": (_sz, [_vp, _i, _vp, _i]),
    "qgemv_chain": (_i, [_i, _vp, _i, _vp, _i, _vp, _sz, _u, _vp]),
    "qg_quantize_act": (_i, [_f32p, _i, _i, _i8p, _f32p, _i32p, _vp]),
    "qg_blockdots": (_i, [_i, _u8p, _u8p, _i, _i, _i8p, _i32p, _vp]),
    "qg_read_floor": (_i, [_vp, _sz, _vp, _u, _vp]),
}

_lock = threading.Lock()
_handle = None


class QGError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib():
    """The loaded ``libqgemv.so`` (raises if it has not been built)."""
    global _handle
    if _handle is None:
        with _lock:
            if _handle is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with quantized_weight_gemv_gb300.build.build() "
                        "(or __graft_entry__.build()); there is no fallback implementation")
                h = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(h, name)
                    fn.restype = res
                    fn.argtypes = args
                _handle = h
    return _handle


def status_string(status: int) -> str:
    return lib().qg_status_string(status).decode()


def _check(rc: int, where: str) -> None:
    if rc != QG_OK:
        raise QGError(rc, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtypes, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtypes and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


_H16 = (torch.float16, torch.int16, torch.uint16)
_U8 = (torch.uint8,)
_F32 = (torch.float32,)


def qgemv_q4(codes, scale, min, x, y=None, flags: int = 0):
    """y[n] = dequant-fused GEMV of Q4 weights (codes [n][k/2] uint8, scale/min [n][k/32] binary16) with x[k]."""
    _need(codes, "codes", _U8)
    dev = codes.device
    for t, nm in ((scale, "scale"), (min, "min")):
        _need(t, nm, _H16, dev)
    _need(x, "x", _F32, dev)
    n, k = codes.shape[0], codes.shape[1] * 2
    if y is None:
        y = torch.empty(n, dtype=torch.float32, device=dev)
    _need(y, "y", _F32, dev)
    with torch.cuda.device(dev):
        _check(lib().qgemv_q4(_ptr(codes), _ptr(scale), _ptr(min), n, k, _ptr(x), _ptr(y), flags, _stream(dev)),
               "qgemv_q4")
    return y


def qgemv_q2(codes, scale, x, y=None, flags: int = 0):
    """y[n] = GEMV of 2-bit weights (codes [n][k/4] uint8, scale [n][k/32] binary16, w = scale*(code-2)) with x[k]."""
    _need(codes, "codes", _U8)
    dev = codes.device
    _need(scale, "scale", _H16, dev)
    _need(x, "x", _F32, dev)
    n, k = codes.shape[0], codes.shape[1] * 4
    if y is None:
        y = torch.empty(n, dtype=torch.float32, device=dev)
    _need(y, "y", _F32, dev)
    with torch.cuda.device(dev):
        _check(lib().qgemv_q2(_ptr(codes), _ptr(scale), n, k, _ptr(x), _ptr(y), flags, _stream(dev)), "qgemv_q2")
    return y


def _k_of(bits, lo):
    return lo.shape[1] * (4 if bits == 2 else 2)


def qgemv_q6(lo, hi, scale, min, x, y=None, flags: int = 0):
    """As :func:`qgemv_q4` for 6-bit codes (lo [n][k/2], hi [n][k/4])."""
    _need(lo, "lo", _U8)
    dev = lo.device
    _need(hi, "hi", _U8, dev)
    for t, nm in ((scale, "scale"), (min, "min")):
        _need(t, nm, _H16, dev)
    _need(x, "x", _F32, dev)
    n, k = lo.shape[0], lo.shape[1] * 2
    if y is None:
        y = torch.empty(n, dtype=torch.float32, device=dev)
    _need(y, "y", _F32, dev)
    with torch.cuda.device(dev):
        _check(lib().qgemv_q6(_ptr(lo), _ptr(hi), _ptr(scale), _ptr(min), n, k, _ptr(x), _ptr(y), flags,
                              _stream(dev)), "qgemv_q6")
    return y


def batched_workspace(bits, k, batch, device):
    """A workspace for :func:`qgemv_batched` (None when the shape needs none)."""
    nbytes = int(lib().qg_batched_workspace_bytes(bits, k, batch))
    return torch.empty(nbytes, dtype=torch.uint8, device=device) if nbytes else None


def qgemv_batched(bits, lo, hi, scale, min, X, Y=None, flags: int = 0, ws="auto"):
    """Y[batch][n] for activation columns X[batch][k] sharing one pass over the weights.
    ``ws``: a workspace tensor, None (no workspace: slower for batch >= 8), or "auto"."""
    _need(lo, "lo", _U8)
    dev = lo.device
    if bits == 6:
        _need(hi, "hi", _U8, dev)
    _need(scale, "scale", _H16, dev)
    if bits != 2:
        _need(min, "min", _H16, dev)
    _need(X, "X", _F32, dev)
    n, k = lo.shape[0], _k_of(bits, lo)
    batch = X.shape[0] if X.dim() == 2 else 1
    if Y is None:
        Y = torch.empty(batch, n, dtype=torch.float32, device=dev)
    _need(Y, "Y", _F32, dev)
    if isinstance(ws, str):
        ws = batched_workspace(bits, k, batch, dev)
    if ws is not None:
        _need(ws, "ws", None, dev)
    with torch.cuda.device(dev):
        _check(lib().qgemv_batched(bits, _ptr(lo), _ptr(hi) if bits == 6 else None, _ptr(scale), _ptr(min) if bits != 2 else None, n, k,
                                   batch, _ptr(X), _ptr(Y), _ptr(ws), 0 if ws is None else ws.numel(), flags,
                                   _stream(dev)), "qgemv_batched")
    return Y


def cq_fwht_matvec(idx, codebook, row_scale, x, group: int = 512, row_start: int = 0, row_count=None, y=None,
                   flags: int = 0):
    """y[row_count] = row_scale * (codebook[idx] . WHT(x)) over rows [row_start, row_start+row_count)."""
    _need(idx, "idx", _U8)
    dev = idx.device
    _need(codebook, "codebook", _H16, dev)
    _need(row_scale, "row_scale", _H16, dev)
    _need(x, "x", _F32, dev)
    n, k = idx.shape[0], idx.shape[1] * 2
    if row_count is None:
        row_count = n - row_start
    if y is None:
        y = torch.empty(max(row_count, 0), dtype=torch.float32, device=dev)
    _need(y, "y", _F32, dev)
    with torch.cuda.device(dev):
        _check(lib().cq_fwht_matvec(_ptr(idx), _ptr(codebook), _ptr(row_scale), n, k, group, row_start, row_count,
                                    _ptr(x), _ptr(y), flags, _stream(dev)), "cq_fwht_matvec")
    return y


def vocab_workspace(device) -> torch.Tensor:
    """A zero-filled workspace for :func:`vocab_softcap_argmax` (reusable; calls leave it zeroed)."""
    return torch.zeros(int(lib().qg_vocab_workspace_bytes()), dtype=torch.uint8, device=device)


def vocab_softcap_argmax(bits, lo, hi, scale, min, x, softcap: float = 30.0, logits=True, argmax=None, ws=None,
                         flags: int = 0):
    """(logits or None, argmax int32[1]) of the soft-capped projection.  ``logits=True`` allocates them,
    ``None``/``False`` skips writing them, a tensor receives them."""
    _need(lo, "lo", _U8)
    dev = lo.device
    if bits == 6:
        _need(hi, "hi", _U8, dev)
    _need(scale, "scale", _H16, dev)
    if bits != 2:
        _need(min, "min", _H16, dev)
    _need(x, "x", _F32, dev)
    n, k = lo.shape[0], _k_of(bits, lo)
    if logits is True:
        logits = torch.empty(n, dtype=torch.float32, device=dev)
    elif logits is False:
        logits = None
    if logits is not None:
        _need(logits, "logits", _F32, dev)
    if argmax is None:
        argmax = torch.empty(1, dtype=torch.int32, device=dev)
    _need(argmax, "argmax", (torch.int32,), dev)
    if ws is None:
        ws = vocab_workspace(dev)
    _need(ws, "ws", None, dev)
    with torch.cuda.device(dev):
        _check(lib().vocab_softcap_argmax(bits, _ptr(lo), _ptr(hi) if bits == 6 else None, _ptr(scale), _ptr(min) if bits != 2 else None, n,
                                          k, _ptr(x), float(softcap), _ptr(logits), _ptr(argmax), _ptr(ws),
                                          ws.numel() * ws.element_size(), flags, _stream(dev)),
               "vocab_softcap_argmax")
    return logits, argmax


class GemvDesc(ctypes.Structure):
    """Mirror of ``qg_gemv_desc``."""
    _fields_ = [("lo", ctypes.c_void_p), ("hi", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("min", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("n", ctypes.c_int), ("k", ctypes.c_int)]


QG_MAX_GROUP = 256


class GroupedGemv:
    """A fixed list of independent GEMVs (one weight format) run by :func:`qgemv_grouped`.

    ``mats``: weight dicts with device tensors ("lo", ["hi"], "scale", "min");
    ``xs``/``ys``: matching device activations [k] and outputs [n].  The descriptor
    array and the workspace are built once; ``run()`` enqueues the two launches.
    """

    def __init__(self, bits, mats, xs, ys, flags: int = 0):
        if not 0 < len(mats) <= QG_MAX_GROUP or len(mats) != len(xs) or len(mats) != len(ys):
            raise ValueError("need 1..256 matching weights, activations and outputs")
        self.bits = bits
        self.flags = flags
        dev = mats[0]["lo"].device
        for m, x, y in zip(mats, xs, ys):
            _need(m["lo"], "lo", _U8, dev)
            if bits == 6:
                _need(m["hi"], "hi", _U8, dev)
            _need(m["scale"], "scale", _H16, dev)
            _need(m["min"], "min", _H16, dev)
            _need(x, "x", _F32, dev)
            _need(y, "y", _F32, dev)
        self.keep = (mats, xs, ys)  # the descriptors hold raw pointers into these tensors
        arr = (GemvDesc * len(mats))()
        for i, (m, x, y) in enumerate(zip(mats, xs, ys)):
            arr[i] = GemvDesc(m["lo"].data_ptr(), m["hi"].data_ptr() if bits == 6 else None,
                              m["scale"].data_ptr(), m["min"].data_ptr(), x.data_ptr(), y.data_ptr(),
                              m["lo"].shape[0], m["lo"].shape[1] * 2)
        self.descs = arr
        self.count = len(mats)
        self.device = dev
        nbytes = int(lib().qg_grouped_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), self.count))
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)

    def run(self):
        with torch.cuda.device(self.device):
            _check(lib().qgemv_grouped(self.bits, ctypes.cast(self.descs, ctypes.c_void_p), self.count,
                                       _ptr(self.ws), self.ws.numel(), self.flags, _stream(self.device)),
                   "qgemv_grouped")


def qgemv_grouped(bits, mats, xs, ys, flags: int = 0):
    """One-shot :class:`GroupedGemv` call; returns ``ys``."""
    GroupedGemv(bits, mats, xs, ys, flags).run()
    return ys


class ChainGemv(GroupedGemv):
    """A fixed dependent chain of GEMVs run by :func:`qgemv_chain`.

    As :class:`GroupedGemv`, plus ``phase_sizes``: the GEMVs are taken in order, the
    next ``phase_sizes[f]`` of them forming phase f; a GEMV's ``xs`` entry may be (a
    view of) the output tensor of a GEMV in an earlier phase.  The workspace is
    zero-filled once here; every completed call leaves its control words zero.
    """

    def __init__(self, bits, mats, xs, ys, phase_sizes, flags: int = 0):
        super().__init__(bits, mats, xs, ys, flags)
        self.phase_sizes = (ctypes.c_int * len(phase_sizes))(*[int(v) for v in phase_sizes])
        self.n_phases = len(phase_sizes)
        nbytes = int(lib().qg_chain_workspace_bytes(ctypes.cast(self.descs, ctypes.c_void_p), self.count,
                                                    ctypes.cast(self.phase_sizes, ctypes.c_void_p), self.n_phases))
        self.ws = torch.zeros(max(nbytes, QG_CHAIN_CTL_BYTES), dtype=torch.uint8, device=self.device)

    def run(self):
        with torch.cuda.device(self.device):
            _check(lib().qgemv_chain(self.bits, ctypes.cast(self.descs, ctypes.c_void_p), self.count,
                                     ctypes.cast(self.phase_sizes, ctypes.c_void_p), self.n_phases, _ptr(self.ws),
                                     self.ws.numel(), self.flags, _stream(self.device)), "qgemv_chain")


def qgemv_chain(bits, mats, xs, ys, phase_sizes, flags: int = 0):
    """One-shot :class:`ChainGemv` call; returns ``ys``."""
    ChainGemv(bits, mats, xs, ys, phase_sizes, flags).run()
    return ys


def select_workspace(device) -> torch.Tensor:
    """A zero-filled workspace for :func:`qg_logits_select` (reusable; calls leave it zeroed)."""
    return torch.zeros(int(lib().qg_select_workspace_bytes()), dtype=torch.uint8, device=device)


def qg_logits_select(logits, allowed=None, token=None, logprob=None, ws=None, flags: int = 0):
    """(token int32[1], logprob fp32[1]): the allowed ID of the largest logit and its
    full-vocabulary log-probability; ``allowed`` is an int32 device tensor of IDs or None."""
    _need(logits, "logits", _F32)
    dev = logits.device
    if allowed is not None:
        _need(allowed, "allowed", (torch.int32,), dev)
    token = torch.empty(1, dtype=torch.int32, device=dev) if token is None else token
    logprob = torch.empty(1, dtype=torch.float32, device=dev) if logprob is None else logprob
    ws = select_workspace(dev) if ws is None else ws
    with torch.cuda.device(dev):
        _check(lib().qg_logits_select(_ptr(logits), logits.numel(), _ptr(allowed),
                                      0 if allowed is None else allowed.numel(), _ptr(token), _ptr(logprob), _ptr(ws),
                                      ws.numel() * ws.element_size(), flags, _stream(dev)), "qg_logits_select")
    return token, logprob


def vocab_select_workspace(device) -> torch.Tensor:
    """A zero-filled workspace for :func:`vocab_softcap_select`."""
    return torch.zeros(int(lib().qg_vocab_select_workspace_bytes()), dtype=torch.uint8, device=device)


def vocab_softcap_select(bits, lo, hi, scale, min, x, softcap: float = 30.0, allowed=None, logits=None, token=None,
                         logprob=None, ws=None, flags: int = 0):
    """(logits, token, logprob) of the soft-capped vocabulary projection with constrained selection."""
    _need(lo, "lo", _U8)
    dev = lo.device
    if bits == 6:
        _need(hi, "hi", _U8, dev)
    _need(scale, "scale", _H16, dev)
    if bits != 2:
        _need(min, "min", _H16, dev)
    _need(x, "x", _F32, dev)
    if allowed is not None:
        _need(allowed, "allowed", (torch.int32,), dev)
    n, k = lo.shape[0], _k_of(bits, lo)
    logits = torch.empty(n, dtype=torch.float32, device=dev) if logits is None else logits
    token = torch.empty(1, dtype=torch.int32, device=dev) if token is None else token
    logprob = torch.empty(1, dtype=torch.float32, device=dev) if logprob is None else logprob
    ws = vocab_select_workspace(dev) if ws is None else ws
    with torch.cuda.device(dev):
        _check(lib().vocab_softcap_select(bits, _ptr(lo), _ptr(hi) if bits == 6 else None, _ptr(scale), _ptr(min) if bits != 2 else None, n,
                                          k, _ptr(x), float(softcap), _ptr(allowed),
                                          0 if allowed is None else allowed.numel(), _ptr(logits), _ptr(token),
                                          _ptr(logprob), _ptr(ws), ws.numel() * ws.element_size(), flags,
                                          _stream(dev)), "vocab_softcap_select")
    return logits, token, logprob


def qg_quantize_act(x):
    """(xq int8 [batch][k], xs fp32 [batch][k/32], xsum int32 [batch][k/32]) for x [batch][k] or [k]."""
    _need(x, "x", _F32)
    dev = x.device
    X = x.reshape(-1, x.shape[-1])
    batch, k = X.shape
    xq = torch.empty(batch, k, dtype=torch.int8, device=dev)
    xs = torch.empty(batch, k // 32, dtype=torch.float32, device=dev)
    xsum = torch.empty(batch, k // 32, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib().qg_quantize_act(_ptr(X), k, batch, _ptr(xq), _ptr(xs), _ptr(xsum), _stream(dev)),
               "qg_quantize_act")
    return xq, xs, xsum


def qg_blockdots(bits, lo, hi, xq):
    """Exact integer block dots int32 [n][k/32] of the codes with int8 xq [k]."""
    _need(lo, "lo", _U8)
    dev = lo.device
    if bits == 6:
        _need(hi, "hi", _U8, dev)
    _need(xq, "xq", (torch.int8,), dev)
    n, k = lo.shape[0], _k_of(bits, lo)
    dots = torch.empty(n, k // 32, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib().qg_blockdots(bits, _ptr(lo), _ptr(hi) if bits == 6 else None, n, k, _ptr(xq), _ptr(dots),
                                  _stream(dev)), "qg_blockdots")
    return dots


def qg_read_floor(buf, out=None, flags: int = 0):
    """Read every byte of the device tensor `buf` once (the plain-read floor); returns the
    uint32 XOR of its words in `out` (an int32 [1] device tensor, XOR-accumulated)."""
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    dev = buf.device
    if out is None:
        out = torch.zeros(1, dtype=torch.int32, device=dev)
    _need(out, "out", (torch.int32,), dev)
    with torch.cuda.device(dev):
        _check(lib().qg_read_floor(_ptr(buf), buf.numel() * buf.element_size(), _ptr(out), flags, _stream(dev)),
               "qg_read_floor")
    return out


def device_error() -> int:
    """Read and clear the device error word (nonzero: a bounded wait in a kernel ran out)."""
    v = ctypes.c_uint32(0)
    _check(lib().qg_device_error(ctypes.byref(v)), "qg_device_error")
    return int(v.value)


def to_device(w: dict, device="cuda") -> dict:
    """Copy a packed weight dict of numpy planes (as made by the input generator) to device tensors."""
    out = dict(w)
    for key in ("lo", "hi", "scale", "min", "idx", "codebook", "row_scale"):
        if key in w and w[key] is not None:
            a = w[key]
            if a.dtype.itemsize == 2:
                a = a.view("int16")  # binary16 bit patterns travel as int16
            out[key] = torch.from_numpy(a).to(device)
    return out
