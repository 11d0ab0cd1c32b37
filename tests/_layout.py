"""Test-side packers for the weight layouts, written independently of ``datagen`` and ``oracle``.

Layout (blocks of 32 along K, rows row-major):
  Q4 byte 16*b + j of a row = code(32b + j) | code(32b + j + 16) << 4
  Q6 lo as Q4 on the low 4 bits; hi byte 8*b + t = sum over s in 0..3 of
     (code(32b + t + 8s) >> 4) << 2s
  Q2 byte 8*b + t of a row = sum over s in 0..3 of code(32b + t + 8s) << 2s
  CQ byte j of a row = idx(2j) | idx(2j + 1) << 4
"""
import numpy as np


def pack_q4(q):
    q = np.asarray(q, dtype=np.uint8)
    n, k = q.shape
    blk = q.reshape(n, k // 32, 32)
    out = (blk[:, :, :16] & 15) | ((blk[:, :, 16:] & 15) << 4)
    return out.reshape(n, k // 2).astype(np.uint8)


def pack_q6(q):
    q = np.asarray(q, dtype=np.uint8)
    n, k = q.shape
    lo = pack_q4(q & 15)
    blk = (q >> 4).reshape(n, k // 32, 4, 8)  # [n][b][s][t] = code 32b + 8s + t
    hi = np.zeros((n, k // 32, 8), dtype=np.uint8)
    for s in range(4):
        hi |= (blk[:, :, s, :] & 3) << (2 * s)
    return lo, hi.reshape(n, k // 4)


def pack_q2(q):
    q = np.asarray(q, dtype=np.uint8)
    n, k = q.shape
    blk = q.reshape(n, k // 32, 4, 8)  # [n][b][s][t] = code 32b + 8s + t
    out = np.zeros((n, k // 32, 8), dtype=np.uint8)
    for s in range(4):
        out |= (blk[:, :, s, :] & 3) << (2 * s)
    return out.reshape(n, k // 4)


def pack_cq(idx):
    idx = np.asarray(idx, dtype=np.uint8)
    return ((idx[:, 0::2] & 15) | ((idx[:, 1::2] & 15) << 4)).astype(np.uint8)


def f16_bits(values):
    return np.asarray(values, dtype=np.float16).view(np.uint16)


def make_w(bits, q, scale, minv):
    """A weight dict from explicit codes [n][k] and fp32-valued scale/min [n][k/32] (stored as f16)."""
    q = np.asarray(q, dtype=np.uint8)
    n, k = q.shape
    if bits == 2:
        lo, hi = pack_q2(q), None
    elif bits == 4:
        lo, hi = pack_q4(q), None
    else:
        lo, hi = pack_q6(q)
    return {"bits": bits, "n": n, "k": k, "lo": lo, "hi": hi,
            "scale": f16_bits(np.broadcast_to(scale, (n, k // 32))).copy(),
            "min": None if bits == 2 else f16_bits(np.broadcast_to(minv, (n, k // 32))).copy()}


def dense_dequant(bits, q, w):
    """W_deq [n][k] in fp64 from known codes and the stored half scale/min."""
    n, k = np.asarray(q).shape
    d = w["scale"].view(np.float16).astype(np.float64)
    if bits == 2:
        return np.repeat(d, 32, axis=1) * (np.asarray(q, np.float64) - 2.0)
    m = w["min"].view(np.float16).astype(np.float64)
    return np.repeat(d, 32, axis=1) * np.asarray(q, np.float64) + np.repeat(m, 32, axis=1)
