"""The five workloads, as seeded recipes over :mod:`datagen`.

Shapes, distributions and seeds:

* ``q4_single``  - Q4 W 1024x1024 (weights N(0, 0.02)), x[1024] N(0, 1); seed 0.
* ``decode_layers`` - 35 layers x 7 Q4 projections of a hidden-2048 / FFN-16384
  decoder (q, k, v, o, gate, up, down as N x K below), each with its own seed
  ``1000 + 7*layer + proj`` and its own x ~ N(0, 1) of length K.
* ``decode_chain`` - the same weights, each GEMV reading an earlier one's output
  (``decode_chain_plan``); one external x[2048] ~ N(0, 1).
* ``vocab_q6``   - Q6 W 262144x2048 (N(0, 0.02)), x[2048] N(0, 1); soft-cap 30; seed 2.
* ``vocab_q2``   - Q2 (zero point 2) W 262144x1536 (N(0, 0.02)), x[1536] N(0, 1); seed 5.
* ``select_allowed`` - ~1 % of the vocabulary ids, uniform, distinct; seed 6.
* ``batched_q4`` - Q4 W 16384x2048 (N(0, 0.02)); X[B][2048] N(0, 1), column b drawn
  from offset b*2048 of the activation stream; seed 3.
* ``cq``         - K = 512 (one 512-value group); codebook 16 x f16 N(0, 0.05),
  f16 row scales 0.5 + U(0, 1), indices U{0..15}; x[512] N(0, 1); seed 4.
  Two matrices: 8192 rows (streams 2..4) and 1024 rows (streams 12..14).

Weights are drawn on stream 0 and activations on stream 1 of their seed.
"""
from __future__ import annotations

import numpy as np

from . import STREAM_X, make_cq, make_quantized, normal_f32, uniform_f32

HIDDEN = 2048
FFN = 16384
N_LAYERS = 35
PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")
# (N, K) per projection
PROJ_SHAPES = (
    (2048, 2048),
    (1024, 2048),
    (1024, 2048),
    (2048, 2048),
    (FFN, 2048),
    (FFN, 2048),
    (2048, FFN),
)
VOCAB = 262144
SOFTCAP = 30.0
BATCHES = (1, 2, 4, 8, 16)
CQ_K = 512
CQ_GROUP = 512
CQ_ROWS = (8192, 1024)


def q4_bytes(n: int, k: int) -> int:
    """Packed Q4 bytes: 16 B codes + 2 B scale + 2 B min per block of 32."""
    return n * (k // 32) * 20


def q6_bytes(n: int, k: int) -> int:
    """Packed Q6 bytes: 16 B lo + 8 B hi + 2 B scale + 2 B min per block of 32."""
    return n * (k // 32) * 28


def q2_bytes(n: int, k: int) -> int:
    """Packed Q2 bytes: 8 B codes + 2 B scale per block of 32 (no min plane)."""
    return n * (k // 32) * 10


def cq_bytes(n: int, k: int) -> int:
    """CQ bytes: k/2 index bytes + 2 B row scale per row, plus the 32-byte codebook."""
    return n * (k // 2 + 2) + 32


def q4_single():
    w = make_quantized(4, 0, 1024, 1024)
    x = normal_f32(0, STREAM_X, 1024)
    return w, x


def decode_seed(layer: int, proj: int) -> int:
    return 1000 + 7 * layer + proj


def decode_projection(layer: int, proj: int, rows: slice | None = None):
    """One projection of the decode-layer stream: (weights, x)."""
    n, k = PROJ_SHAPES[proj]
    seed = decode_seed(layer, proj)
    w = make_quantized(4, seed, n, k)
    x = normal_f32(seed, STREAM_X, k)
    return w, x


def decode_chain_plan(n_layers: int = N_LAYERS):
    """Wiring of the dependent decode chain over the decode-layer projections.

    GEMV 7*layer + proj is projection ``proj`` of ``layer`` (same weights as
    ``decode_projection``).  Returns (src, stage_sizes): src[j] is the GEMV whose
    output GEMV j reads (-1: the external input, ``decode_chain_x``), stage_sizes
    the GEMVs per stage in order.  Per layer four stages:
      q, k, v  <- the layer input (layer 0: the external input; then the previous down)
      o        <- q      (stands for the attention output: 2048 values)
      gate, up <- o      (stands for the normalised residual stream: 2048 values)
      down     <- gate   (stands for the gated FFN activation: 16384 values)
    Attention, norms, residual adds and the gate nonlinearity are not part of the
    chain; each link is one quantised GEMV on the previous link's fp32 output.
    """
    src, stages = [], []
    for layer in range(n_layers):
        base = 7 * layer
        inp = -1 if layer == 0 else base - 1
        src += [inp, inp, inp, base + 0, base + 3, base + 3, base + 4]
        stages += [3, 1, 2, 1]
    return src, stages


def decode_chain_x() -> np.ndarray:
    """External input of the decode chain: x[2048] ~ N(0, 1), the layer-0 q activation."""
    return normal_f32(decode_seed(0, 0), STREAM_X, HIDDEN)


def decode_pass_bytes(n_layers: int = N_LAYERS) -> int:
    return n_layers * sum(q4_bytes(n, k) for n, k in PROJ_SHAPES)


def vocab_q6():
    w = make_quantized(6, 2, VOCAB, HIDDEN)
    x = normal_f32(2, STREAM_X, HIDDEN)
    return w, x


VOCAB_Q2_K = 1536  # the int2 LM head's width (Gemma WebGPU Engine, "Roadmap": 262,144 x 1536)


def vocab_q2():
    """The int2 (zero point 2) LM head: Q2 W 262144x1536 ~ N(0, 0.02), x[1536] ~ N(0, 1); seed 5."""
    w = make_quantized(2, 5, VOCAB, VOCAB_Q2_K)
    x = normal_f32(5, STREAM_X, VOCAB_Q2_K)
    return w, x


def select_allowed(n: int = VOCAB, frac: float = 0.01, seed: int = 6) -> np.ndarray:
    """A constrained-decoding allowed list: distinct sorted int32 ids, about frac * n of
    them, drawn uniformly (stream 2 of the seed)."""
    m = max(1, int(n * frac))
    ids = np.unique((uniform_f32(seed, 2, m) * n).astype(np.int64) % n)
    return ids.astype(np.int32)


def batched_q4_weights():
    return make_quantized(4, 3, FFN, HIDDEN)


def batched_q4_x(batch: int) -> np.ndarray:
    return normal_f32(3, STREAM_X, batch * HIDDEN).reshape(batch, HIDDEN)


def cq_matrix(which: int):
    """which = 0: the 8192-row matrix; 1: the 1024-row matrix."""
    return make_cq(4, CQ_ROWS[which], CQ_K, stream_base=10 * which)


def cq_x() -> np.ndarray:
    return normal_f32(4, STREAM_X, CQ_K)
