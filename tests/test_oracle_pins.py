"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against a hand-worked fixture, a closed
form, a textbook matrix, a library routine, brute force on tiny inputs or an
exhaustive enumeration, chosen so that a plausible slip (a swapped nibble, a
wrong sign of the min term, a transposed Hadamard, a dropped scale) fails.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import datagen
import oracle
from tests import _golden as G
from tests._layout import dense_dequant, f16_bits, make_w, pack_cq, pack_q4, pack_q6


# ------------------------------------------------------------------ binary16
def test_half_decoder_exhaustive_against_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


# ------------------------------------------------------------------ activation quantisation
@pytest.mark.parametrize("blk", ["A", "B", "C"])
def test_act_quant_golden(blk):
    g = G.load("act_quant_block.txt")
    x = np.array(G.floats(g[f"{blk}.x"]), np.float32)
    xq, s, S = oracle.quantize_act(x)
    assert xq.tolist() == G.ints(g[f"{blk}.xq"])
    assert s[0] == np.float32(G.floats(g[f"{blk}.s"])[0])
    assert S[0] == G.ints(g[f"{blk}.S"])[0]


def test_act_quant_unit_vector():
    for a in (3.0, -0.125, 1e-3, 7e4):
        for i in (0, 13, 31):
            x = np.zeros(64, np.float32)
            x[32 + i] = a
            xq, s, S = oracle.quantize_act(x)
            assert s[0] == 0 and S[0] == 0 and not xq[:32].any()
            expect = np.zeros(32, np.int8)
            expect[i] = 127 if a > 0 else -127
            assert np.array_equal(xq[32:], expect)
            assert s[1] == np.float32(abs(np.float32(a))) / np.float32(127)


def test_act_quant_invariants_random():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(32 * 400) * rng.choice([1e-3, 1.0, 50.0], 32 * 400)).astype(np.float32)
    xq, s, S = oracle.quantize_act(x)
    xb = x.reshape(-1, 32).astype(np.float64)
    qb = xq.reshape(-1, 32).astype(np.int64)
    assert np.all(np.abs(qb) <= 127)
    assert np.array_equal(S, qb.sum(1))
    # the element of largest magnitude maps to +-127 with its sign
    i = np.argmax(np.abs(xb), 1)
    assert np.array_equal(qb[np.arange(len(i)), i], np.where(xb[np.arange(len(i)), i] > 0, 127, -127))
    # round-trip bound |x - s*xq| <= s/2 (plus a few ulps of the fp32 division)
    err = np.abs(xb - s[:, None].astype(np.float64) * qb)
    assert np.all(err <= s[:, None] * (0.5 + 1e-5))
    # signs agree wherever the code is nonzero
    assert np.all((qb == 0) | (np.sign(qb) == np.sign(xb)))


# ------------------------------------------------------------------ code extraction
def test_q4_block_golden():
    g = G.load("q4_block.txt")
    codes = G.ints(g["codes"])
    packed = np.array(G.hexbytes(g["bytes"]), np.uint8)[None, :]
    assert np.array_equal(pack_q4(np.array([codes])), packed)  # test packer agrees with the hand packing
    w = {"bits": 4, "n": 1, "k": 32, "lo": packed, "hi": None,
         "scale": f16_bits([[1.0]]), "min": f16_bits([[0.0]])}
    assert oracle.codes(w)[0].tolist() == codes


def test_q6_block_golden():
    g = G.load("q6_block.txt")
    codes = G.ints(g["codes"])
    lo = np.array(G.hexbytes(g["lo"]), np.uint8)[None, :]
    hi = np.array(G.hexbytes(g["hi"]), np.uint8)[None, :]
    plo, phi = pack_q6(np.array([codes]))
    assert np.array_equal(plo, lo) and np.array_equal(phi, hi)
    w = {"bits": 6, "n": 1, "k": 32, "lo": lo, "hi": hi,
         "scale": f16_bits([[1.0]]), "min": f16_bits([[0.0]])}
    assert oracle.codes(w)[0].tolist() == codes


@pytest.mark.parametrize("bits", [4, 6])
def test_codes_roundtrip_random(bits):
    rng = np.random.default_rng(bits)
    q = rng.integers(0, 16 if bits == 4 else 64, size=(7, 96), dtype=np.uint8)
    w = make_w(bits, q, 1.0, 0.0)
    assert np.array_equal(oracle.codes(w), q.astype(np.int32))
    # the shared input packer writes the same bytes as the test packer
    if bits == 4:
        assert np.array_equal(datagen.pack_q4_codes(q), w["lo"])
    else:
        lo, hi = datagen.pack_q6_codes(q)
        assert np.array_equal(lo, w["lo"]) and np.array_equal(hi, w["hi"])


# ------------------------------------------------------------------ dequantisation
@pytest.mark.parametrize("bits", [4, 6])
def test_dequant_matches_dense_definition(bits):
    rng = np.random.default_rng(10 + bits)
    n, k = 5, 128
    q = rng.integers(0, 16 if bits == 4 else 64, size=(n, k), dtype=np.uint8)
    scale = rng.uniform(0.001, 0.01, size=(n, k // 32)).astype(np.float32)
    mn = rng.uniform(-0.1, 0.0, size=(n, k // 32)).astype(np.float32)
    w = make_w(bits, q, scale, mn)
    assert np.array_equal(oracle.dequant(w), dense_dequant(bits, q, w))


@pytest.mark.parametrize("bits", [4, 6])
def test_dequant_reconstructs_the_drawn_weights(bits):
    """w_deq of the seeded quantiser stays within half a step (plus fp16 rounding) of the fp32 weights."""
    n, k = 16, 256
    wq = datagen.make_quantized(bits, 77, n, k)
    raw = datagen.weights_f32(77, n, k).astype(np.float64)
    deq = oracle.dequant(wq)
    d = np.repeat(wq["scale"].view(np.float16).astype(np.float64), 32, 1)
    lo = np.repeat(raw.reshape(n, k // 32, 32).min(2), 32, 1)
    qmax = 15 if bits == 4 else 63
    bound = 0.5 * d + 2.0 ** -10 * (np.abs(lo) + (qmax + 1) * d) + 1e-9
    assert np.all(np.abs(deq - raw) <= bound)
    # and the error is not trivially small: the quantiser really is 4/6-bit
    assert np.max(np.abs(deq - raw) / d) > 0.3


# ------------------------------------------------------------------ block dots
@pytest.mark.parametrize("bits", [4, 6])
def test_blockdots_exhaustive_constant_blocks(bits):
    """Every code value against every int8 value: D = 32 * c * v."""
    cmax = 16 if bits == 4 else 64
    vals = np.arange(-127, 128, dtype=np.int64)
    q = np.repeat(np.arange(cmax, dtype=np.uint8), 32)[None, :]  # block c has all codes c
    w = make_w(bits, q, 1.0, 0.0)
    for v in vals:
        xq = np.full(q.shape[1], v, np.int8)
        D = oracle.blockdots(w, xq)[0]
        assert np.array_equal(D, 32 * np.arange(cmax) * v)


@pytest.mark.parametrize("bits", [4, 6])
def test_blockdots_brute_force_random(bits):
    rng = np.random.default_rng(20 + bits)
    n, k = 8, 128
    q = rng.integers(0, 16 if bits == 4 else 64, size=(n, k), dtype=np.uint8)
    xq = rng.integers(-127, 128, size=k).astype(np.int8)
    w = make_w(bits, q, 1.0, 0.0)
    ref = np.zeros((n, k // 32), np.int64)
    for r in range(n):
        for b in range(k // 32):
            for i in range(32):
                ref[r, b] += int(q[r, 32 * b + i]) * int(xq[32 * b + i])
    assert np.array_equal(oracle.blockdots(w, xq), ref)


def test_blockdots_golden():
    g = G.load("q4_block.txt")
    a = G.load("act_quant_block.txt")
    q = np.array([G.ints(g["codes"])], np.uint8)
    w = make_w(4, q, 1.0, 0.0)
    assert oracle.blockdots(w, np.array(G.ints(a["A.xq"]), np.int8))[0, 0] == G.ints(g["gemv.D"])[0]


# ------------------------------------------------------------------ GEMV
def test_gemv_golden():
    g = G.load("q4_block.txt")
    a = G.load("act_quant_block.txt")
    q = np.array([G.ints(g["codes"])], np.uint8)
    w = make_w(4, q, G.floats(g["gemv.scale"])[0], G.floats(g["gemv.min"])[0])
    y = oracle.gemv(w, np.array(G.floats(a["A.x"]), np.float32))
    assert y[0] == G.floats(g["gemv.y"])[0]


@pytest.mark.parametrize("bits", [4, 6])
def test_gemv_dense_fp64_matmul(bits):
    """y equals the dense fp64 matmul of the explicitly materialised W_deq with x_deq."""
    rng = np.random.default_rng(30 + bits)
    n, k = 6, 160
    q = rng.integers(0, 16 if bits == 4 else 64, size=(n, k), dtype=np.uint8)
    scale = rng.uniform(1e-3, 2e-2, size=(n, k // 32)).astype(np.float32)
    mn = rng.uniform(-0.2, 0.05, size=(n, k // 32)).astype(np.float32)
    w = make_w(bits, q, scale, mn)
    x = rng.standard_normal(k).astype(np.float32)
    xq, s, S = oracle.quantize_act(x)
    xdeq = np.repeat(s.astype(np.float64), 32) * xq
    ref = dense_dequant(bits, q, w) @ xdeq
    y = oracle.gemv(w, x)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13 * np.abs(ref).max())
    # row sub-ranges and explicit row lists agree with the full product
    assert np.array_equal(oracle.gemv(w, x, row0=2, nrows=3), y[2:5])
    assert np.array_equal(oracle.gemv_rows(w, x, [4, 0, 5]), y[[4, 0, 5]])


@pytest.mark.parametrize("bits", [4, 6])
def test_gemv_constant_code_closed_form(bits):
    """A constant-code block c contributes (scale*c + min) * sum(x_deq) = s*(scale*c + min)*S."""
    rng = np.random.default_rng(40 + bits)
    k = 96
    cvals = [3, 11] if bits == 4 else [3, 50]
    q = np.array([[c] * k for c in cvals], np.uint8)
    d, m = 0.0078125, -0.0625  # exact in fp16
    w = make_w(bits, q, d, m)
    x = rng.standard_normal(k).astype(np.float32)
    xq, s, S = oracle.quantize_act(x)
    for r, c in enumerate(cvals):
        ref = sum(float(s[b]) * (d * c + m) * int(S[b]) for b in range(k // 32))
        assert math.isclose(oracle.gemv(w, x)[r], ref, rel_tol=1e-14)


def test_gemv_zero_codes_min_term_only():
    rng = np.random.default_rng(50)
    k = 128
    q = np.zeros((1, k), np.uint8)
    mn = rng.uniform(-0.1, 0.1, size=(1, k // 32)).astype(np.float32)
    w = make_w(4, q, 0.01, mn)
    x = rng.standard_normal(k).astype(np.float32)
    xq, s, S = oracle.quantize_act(x)
    m16 = w["min"].view(np.float16).astype(np.float64)[0]
    ref = float(np.sum(m16 * s.astype(np.float64) * S))
    assert math.isclose(oracle.gemv(w, x)[0], ref, rel_tol=1e-13)


def test_gemv_sign_of_min_term():
    """w = scale*code + min: a block of code 0 with min = -1 gives y = -sum(x_deq)."""
    k = 32
    w = make_w(4, np.zeros((1, k), np.uint8), 0.5, -1.0)
    x = np.linspace(-1, 3, k).astype(np.float32)
    xq, s, S = oracle.quantize_act(x)
    assert oracle.gemv(w, x)[0] == -float(s[0]) * int(S[0])


def test_gemv_close_to_unquantised_product():
    """The quantised product tracks the fp32 product of the drawn weights (information, loose bound)."""
    n, k = 64, 2048
    wq = datagen.make_quantized(4, 9, n, k)
    raw = datagen.weights_f32(9, n, k).astype(np.float64)
    x = datagen.normal_f32(9, 1, k)
    y = oracle.gemv(wq, x)
    ref = raw @ x.astype(np.float64)
    assert np.sqrt(np.mean((y - ref) ** 2)) < 0.15 * np.sqrt(np.mean(ref ** 2))


# ------------------------------------------------------------------ soft-cap and argmax
def test_softcap_golden():
    g = G.load("softcap.txt")
    c = G.floats(g["c"])[0]
    got = oracle.softcap(np.array(G.floats(g["z"])), c)
    assert np.allclose(got, G.floats(g["l"]), rtol=1e-15, atol=1e-15)


def test_softcap_properties():
    z = np.linspace(-200, 200, 4001)
    l = oracle.softcap(z, 30.0)
    assert np.all(np.abs(l) < 30.0 + 1e-12)
    assert np.all(np.diff(l) >= 0)
    assert np.allclose(oracle.softcap(-z, 30.0), -l)
    small = np.array([1e-3, -2e-3, 0.05])
    assert np.allclose(oracle.softcap(small, 30.0), small - small ** 3 / (3 * 900.0), rtol=1e-12)
    assert np.array_equal(oracle.softcap(z, 0.0), z)


def test_argmax_brute_force_and_ties():
    rng = np.random.default_rng(60)
    for _ in range(20):
        v = rng.integers(-5, 5, size=rng.integers(1, 300)).astype(np.float64)
        m = v.max()
        assert oracle.argmax(v) == min(i for i in range(len(v)) if v[i] == m)
        assert oracle.argmax(v.astype(np.float32)) == oracle.argmax(v)
    v = np.array([np.nan, 1.0, 3.0, np.nan, 3.0])
    assert oracle.argmax(v) == 2
    assert oracle.argmax(np.array([np.nan, np.nan])) == 0


def test_vocab_planted_maximum():
    rng = np.random.default_rng(61)
    n, k = 300, 64
    q = rng.integers(0, 64, size=(n, k), dtype=np.uint8)
    q[217] = 63  # every code at its maximum with a positive scale and x > 0
    w = make_w(6, q, 0.01, 0.0)
    x = np.abs(rng.standard_normal(k)).astype(np.float32) + 0.1
    logits, idx = oracle.vocab_softcap_argmax(w, x, 30.0)
    assert idx == 217
    z = oracle.gemv(w, x)
    assert oracle.argmax(z) == idx  # the cap is monotone


# ------------------------------------------------------------------ Walsh-Hadamard
@pytest.mark.parametrize("g", [1, 2, 4, 8, 16, 64, 512])
def test_wht_matches_sylvester_hadamard(g):
    rng = np.random.default_rng(g)
    x = rng.standard_normal(g)
    ref = scipy.linalg.hadamard(g).astype(np.float64) @ x / math.sqrt(g)
    assert np.allclose(oracle.wht(x), ref, rtol=1e-12, atol=1e-12)


def test_wht_golden():
    h = G.load("hadamard.txt")
    for g in ("g2", "g4", "g8"):
        got = oracle.wht(np.array(G.floats(h[g + ".x"])))
        assert np.allclose(got, G.floats(h[g + ".u"]), rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("g", [2, 32, 512])
def test_wht_orthonormal(g):
    rng = np.random.default_rng(100 + g)
    x = rng.standard_normal(g)
    u = oracle.wht(x)
    assert math.isclose(np.linalg.norm(u), np.linalg.norm(x), rel_tol=1e-12)
    assert np.allclose(oracle.wht(u), x, atol=1e-12)  # H H = I (normalised)
    e0 = np.zeros(g)
    e0[0] = 1
    assert np.allclose(oracle.wht(e0), np.full(g, 1 / math.sqrt(g)))
    assert np.allclose(oracle.wht(np.ones(g)), math.sqrt(g) * e0)


def test_wht_explicit_matrix_is_involutive_for_all_sizes():
    for lg in range(1, 10):
        g = 1 << lg
        H = np.stack([oracle.wht(np.eye(g)[j]) for j in range(g)], 1)  # columns = transforms of unit vectors
        assert np.allclose(H @ H, np.eye(g), atol=1e-12)


# ------------------------------------------------------------------ CQ matvec
def _cq_dict(idx, cb, rs):
    n, k = idx.shape
    return {"n": n, "k": k, "idx": pack_cq(idx), "codebook": f16_bits(cb), "row_scale": f16_bits(rs)}


def test_cq_constant_index_closed_form():
    """All indices c: y_r = scale_r * cb[c] * sum_i u_i = scale_r * cb[c] * sqrt(g) * (x_0 of each group)."""
    rng = np.random.default_rng(70)
    g, k = 512, 1024
    cb = np.linspace(-0.1, 0.1, 16).astype(np.float32)
    rs = np.array([0.5, 1.25, 0.75], np.float32)
    idx = np.array([[3] * k, [9] * k, [15] * k], np.uint8)
    m = _cq_dict(idx, cb, rs)
    x = rng.standard_normal(k).astype(np.float32)
    y = oracle.cq_matvec(m, x, g)
    cb16 = m["codebook"].view(np.float16).astype(np.float64)
    rs16 = m["row_scale"].view(np.float16).astype(np.float64)
    for r, c in enumerate((3, 9, 15)):
        ref = rs16[r] * cb16[c] * math.sqrt(g) * (float(x[0]) + float(x[g]))
        assert math.isclose(y[r], ref, rel_tol=1e-12)


def test_cq_dense_transform_domain_identity():
    """W~ (H x / sqrt g) equals (W~ H / sqrt g) x: the inverse transform never needs a dense matrix."""
    rng = np.random.default_rng(71)
    g, k, n = 64, 128, 9
    idx = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
    cb = rng.standard_normal(16).astype(np.float32) * 0.05
    rs = rng.uniform(0.5, 1.5, n).astype(np.float32)
    m = _cq_dict(idx, cb, rs)
    x = rng.standard_normal(k).astype(np.float32)
    cb16 = m["codebook"].view(np.float16).astype(np.float64)
    rs16 = m["row_scale"].view(np.float16).astype(np.float64)
    Wt = rs16[:, None] * cb16[idx]
    Hn = scipy.linalg.block_diag(*([scipy.linalg.hadamard(g) / math.sqrt(g)] * (k // g)))
    ref = (Wt @ Hn) @ x.astype(np.float64)
    assert np.allclose(oracle.cq_matvec(m, x, g), ref, rtol=1e-12, atol=1e-12)


def test_cq_row_range_is_a_slice():
    m = datagen.make_cq(4, 40, 512)
    x = datagen.normal_f32(4, 1, 512)
    full = oracle.cq_matvec(m, x, 512)
    assert np.array_equal(oracle.cq_matvec(m, x, 512, row_start=13, row_count=11), full[13:24])
    assert oracle.cq_matvec(m, x, 512, row_start=5, row_count=0).size == 0


# ------------------------------------------------------------------ error measure
def test_normwise_error_definition():
    ref = np.array([1.0, -2.0, 0.0, 1e-9])
    rms = math.sqrt((1 + 4) / 4)
    y = ref + np.array([1e-4, 0.0, 2e-4, 0.0])
    assert math.isclose(oracle.normwise_error(y, ref), 2e-4 / rms, rel_tol=1e-12)


# ------------------------------------------------------------------ constrained selection
def test_logsumexp_closed_forms_and_scipy():
    import scipy.special
    assert math.isclose(oracle.logsumexp(np.zeros(1000)), math.log(1000), rel_tol=1e-15)
    assert math.isclose(oracle.logsumexp(np.array([0.0, math.log(3.0)])), math.log(4.0), rel_tol=1e-15)
    rng = np.random.default_rng(80)
    v = rng.standard_normal(5000) * 7
    assert math.isclose(oracle.logsumexp(v), float(scipy.special.logsumexp(v)), rel_tol=1e-13)
    assert math.isclose(oracle.logsumexp(v + 1000.0), oracle.logsumexp(v) + 1000.0, rel_tol=1e-13)  # shift-invariant
    assert oracle.logsumexp(np.array([np.nan, 2.0])) == 2.0


def test_select_closed_forms():
    n = 4096
    idx, lp = oracle.select(np.zeros(n))
    assert idx == 0 and math.isclose(lp, -math.log(n), rel_tol=1e-14)  # uniform: ties to the lowest id
    v = np.zeros(8)
    v[5] = math.log(3.0)
    idx, lp = oracle.select(v)
    assert idx == 5 and math.isclose(lp, math.log(3.0 / 10.0), rel_tol=1e-14)
    idx, lp = oracle.select(v, [1, 2, 7])
    assert idx == 1 and math.isclose(lp, math.log(1.0 / 10.0), rel_tol=1e-14)
    assert oracle.select(v, [])[0] == -1


def test_select_brute_force_and_probabilities_sum_to_one():
    rng = np.random.default_rng(81)
    for trial in range(20):
        n = int(rng.integers(2, 3000))
        v = np.round(rng.standard_normal(n) * 4, 1)  # repeats make ties likely
        allowed = np.sort(rng.choice(n, size=int(rng.integers(1, n)), replace=False)).astype(np.int32)
        idx, lp = oracle.select(v, allowed)
        best = max(allowed.tolist(), key=lambda i: (v[i], -i))
        assert idx == best
        probs = np.exp(v - oracle.logsumexp(v))
        assert math.isclose(probs.sum(), 1.0, rel_tol=1e-12)
        assert math.isclose(math.exp(lp), probs[idx], rel_tol=1e-12)


# ------------------------------------------------------------------ 2-bit codes, zero point 2
def test_q2_block_golden():
    g = G.load("q2_block.txt")
    codes = G.ints(g["codes"])
    packed = np.array(G.hexbytes(g["bytes"]), np.uint8)[None, :]
    from tests._layout import pack_q2
    assert np.array_equal(pack_q2(np.array([codes])), packed)
    assert np.array_equal(datagen.pack_q2_codes(np.array([codes], np.uint8)), packed)
    w = {"bits": 2, "n": 1, "k": 32, "lo": packed, "hi": None, "scale": f16_bits([[G.floats(g["gemv.scale"])[0]]]),
         "min": None}
    assert oracle.codes(w)[0].tolist() == codes
    y = oracle.gemv(w, np.ones(32, np.float32))
    assert math.isclose(y[0], G.floats(g["gemv.y"])[0], rel_tol=1e-6)


def test_q2_codes_dequant_and_dots():
    rng = np.random.default_rng(90)
    n, k = 6, 160
    q = rng.integers(0, 4, size=(n, k), dtype=np.uint8)
    scale = rng.uniform(1e-3, 2e-2, size=(n, k // 32)).astype(np.float32)
    w = make_w(2, q, scale, None)
    assert np.array_equal(oracle.codes(w), q.astype(np.int32))
    assert np.array_equal(oracle.dequant(w), dense_dequant(2, q, w))
    xq = rng.integers(-127, 128, size=k).astype(np.int8)
    ref = (q.reshape(n, k // 32, 32).astype(np.int64) * xq.reshape(k // 32, 32)).sum(2)
    assert np.array_equal(oracle.blockdots(w, xq), ref)
    x = rng.standard_normal(k).astype(np.float32)
    xq2, s, S = oracle.quantize_act(x)
    assert np.allclose(oracle.gemv(w, x), dense_dequant(2, q, w) @ (np.repeat(s.astype(np.float64), 32) * xq2),
                       rtol=1e-13, atol=1e-15)


def test_q2_zero_point_closed_forms():
    """All codes 2 decode to zero weights; all codes 3 give y = scale * sum(x_deq)."""
    k = 96
    x = datagen.normal_f32(91, 1, k)
    xq, s, S = oracle.quantize_act(x)
    assert oracle.gemv(make_w(2, np.full((1, k), 2, np.uint8), 0.5, None), x)[0] == 0.0
    ref = sum(0.5 * float(s[b]) * int(S[b]) for b in range(k // 32))
    assert math.isclose(oracle.gemv(make_w(2, np.full((1, k), 3, np.uint8), 0.5, None), x)[0], ref, rel_tol=1e-14)


def test_q2_reconstructs_the_drawn_weights():
    n, k = 16, 256
    wq = datagen.make_quantized(2, 92, n, k)
    raw = datagen.weights_f32(92, n, k).astype(np.float64)
    d = np.repeat(wq["scale"].view(np.float16).astype(np.float64), 32, 1)
    err = np.abs(oracle.dequant(wq) - raw)
    assert np.all(err <= 0.5 * d * (1 + 2.0 ** -9) + 1e-12)
    assert np.max(err / d) > 0.3


# ---------------------------------------------------------------- dependent chain
def _const_w(bits, n, k, code, scale, minv):
    q = np.full((n, k), code, np.uint8)
    return make_w(bits, q, np.full((n, k // 32), scale), None if bits == 2 else np.full((n, k // 32), minv))


def _const_gemv(c, k, w):
    """Closed form of a GEMV whose input is the constant fp32 vector c and whose weights
    are all w: each block has amax |c|, s = fp32(|c| / 127), every code is sign(c)*127,
    so y_r = k * w * sign(c) * 127 * s for every row (exact in fp64)."""
    c = np.float32(c)
    s = np.float32(np.float32(abs(c)) / np.float32(127.0))
    return float(k) * w * float(np.sign(c)) * 127.0 * float(s)


def test_chain_constant_closed_form():
    # (bits, n, k, code, scale, min, weight value, source)
    spec = [
        (4, 96, 64, 3, 0.5, -1.0, 0.5, -1),
        (4, 32, 96, 1, 0.25, -0.5, -0.25, 0),
        (6, 64, 32, 40, 0.0625, -2.0, 0.5, 1),
        (2, 32, 96, 3, 0.75, None, 0.75, 0),  # reads GEMV 0, not the latest output
    ]
    mats = [_const_w(b, n, k, c, d, m) for b, n, k, c, d, m, _, _ in spec]
    src = [t[7] for t in spec]
    x0 = np.full(64, 0.7, np.float32)
    outs = oracle.gemv_chain(mats, src, [x0])
    vals = []
    for j, (b, n, k, c, d, m, wv, sj) in enumerate(spec):
        cin = 0.7 if sj < 0 else np.float32(vals[sj])
        vals.append(_const_gemv(cin, k, wv))
        assert outs[j].shape == (n,)
        assert np.all(outs[j] == vals[j]), (j, outs[j][:3], vals[j])
    assert vals[0] > 0 and vals[1] < 0 and vals[2] < 0 and vals[3] > 0  # signs follow the weights
    assert len({round(v, 6) for v in vals}) == 4


def _random_chain():
    shapes = [(64, 96), (96, 64), (32, 96), (64, 64)]  # (n, k) per GEMV
    mats = [datagen.make_quantized(bits, 70 + i, n, k) for i, ((n, k), bits) in enumerate(zip(shapes, (4, 6, 2, 4)))]
    return mats, [-1, 0, 1, 0]


def test_chain_power_of_two_and_sign_equivariance():
    mats, src = _random_chain()
    x0 = datagen.normal_f32(71, 1, 96)
    base = oracle.gemv_chain(mats, src, [x0])
    four = oracle.gemv_chain(mats, src, [x0 * np.float32(4.0)])
    neg = oracle.gemv_chain(mats, src, [-x0])
    for a, b, c in zip(base, four, neg):
        assert np.array_equal(b, 4.0 * a)
        assert np.array_equal(c, -a)


def test_chain_hands_over_fp32():
    """A link reads the fp32 rounding of the earlier fp64 output: feeding GEMV 1 that
    rounding by hand gives the same vector bit for bit, while the chain input differs
    from the fp64 output itself."""
    mats, src = _random_chain()
    x0 = datagen.normal_f32(72, 1, 96)
    outs = oracle.gemv_chain(mats, src, [x0])
    assert not np.array_equal(outs[0].astype(np.float32).astype(np.float64), outs[0])
    assert np.array_equal(oracle.gemv(mats[1], outs[0].astype(np.float32)), outs[1])


def test_decode_chain_plan_shapes():
    """Every link of the decode chain reads a vector of its own k."""
    from datagen import workloads as W

    src, stages = W.decode_chain_plan(3)
    assert sum(stages) == len(src) == 21 and stages[:4] == [3, 1, 2, 1]
    for j, sj in enumerate(src):
        k = W.PROJ_SHAPES[j % 7][1]
        n_in = W.HIDDEN if sj < 0 else W.PROJ_SHAPES[sj % 7][0]
        assert n_in == k, (j, sj)
        assert sj < j
    # a link reads only outputs of earlier stages
    first = np.repeat(np.cumsum([0] + stages[:-1]), stages)
    assert all(sj < first[j] for j, sj in enumerate(src))


def test_logsumexp_infinities_match_scipy():
    """log sum exp with infinite terms: +inf if any term is +inf, -inf if all are -inf,
    -inf terms contribute nothing (scipy.special.logsumexp fixes these values)."""
    from scipy.special import logsumexp as sp_lse

    cases = [[np.inf, 1.0, -2.0], [-np.inf, -np.inf], [-np.inf, 0.5, 3.0], [np.inf, np.inf]]
    for c in cases:
        assert oracle.logsumexp(np.array(c)) == sp_lse(np.array(c)), c
    # NaN skipped, the rest as scipy
    assert oracle.logsumexp(np.array([np.nan, 1.0, 2.0])) == pytest.approx(sp_lse([1.0, 2.0]), rel=1e-15)
