"""GPU parity: the CUDA kernels, called through the C ABI, against the CPU oracle.

Integer work (activation codes, block dots, argmax) must match bit for bit;
fp32 outputs must be within TOL = 1e-3 of the fp64 oracle by the normwise rule
|y - ref| <= TOL * max(|ref|, rms(ref)).
"""
import numpy as np
import pytest
import torch

import datagen
import oracle
import quantized_weight_gemv_gb300 as qg
from tests._gpu import DEV, TOL, assert_close, dev_w, gpu_gemv, oracle_gemv_par
from tests._layout import make_w

pytestmark = pytest.mark.gpu

FLAGS = [0, qg.QG_FLAG_PLAIN, qg.QG_FLAG_PDL]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from quantized_weight_gemv_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    yield
    assert qg.device_error() == 0


# ---------------------------------------------------------------- activation quantisation (bit-exact)
def _special_x(k, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(k).astype(np.float32)
    nb = k // 32
    if nb > 1:
        x[32:64] = 0.0                           # all-zero block
    if nb > 2:
        x[64:96] = 0.0
        x[64 + 7] = -3.5                         # unit vector
    if nb > 3:
        x[96:128] *= 1e-30                       # tiny (subnormal scale)
    if nb > 4:
        x[128:160] = np.float32(127.0) * np.round(rng.standard_normal(32) * 20) / 127  # exact halves
    if nb > 5:
        x[160:192] *= 1e30
    return x


@pytest.mark.parametrize("k,batch", [(32, 1), (2048, 1), (16384, 1), (1024, 5)])
def test_quantize_act_bit_exact(k, batch):
    X = np.stack([_special_x(k, 100 + b) for b in range(batch)])
    xq, xs, xsum = qg.qg_quantize_act(torch.from_numpy(X).to(DEV))
    for b in range(batch):
        oq, os_, oS = oracle.quantize_act(X[b])
        assert np.array_equal(xq[b].cpu().numpy(), oq)
        assert np.array_equal(xs[b].cpu().numpy().view(np.uint32), os_.view(np.uint32))
        assert np.array_equal(xsum[b].cpu().numpy(), oS)


# ---------------------------------------------------------------- block dots (bit-exact)
@pytest.mark.parametrize("bits", [2, 4, 6])
@pytest.mark.parametrize("n,k", [(1, 32), (37, 96), (300, 2048)])
def test_blockdots_bit_exact(bits, n, k):
    rng = np.random.default_rng(n + k + bits)
    q = rng.integers(0, 1 << bits, size=(n, k), dtype=np.uint8)
    w = make_w(bits, q, 1.0, 0.0)
    xq = rng.integers(-127, 128, size=k).astype(np.int8)
    wd = dev_w(w)
    D = qg.qg_blockdots(bits, wd["lo"], wd.get("hi"), torch.from_numpy(xq).to(DEV)).cpu().numpy()
    assert np.array_equal(D, oracle.blockdots(w, xq))


def test_blockdots_extremes_bit_exact():
    """Largest magnitudes: codes 63 against xq = +-127 (|D| = 32*63*127)."""
    k = 64
    q = np.full((2, k), 63, np.uint8)
    q[1, ::2] = 0
    w = make_w(6, q, 1.0, 0.0)
    wd = dev_w(w)
    for v in (127, -127):
        xq = np.full(k, v, np.int8)
        D = qg.qg_blockdots(6, wd["lo"], wd["hi"], torch.from_numpy(xq).to(DEV)).cpu().numpy()
        assert np.array_equal(D, oracle.blockdots(w, xq))
        assert D[0, 0] == 32 * 63 * v


# ---------------------------------------------------------------- GEMV
SHAPES = [(1, 32), (7, 96), (33, 256), (100, 512), (1000, 1024), (1024, 1024), (333, 2048), (2049, 2048),
          (77, 4096), (19, 8192), (40, 16384), (3, 1056), (5, 32768), (1, 1536), (4, 1536), (1234, 1536),
          (3, 65536)]  # the largest k the calls accept (QG_MAX_K)


@pytest.mark.parametrize("bits", [2, 4, 6])
@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("flags", FLAGS)
def test_gemv_random(bits, n, k, flags):
    w = datagen.make_quantized(bits, 7 * n + k, n, k)
    x = datagen.normal_f32(7 * n + k, 1, k)
    y = gpu_gemv(dev_w(w), x, flags)
    assert_close(y, oracle.gemv(w, x))


@pytest.mark.parametrize("n,k", [(304 * 23 + 7, 1536), (304 * 37 + 5, 1024), (304 * 17 + 3, 2048),
                                 (304 * 9 + 1, 4096)])
def test_q2_stage_tails(n, k):
    """Q2 at one column streams 512-block stages (10 rows of k = 1536, 16 / 8 / 4 rows of
    k = 1024 / 2048 / 4096): with 2 CTAs per SM on 152 SMs each CTA here holds several
    full stages and a ragged last one.  GEMV and the soft-cap + argmax epilogue."""
    w = datagen.make_quantized(2, 31 * n + k, n, k)
    x = datagen.normal_f32(31 * n + k, 1, k)
    wd = dev_w(w)
    ref = oracle.gemv(w, x)
    for flags in (0, qg.QG_FLAG_PDL):
        assert_close(gpu_gemv(wd, x, flags), ref)
    _vocab_check(w, x, 30.0, 0)


@pytest.mark.parametrize("bits", [4, 6])
def test_gemv_special_activations(bits):
    n, k = 64, 2048
    w = datagen.make_quantized(bits, 55, n, k)
    wd = dev_w(w)
    for x in (np.zeros(k, np.float32), _special_x(k, 3)):
        for flags in (0, qg.QG_FLAG_PLAIN):
            y = gpu_gemv(wd, x, flags)
            ref = oracle.gemv(w, x)
            if not x.any():
                assert np.array_equal(y, np.zeros(n))
            else:
                assert_close(y, ref)


@pytest.mark.parametrize("bits", [4, 6])
def test_gemv_constant_code_closed_form(bits):
    """Constant-code rows: y = sum_b s_b * (scale*c + min) * S_b, checked against the oracle's closed form."""
    k = 1024
    cvals = [0, 5, 15] if bits == 4 else [0, 33, 63]
    q = np.array([[c] * k for c in cvals], np.uint8)
    w = make_w(bits, q, 0.0078125, -0.0625)
    x = datagen.normal_f32(12, 1, k)
    y = gpu_gemv(dev_w(w), x)
    xq, s, S = oracle.quantize_act(x)
    ref = np.array([sum(float(s[b]) * (0.0078125 * c - 0.0625) * int(S[b]) for b in range(k // 32)) for c in cvals])
    assert_close(y, ref)


def test_gemv_paths_agree():
    """The bulk-copy ring and the plain-load kernel give the same rows to fp32 rounding."""
    n, k = 4096, 2048
    w = datagen.make_quantized(4, 99, n, k)
    x = datagen.normal_f32(99, 1, k)
    wd = dev_w(w)
    a = gpu_gemv(wd, x, 0)
    b = gpu_gemv(wd, x, qg.QG_FLAG_PLAIN)
    assert oracle.normwise_error(a, b) < 1e-5


def test_gemv_outputs_only_their_rows():
    """Guard bands around y stay untouched (no out-of-range stores)."""
    n, k = 333, 2048
    w = datagen.make_quantized(4, 5, n, k)
    x = torch.from_numpy(datagen.normal_f32(5, 1, k)).to(DEV)
    wd = dev_w(w)
    for flags in (0, qg.QG_FLAG_PLAIN):
        buf = torch.full((n + 64,), float("nan"), device=DEV)
        y = buf[16:16 + n]
        qg.qgemv_q4(wd["lo"], wd["scale"], wd["min"], x, y=y, flags=flags)
        host = buf.cpu().numpy()
        assert np.all(np.isnan(host[:16])) and np.all(np.isnan(host[16 + n:]))
        assert np.all(np.isfinite(host[16:16 + n]))


def test_gemv_empty_is_noop():
    z = torch.zeros(0, 16, dtype=torch.uint8, device=DEV)
    h = torch.zeros(0, 1, dtype=torch.float16, device=DEV)
    y = qg.qgemv_q4(z, h, h, torch.zeros(32, device=DEV))
    assert y.numel() == 0


# ---------------------------------------------------------------- batched
@pytest.mark.parametrize("bits", [2, 4, 6])
@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("flags", [0, qg.QG_FLAG_PLAIN])
@pytest.mark.parametrize("k", [2048, 1536])
def test_batched(bits, batch, flags, k):
    n = 1000
    w = datagen.make_quantized(bits, 300 + batch, n, k)
    X = datagen.normal_f32(300 + batch, 1, batch * k).reshape(batch, k)
    wd = dev_w(w)
    Y = qg.qgemv_batched(bits, wd["lo"], wd.get("hi"), wd["scale"], wd["min"], torch.from_numpy(X).to(DEV),
                         flags=flags).cpu().numpy()
    for b in range(batch):
        assert_close(Y[b], oracle.gemv(w, X[b]))


def test_batched_columns_match_single():
    n, k, batch = 512, 2048, 4
    w = datagen.make_quantized(4, 31, n, k)
    X = datagen.normal_f32(31, 1, batch * k).reshape(batch, k)
    wd = dev_w(w)
    Y = qg.qgemv_batched(4, wd["lo"], None, wd["scale"], wd["min"], torch.from_numpy(X).to(DEV)).cpu().numpy()
    for b in range(batch):
        assert oracle.normwise_error(Y[b], gpu_gemv(wd, X[b])) < 1e-5


# ---------------------------------------------------------------- vocab soft-cap + argmax
def _vocab_check(w, x, softcap, flags=0, ws=None):
    wd = dev_w(w)
    xt = torch.from_numpy(x).to(DEV)
    logits, am = qg.vocab_softcap_argmax(w["bits"], wd["lo"], wd.get("hi"), wd["scale"], wd["min"], xt, softcap,
                                         ws=ws, flags=flags)
    l = logits.cpu().numpy()
    idx = int(am.item())
    ref_l = oracle.softcap(oracle_gemv_par(w, x), softcap)
    assert_close(l, ref_l)
    # exact self-consistency: the index is the lowest argmax of the returned logits
    assert idx == oracle.argmax(l)
    # against the oracle wherever its top-2 margin exceeds the tolerance
    order = np.argsort(-ref_l, kind="stable")
    rms = float(np.sqrt(np.mean(ref_l ** 2)))
    margin = ref_l[order[0]] - ref_l[order[1]] if ref_l.size > 1 else np.inf
    if margin > 2 * TOL * max(abs(ref_l[order[0]]), rms):
        assert idx == oracle.argmax(ref_l)
    # without logits the index is the same
    _, am2 = qg.vocab_softcap_argmax(w["bits"], wd["lo"], wd.get("hi"), wd["scale"], wd["min"], xt, softcap,
                                     logits=None, ws=ws, flags=flags)
    assert int(am2.item()) == idx
    return idx


@pytest.mark.parametrize("bits", [2, 4, 6])
@pytest.mark.parametrize("n,k", [(1, 32), (1000, 256), (5000, 2048), (3001, 1056), (700, 16384), (4099, 1536)])
@pytest.mark.parametrize("flags", [0, qg.QG_FLAG_PLAIN])
def test_vocab_random(bits, n, k, flags):
    w = datagen.make_quantized(bits, n + 3 * k, n, k)
    x = datagen.normal_f32(n + 3 * k, 1, k)
    _vocab_check(w, x, 30.0, flags)


@pytest.mark.parametrize("flags", [0, qg.QG_FLAG_PLAIN])
def test_vocab_planted_maximum_and_ties(flags):
    n, k = 20000, 2048
    rng = np.random.default_rng(8)
    q = rng.integers(0, 64, size=(n, k), dtype=np.uint8)
    q[12345] = 63
    q[17000] = 63      # an exact tie with a higher index: the lower one wins
    w = make_w(6, q, 0.001, 0.0)
    x = (np.abs(rng.standard_normal(k)) + 0.1).astype(np.float32)
    assert _vocab_check(w, x, 30.0, flags) == 12345


@pytest.mark.parametrize("k", [256, 1536])
@pytest.mark.parametrize("softcap", [30.0, 0.0])
@pytest.mark.parametrize("flags", [0, qg.QG_FLAG_PLAIN])
def test_vocab_argmax_order_edge_cases(k, softcap, flags):
    """The argmax order across CTAs on constructed logits (Q2, all codes 0, x = 127:
    every row's value is -nb * 8128 * scale exactly): all logits negative with the
    maximum tied between rows in different CTAs (the lower index wins), -0 against +0
    (equal: the lower index wins, whichever sign it has), every logit NaN (index 0),
    and NaN everywhere but one row."""
    n = 5000
    q = np.zeros((n, k), np.uint8)
    x = np.full(k, 127.0, np.float32)
    base = np.full(n, 2.0 ** -13)
    cases = []
    a = base.copy()
    a[[17, 4321]] = 2.0 ** -14
    cases.append((a, 17))
    for s2, s4000 in ((0.0, -0.0), (-0.0, 0.0)):
        a = base.copy()
        a[2], a[4000] = s2, s4000
        cases.append((a, 2))
    cases.append((np.full(n, np.nan), 0))
    a = np.full(n, np.nan)
    a[3333] = 2.0 ** -13
    cases.append((a, 3333))
    a = base.copy()
    a[0] = np.nan
    a[1] = 2.0 ** -14
    cases.append((a, 1))
    ws = qg.vocab_workspace(DEV)
    for scale, want in cases:
        w = make_w(2, q, np.repeat(scale[:, None], k // 32, axis=1), None)
        wd = dev_w(w)
        xt = torch.from_numpy(x).to(DEV)
        logits, am = qg.vocab_softcap_argmax(2, wd["lo"], None, wd["scale"], None, xt, softcap, ws=ws, flags=flags)
        l = logits.cpu().numpy()
        assert int(am.item()) == want == oracle.argmax(l), (want, int(am.item()))


def test_vocab_softcap_off_and_workspace_reuse():
    n, k = 4096, 2048
    w = datagen.make_quantized(6, 21, n, k)
    x = datagen.normal_f32(21, 1, k)
    ws = qg.vocab_workspace(DEV)
    a = _vocab_check(w, x, 0.0, ws=ws)
    b = _vocab_check(w, x, 30.0, ws=ws)
    assert a == b  # the cap is monotone
    assert int(ws[:4].view(torch.int32).item()) == 0  # the completion counter is re-armed


# ---------------------------------------------------------------- CQ
@pytest.mark.parametrize("group", [128, 256, 512, 1024])
@pytest.mark.parametrize("n,k_groups", [(1, 1), (1024, 1), (8192, 1), (333, 2), (50, 5), (777, 3), (8192, 4), (300, 8)])
def test_cq(group, n, k_groups):
    k = group * k_groups
    m = datagen.make_cq(4 + group, n, k)
    x = datagen.normal_f32(4 + group, 1, k)
    md = dev_w(m)
    y = qg.cq_fwht_matvec(md["idx"], md["codebook"], md["row_scale"], torch.from_numpy(x).to(DEV), group)
    assert_close(y.cpu().numpy(), oracle.cq_matvec(m, x, group))


@pytest.mark.parametrize("k,group", [(512, 512), (2048, 512), (2048, 256)])
def test_cq_row_ranges(k, group):
    n = 8192
    m = datagen.make_cq(4, n, k)
    x = datagen.normal_f32(4, 1, k)
    md = dev_w(m)
    xt = torch.from_numpy(x).to(DEV)
    full = oracle.cq_matvec(m, x, group)
    for start, count in ((0, 1), (5, 100), (8000, 192), (4096, 0), (1, 8191)):
        y = qg.cq_fwht_matvec(md["idx"], md["codebook"], md["row_scale"], xt, group, start, count).cpu().numpy()
        if count:
            assert_close(y, full[start:start + count])


@pytest.mark.parametrize("g,k_groups", [(512, 1), (512, 4), (256, 8), (1024, 2)])
def test_cq_constant_index_closed_form(g, k_groups):
    """Every index 7: each group's transformed values sum to sqrt(g) times its first
    element (the Hadamard matrix's column sums are g for column 0 and 0 for the others), so
    y = scale * C[7] * sqrt(g) * (sum of x[group start]) over the row's groups."""
    k = g * k_groups
    idx = np.full((4, k), 7, np.uint8)
    from tests._layout import f16_bits, pack_cq
    cb = np.linspace(-0.1, 0.1, 16).astype(np.float32)
    m = {"n": 4, "k": k, "idx": pack_cq(idx), "codebook": f16_bits(cb),
         "row_scale": f16_bits(np.array([0.5, 1.0, 1.25, 1.5], np.float32))}
    x = datagen.normal_f32(44, 1, k)
    md = dev_w(m)
    y = qg.cq_fwht_matvec(md["idx"], md["codebook"], md["row_scale"], torch.from_numpy(x).to(DEV), g).cpu().numpy()
    heads = float(np.sum(x[::g].astype(np.float64)))
    ref = m["row_scale"].view(np.float16).astype(np.float64) * float(np.float16(cb[7])) * np.sqrt(g) * heads
    assert_close(y, ref)


# ---------------------------------------------------------------- grouped
@pytest.mark.parametrize("bits", [4, 6])
def test_grouped_mixed_shapes(bits):
    shapes = [(2048, 2048), (1024, 2048), (7, 1024), (0, 2048), (300, 16384), (1, 4096), (513, 8192), (16384, 2048),
              (33, 1024), (2048, 16384)]
    mats, xs, ys, ws_np, x_np = [], [], [], [], []
    shared = datagen.normal_f32(999, 1, 2048)
    for i, (n, k) in enumerate(shapes):
        w = datagen.make_quantized(bits, 500 + i, n, k)
        x = shared if k == 2048 and i % 2 == 0 else datagen.normal_f32(500 + i, 1, k)
        ws_np.append(w)
        x_np.append(x)
        wd = dev_w(w)
        mats.append(wd)
        xs.append(torch.from_numpy(x).to(DEV))
        ys.append(torch.full((n,), float("nan"), device=DEV))
    for flags in (0, qg.QG_FLAG_PDL):
        for y in ys:
            y.fill_(float("nan"))
        qg.qgemv_grouped(bits, mats, xs, ys, flags=flags)
        for w, x, y in zip(ws_np, x_np, ys):
            if w["n"] == 0:
                continue
            ref = oracle_gemv_par(w, x) if w["n"] > 2000 else oracle.gemv(w, x)
            assert_close(y.cpu().numpy().astype(np.float64), ref)


def test_grouped_matches_single_calls_and_repeats():
    """The grouped launch and per-call launches give the same rows; repeated runs are identical."""
    shapes = [(2048, 2048), (1024, 2048), (1024, 2048), (2048, 2048), (16384, 2048), (16384, 2048), (2048, 16384)]
    mats, xs, ys = [], [], []
    for i, (n, k) in enumerate(shapes):
        w = datagen.make_quantized(4, 1000 + i, n, k)
        mats.append(dev_w(w))
        xs.append(torch.from_numpy(datagen.normal_f32(1000 + i, 1, k)).to(DEV))
        ys.append(torch.empty(n, device=DEV))
    g = qg.GroupedGemv(4, mats, xs, ys)
    g.run()
    first = [y.clone() for y in ys]
    g.run()
    for a, b, m, x in zip(first, ys, mats, xs):
        assert torch.equal(a, b)  # deterministic
        single = qg.qgemv_q4(m["lo"], m["scale"], m["min"], x)
        assert oracle.normwise_error(a.cpu().numpy(), single.cpu().numpy()) < 1e-5


def test_grouped_many_descriptors():
    """256 small descriptors (the maximum), each a few rows."""
    mats, xs, ys, ref = [], [], [], []
    for i in range(256):
        n = 1 + (i * 7) % 40
        w = datagen.make_quantized(4, 2000 + i, n, 1024)
        x = datagen.normal_f32(2000 + i, 1, 1024)
        mats.append(dev_w(w))
        xs.append(torch.from_numpy(x).to(DEV))
        ys.append(torch.empty(n, device=DEV))
        ref.append(oracle.gemv(w, x))
    qg.qgemv_grouped(4, mats, xs, ys)
    for y, r in zip(ys, ref):
        assert_close(y.cpu().numpy().astype(np.float64), r)


@pytest.mark.parametrize("batch", [8, 12, 16])
@pytest.mark.parametrize("k", [512, 1024, 2048, 4096])
def test_batched_tensor_core_with_and_without_workspace(batch, k):
    """The tensor-core path quantises once into a workspace, or per CTA without one; both match the oracle."""
    n = 777
    w = datagen.make_quantized(4, 900 + k + batch, n, k)
    X = datagen.normal_f32(900 + k + batch, 1, batch * k).reshape(batch, k)
    wd = dev_w(w)
    Xt = torch.from_numpy(X).to(DEV)
    refs = [oracle.gemv(w, X[b]) for b in range(batch)]
    for ws in ("auto", None):
        Y = qg.qgemv_batched(4, wd["lo"], None, wd["scale"], wd["min"], Xt, ws=ws).cpu().numpy()
        for b in range(batch):
            assert_close(Y[b], refs[b])


@pytest.mark.parametrize("batch", [8, 11, 16])
@pytest.mark.parametrize("k", [512, 1024, 2048])
def test_batched_tensor_core_launch_forms_identical(batch, k):
    """The tensor-core path's two forms make the same activation image, so the same bits:
    the image quantised once into a workspace (two launches) and every CTA quantising
    alone (no workspace); both against the oracle too.  Row counts below and above the
    grid, one ragged row group."""
    for n in (50, 16384 + 9):
        w = datagen.make_quantized(4, 2600 + k + batch + n, n, k)
        X = datagen.normal_f32(2600 + k + batch + n, 1, batch * k).reshape(batch, k)
        wd = dev_w(w)
        Xt = torch.from_numpy(X).to(DEV)
        Ya = qg.qgemv_batched(4, wd["lo"], None, wd["scale"], wd["min"], Xt, ws="auto").cpu().numpy()
        Yn = qg.qgemv_batched(4, wd["lo"], None, wd["scale"], wd["min"], Xt, ws=None).cpu().numpy()
        assert np.array_equal(Ya, Yn)
        for b in (0, batch // 2, batch - 1):
            assert_close(Ya[b], oracle_gemv_par(w, X[b]) if n > 1000 else oracle.gemv(w, X[b]))
    assert qg.device_error() == 0


@pytest.mark.parametrize("batch", [8, 12, 16])
@pytest.mark.parametrize("k", [512, 2048])
def test_batched_tensor_core_block_dot_exact(batch, k):
    """The tensor-core block dot is the exact integer sum of code x int8 activation.

    Only block 0 carries weight (scale 1, min 0; every other block scale 0, min 0), and
    every column has block-0 activations that are integers of absolute maximum 127, so
    s = 1, xq = x and each output is block 0's integer dot itself: the oracle's fp64
    value, compared bit for bit.  Rows 0-3 and columns 0-2 reach the extremes: all codes
    15 or 0 against all +127, all -127 and a +127 / -127 split of the block's halves."""
    n, nb = 150, k // 32
    rng = np.random.default_rng(7000 + k + batch)
    q = rng.integers(0, 16, (n, k)).astype(np.uint8)
    q[0], q[1] = 15, 0
    q[2, :16], q[2, 16:] = 15, 0
    q[3, :16], q[3, 16:] = 0, 15
    scale = np.zeros((n, nb))
    scale[:, 0] = 1.0
    w = make_w(4, q, scale, np.zeros((n, nb)))
    X = rng.integers(-127, 128, (batch, k)).astype(np.float32)
    X[:, 5] = 127.0
    X[0, :32], X[1, :32] = 127.0, -127.0
    X[2, :16], X[2, 16:32] = 127.0, -127.0
    wd = dev_w(w)
    Xt = torch.from_numpy(X).to(DEV)
    refs = [oracle.gemv(w, X[b]) for b in range(batch)]
    for b in range(batch):  # the reference is the integer dot itself
        assert np.array_equal(refs[b], (q[:, :32].astype(np.int64) @ X[b, :32].astype(np.int64)).astype(np.float64))
    for ws in ("auto", None):
        Y = qg.qgemv_batched(4, wd["lo"], None, wd["scale"], wd["min"], Xt, ws=ws).cpu().numpy()
        for b in range(batch):
            assert np.array_equal(Y[b].astype(np.float64), refs[b]), (ws, b)


# ---------------------------------------------------------------- constrained selection
def _allowed_cases(n, rng):
    yield None
    yield np.sort(rng.choice(n, size=max(1, n // 100), replace=False)).astype(np.int32)
    yield np.array([n - 1], np.int32)
    yield np.array([3, 3, -5, n + 7, 1], np.int32)  # duplicates and out-of-range IDs are ignored
    yield np.arange(n, dtype=np.int32)


@pytest.mark.parametrize("n", [1, 1000, 262144])
def test_logits_select(n):
    rng = np.random.default_rng(n)
    logits = (rng.standard_normal(n) * 5).astype(np.float32)
    logits[rng.integers(0, n, size=min(n, 50))] = np.float32(2.5)  # exact ties
    lt = torch.from_numpy(logits).to(DEV)
    ws = qg.select_workspace(DEV)
    for allowed in _allowed_cases(n, rng):
        at = None if allowed is None else torch.from_numpy(allowed).to(DEV)
        tok, lp = qg.qg_logits_select(lt, at, ws=ws)
        ref_tok, ref_lp = oracle.select(logits.astype(np.float64), allowed)
        assert int(tok.item()) == ref_tok
        if ref_tok < 0:
            assert np.isnan(float(lp.item()))  # nothing selectable
        else:
            assert abs(float(lp.item()) - ref_lp) <= TOL * max(1.0, abs(ref_lp))
    assert int(ws[:4].view(torch.int32).item()) == 0  # the completion counter is re-armed


def test_logits_select_nothing_allowed():
    lt = torch.randn(100, device=DEV)
    tok, lp = qg.qg_logits_select(lt, torch.tensor([200, -1], dtype=torch.int32, device=DEV))
    assert int(tok.item()) == -1 and np.isnan(float(lp.item()))


@pytest.mark.parametrize("bits", [2, 4, 6])
def test_vocab_softcap_select(bits):
    """One launch (the stream kernel's selection epilogue) for no list or up to
    QG_SELECT_FUSED_MAX_ALLOWED ids, two launches for a longer list (here 20000 ids,
    unsorted, with duplicates and out-of-range ids) or the plain kernel."""
    n, k = 40000, 1536 if bits == 2 else 2048
    w = datagen.make_quantized(bits, 66, n, k)
    x = datagen.normal_f32(66, 1, k)
    wd = dev_w(w)
    xt = torch.from_numpy(x).to(DEV)
    ref_l = oracle.softcap(oracle_gemv_par(w, x), 30.0)
    rng = np.random.default_rng(67)
    ws = qg.vocab_select_workspace(DEV)
    long_list = np.concatenate([rng.integers(0, n, 19990), [-3, n, n + 5, 7, 7, 7, 11, 0, 1, 2]]).astype(np.int32)
    for allowed in (None, np.sort(rng.choice(n, size=500, replace=False)).astype(np.int32), long_list):
        at = None if allowed is None else torch.from_numpy(allowed).to(DEV)
        for flags in (0, qg.QG_FLAG_PDL, qg.QG_FLAG_PLAIN):
            logits, tok, lp = qg.vocab_softcap_select(bits, wd["lo"], wd.get("hi"), wd["scale"], wd["min"], xt, 30.0,
                                                      allowed=at, ws=ws, flags=flags)
            l = logits.cpu().numpy()
            assert_close(l, ref_l)
            # exact against the GPU's own logits; against the oracle's when the margin clears the tolerance
            own_tok, _ = oracle.select(l.astype(np.float64), allowed)
            assert int(tok.item()) == own_tok
            ref_tok, ref_lp = oracle.select(ref_l, allowed)
            cand = ref_l if allowed is None else ref_l[np.unique(allowed[(allowed >= 0) & (allowed < n)])]
            top2 = np.sort(cand)[-2:]
            if top2[1] - top2[0] > 2 * TOL * max(abs(top2[1]), float(np.sqrt(np.mean(ref_l ** 2)))):
                assert int(tok.item()) == ref_tok
            assert abs(float(lp.item()) - ref_lp) <= TOL * max(1.0, abs(ref_lp))


@pytest.mark.parametrize("bits", [2, 4, 6])
@pytest.mark.parametrize("n", [1, 7, 33, 300, 1025])
def test_vocab_softcap_select_small_vocab(bits, n):
    """The one-launch selection on vocabularies smaller than or not divisible by the grid:
    every CTA's row range holds a few rows or one; no list, only out-of-range ids, one
    allowed id, and a duplicated list."""
    k = 1536 if bits == 2 else 2048
    w = datagen.make_quantized(bits, 1300 + n, n, k)
    x = datagen.normal_f32(1300 + n, 1, k)
    wd = dev_w(w)
    xt = torch.from_numpy(x).to(DEV)
    ws = qg.vocab_select_workspace(DEV)
    lists = (None, np.array([-1, n, n + 3], np.int32), np.array([n - 1], np.int32),
             np.array([0, n // 2, 0, n // 2, n - 1], np.int32))
    for allowed in lists:
        at = None if allowed is None else torch.from_numpy(allowed).to(DEV)
        logits, tok, lp = qg.vocab_softcap_select(bits, wd["lo"], wd.get("hi"), wd["scale"], wd["min"], xt, 30.0,
                                                  allowed=at, ws=ws)
        l = logits.cpu().numpy()
        own_tok, own_lp = oracle.select(l.astype(np.float64), allowed)
        assert int(tok.item()) == own_tok, (allowed, int(tok.item()), own_tok)
        if own_tok < 0:
            assert np.isnan(float(lp.item()))
        else:
            assert abs(float(lp.item()) - own_lp) <= TOL * max(1.0, abs(own_lp))
    # the four calls share one workspace: a counter left armed would break the next merge


# ---------------------------------------------------------------- 2-bit codes, zero point 2
def test_q2_zero_point_closed_forms():
    """Codes 2 decode to zero weights (y = 0 exactly); codes 3 give y = scale * sum(x_deq)."""
    k = 2048
    x = datagen.normal_f32(95, 1, k)
    xq, s, S = oracle.quantize_act(x)
    for code, ref in ((2, 0.0), (3, sum(0.25 * float(s[b]) * int(S[b]) for b in range(k // 32)))):
        w = make_w(2, np.full((40, k), code, np.uint8), 0.25, None)
        for flags in (0, qg.QG_FLAG_PLAIN):
            y = gpu_gemv(dev_w(w), x, flags)
            if code == 2:
                assert np.array_equal(y, np.zeros(40))
            else:
                assert_close(y, np.full(40, ref))


def test_q2_vocab_head_shape():
    """The pages' int2 LM head shape class: many rows, short k (262144 x 1536 there; 65536 x 2048 here)."""
    n, k = 65536, 2048
    w = datagen.make_quantized(2, 96, n, k)
    x = datagen.normal_f32(96, 1, k)
    _vocab_check(w, x, 30.0)


# ---------------------------------------------------------------- int8 decisions at ties
def _tie_x(k, seed):
    """Activations sitting on the quantiser's rounding boundaries: in every block one
    element is the maximum 127*c (so s = fl32(127c / 127)), the others fl32((j + 1/2) s)
    for random j, so x/s is a half-integer or within an ulp of one."""
    rng = np.random.default_rng(seed)
    nb = k // 32
    x = np.empty((nb, 32), np.float32)
    for b in range(nb):
        c = np.float32(rng.uniform(0.5, 2.0) * 2.0 ** rng.integers(-12, 12))
        amax = np.float32(np.float32(127.0) * c)
        s = np.float32(amax / np.float32(127.0))
        j = rng.integers(-127, 127, size=32).astype(np.float64)
        x[b] = (np.float32(1.0) * ((j + 0.5) * np.float64(s))).astype(np.float32)
        x[b, rng.integers(0, 32)] = amax * np.float32(rng.choice([-1.0, 1.0]))
    return x.ravel()


def _picker(n, k, col):
    """Q4 weights with scale 1, min 0 and code 1 at (r, col[r]), 0 elsewhere: row r of
    the GEMV is then s_b * xq[col[r]] exactly, the kernel's own int8 decision."""
    q = np.zeros((n, k), np.uint8)
    q[np.arange(n), col] = 1
    return make_w(4, q, np.ones((n, k // 32)), np.zeros((n, k // 32)))


def _expect_picked(x, col):
    xq, s, _ = oracle.quantize_act(x)
    return (s[col // 32].astype(np.float32) * xq[col].astype(np.float32)).astype(np.float32)


def test_quantize_act_ties_bit_exact():
    for k, seed in ((1024, 1), (16384, 2)):
        x = _tie_x(k, seed)
        xq, xs, xsum = qg.qg_quantize_act(torch.from_numpy(x).to(DEV))
        oq, os_, oS = oracle.quantize_act(x)
        assert np.array_equal(xq[0].cpu().numpy(), oq)
        assert np.array_equal(xs[0].cpu().numpy().view(np.uint32), os_.view(np.uint32))
        assert np.array_equal(xsum[0].cpu().numpy(), oS)
        # the inputs really sit on boundaries: many exact ties
        t = np.abs(x / np.repeat(os_, 32))
        assert np.sum(np.abs(t - np.floor(t) - 0.5) == 0) > k // 8


@pytest.mark.parametrize("k", [1024, 2048, 16384])
def test_int8_decisions_every_kernel(k):
    """Every kernel that quantises activations takes the oracle's int8 decisions on tie
    inputs: single-vector stream and plain kernels, the grouped and chain GEMVs, and the
    batched dp4a and tensor-core kernels."""
    n = 2048
    r = np.arange(n)
    col = r % k if k <= n else r * (k // n) + r % (k // n)  # every column, or spread over all positions
    w = dev_w(_picker(n, k, col))
    X = np.stack([_tie_x(k, 10 + b) for b in range(8)])
    Xt = torch.from_numpy(X).to(DEV)
    want = [_expect_picked(X[b], col) for b in range(8)]
    got = {}
    for flags in (0, qg.QG_FLAG_PLAIN):
        got[f"q4 flags={flags}"] = [qg.qgemv_q4(w["lo"], w["scale"], w["min"], Xt[0], flags=flags)]
    y = torch.empty(n, device=DEV)
    qg.qgemv_grouped(4, [w], [Xt[0]], [y])
    got["grouped"] = [y]
    yc = [torch.empty(n, device=DEV) for _ in range(2)]
    if k <= 16384:
        qg.qgemv_chain(4, [w, w], [Xt[0], Xt[1]], yc, [1, 1])
        got["chain"] = [yc[0], yc[1]]
    for B in (2, 8):
        Y = qg.qgemv_batched(4, w["lo"], None, w["scale"], w["min"], Xt[:B])
        got[f"batched B={B}"] = [Y[b] for b in range(B)]
    for name, ys in got.items():
        for b, yv in enumerate(ys):
            assert np.array_equal(yv.cpu().numpy().view(np.uint32), want[b].view(np.uint32)), (name, b)


def test_int2_vocab_head_pages_shape():
    """The int2 LM head at the pages' shape (262144 x 1536, Gemma WebGPU Engine "Roadmap")."""
    n, k = 262144, 1536
    w = datagen.make_quantized(2, 97, n, k)
    x = datagen.normal_f32(97, 1, k)
    _vocab_check(w, x, 30.0)


@pytest.mark.parametrize("k", [1536, 2048, 512])
@pytest.mark.parametrize("batch", [1, 2, 3, 4])
def test_q2_gemv_integer_exact(k, batch):
    """Q2 (zero point 2) with the zero-point term inside the integer dot: with weight
    scales 1 on three blocks of every row (0, 17 and the last: lanes of both half warps
    and all three of a lane's blocks at k = 1536), 0 elsewhere, and integer activations
    whose blocks all reach 127 (s = 1, xq = x), every output is the exact integer
    sum over those blocks of (code - 2) * x, the oracle's fp64 value, compared bit for
    bit.  Rows 0-3 reach the extremes (all codes 3 or 0, halves split)."""
    n, nb = 150, k // 32
    rng = np.random.default_rng(7100 + k + batch)
    q = rng.integers(0, 4, (n, k)).astype(np.uint8)
    q[0], q[1] = 3, 0
    q[2, ::2], q[3, 1::2] = 3, 0
    live = [0, 17 % nb, nb - 1]
    scale = np.zeros((n, nb))
    scale[:, live] = 1.0
    w = make_w(2, q, scale, None)
    X = rng.integers(-127, 128, (batch, k)).astype(np.float32)
    X[:, ::32] = 127.0
    X[0, :] = 127.0
    if batch > 1:
        X[1, :] = -127.0
        X[1, ::32] = 127.0
    wd = dev_w(w)
    Xt = torch.from_numpy(X).to(DEV)
    cols = np.concatenate([np.arange(32 * b, 32 * b + 32) for b in sorted(set(live))])
    for b in range(batch):  # the reference is the integer sum itself
        ref = oracle.gemv(w, X[b])
        want = (q[:, cols].astype(np.int64) - 2) @ X[b, cols].astype(np.int64)
        assert np.array_equal(ref, want.astype(np.float64))
    for ws in ("auto", None):
        Y = qg.qgemv_batched(2, wd["lo"], None, wd["scale"], None, Xt, ws=ws).cpu().numpy()
        for b in range(batch):
            assert np.array_equal(Y[b].astype(np.float64), oracle.gemv(w, X[b])), (ws, b)
    y = gpu_gemv(wd, X[0])
    assert np.array_equal(y, oracle.gemv(w, X[0]))


def test_logits_select_infinities():
    """An infinite logit: the log-sum-exp is +inf, the selected id is the +inf one when it
    is allowed (log-probability inf - inf = NaN on both sides); -inf logits are never
    better than finite ones and add nothing to the sum."""
    n = 5000
    v = datagen.normal_f32(77, 1, n)
    v[100] = -np.inf
    v[4000] = np.inf
    t = torch.from_numpy(v).to(DEV)
    for allowed in (None, np.array([5, 100, 4000], np.int32), np.array([5, 100], np.int32)):
        a = None if allowed is None else torch.from_numpy(allowed).to(DEV)
        tok, lp = qg.qg_logits_select(t, a)
        ref_tok, ref_lp = oracle.select(v.astype(np.float64), allowed)
        assert int(tok.item()) == ref_tok
        got = float(lp.item())
        assert (np.isnan(got) and np.isnan(ref_lp)) or got == ref_lp == -np.inf or abs(got - ref_lp) < 1e-9, (got, ref_lp)


# ---------------------------------------------------------------- split-K (short N, long K)
@pytest.mark.parametrize("bits", [2, 4, 6])
@pytest.mark.parametrize("k", [4096, 8192, 16384])
@pytest.mark.parametrize("n", [1, 5, 37, 300, 2048, 8192])
def test_gemv_split_k(bits, n, k):
    """Long activations and at most 8192 rows take the split-K kernel (clusters of k/2048
    CTAs, each one k slice, partial sums added in slice order through distributed shared
    memory): ragged row ranges per cluster, one row, more clusters than rows."""
    w = datagen.make_quantized(bits, 11 * n + k + bits, n, k)
    x = datagen.normal_f32(11 * n + k + bits, 1, k)
    wd = dev_w(w)
    ref = oracle_gemv_par(w, x) if n * k >= (1 << 24) else oracle.gemv(w, x)
    for flags in (0, qg.QG_FLAG_PDL):
        y = gpu_gemv(wd, x, flags)
        assert_close(y, ref)
    # deterministic: the slice order of the sum is fixed
    assert np.array_equal(gpu_gemv(wd, x), gpu_gemv(wd, x))


def test_gemv_split_k_down_projection_as_benched():
    """The decode stream's down projection (2048 x 16384, layer 0) as one call per matrix,
    24 back-to-back PDL calls in a CUDA graph (as timed), against the oracle."""
    from datagen import workloads as W
    w, x = W.decode_projection(0, 6)
    wd = dev_w(w)
    xt = torch.from_numpy(x).to(DEV)
    ref = oracle_gemv_par(w, x)
    ys = [torch.full((2048,), float("nan"), device=DEV) for _ in range(24)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for y in ys:
            qg.qgemv_q4(wd["lo"], wd["scale"], wd["min"], xt, y=y, flags=qg.QG_FLAG_PDL)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for y in ys:
            qg.qgemv_q4(wd["lo"], wd["scale"], wd["min"], xt, y=y, flags=qg.QG_FLAG_PDL)
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    first = ys[0].cpu().numpy()
    assert_close(first.astype(np.float64), ref)
    for y in ys[1:]:
        assert np.array_equal(y.cpu().numpy(), first)


# ---------------------------------------------------------------- 16-warp, whole-share-in-flight layout
@pytest.mark.parametrize("bits", [2, 4, 6])
@pytest.mark.parametrize("n,k", [(12345, 2048), (16384 + 77, 2048), (30001, 1024), (15003, 1536), (9300, 2048)])
@pytest.mark.parametrize("batch", [1, 2, 4])
def test_gemv_sixteen_warp_layout(bits, n, k, batch):
    """Shapes whose share per SM is 16 to 64 stages take one 16-warp CTA per SM with the
    first stage fetched before the dependency wait: ragged last stages and row ranges, one
    to four columns (four columns read their activation words from shared memory)."""
    w = datagen.make_quantized(bits, 13 * n + k + batch, n, k)
    X = datagen.normal_f32(13 * n + k + batch, 1, batch * k).reshape(batch, k)
    wd = dev_w(w)
    Xt = torch.from_numpy(X).to(DEV)
    for flags in (0, qg.QG_FLAG_PDL):
        Y = qg.qgemv_batched(bits, wd["lo"], wd.get("hi"), wd["scale"], wd["min"], Xt, flags=flags).cpu().numpy()
        for b in range(batch):
            assert_close(Y[b].astype(np.float64), oracle_gemv_par(w, X[b]))
