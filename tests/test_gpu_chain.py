"""GPU parity of the dependent GEMV chain (qgemv_chain) against the oracle's chain.

Both launch modes are covered: per-phase grouped launches (default) and the
persistent cooperative kernel (QG_FLAG_CHAIN_PERSISTENT)."""
import numpy as np
import pytest
import torch

import datagen
import oracle
import quantized_weight_gemv_gb300 as qg
from datagen import workloads as W
from tests._gpu import DEV, assert_close, dev_w, oracle_gemv_par

pytestmark = pytest.mark.gpu
MODES = [0, qg.QG_FLAG_CHAIN_PERSISTENT]


def _oracle_fn(w, x):
    return oracle_gemv_par(w, x) if w["n"] * w["k"] >= (1 << 22) else oracle.gemv(w, x)


def _run_spec(bits, spec, phase_sizes, ext, flags, seed):
    """spec: [(n, k, src)], src < 0 -> external input -src-1.  Returns (numpy weights,
    device outputs, chain object)."""
    ws_np, mats, xs, ys = [], [], [], []
    ext_t = [torch.from_numpy(e).to(DEV) for e in ext]
    for i, (n, k, src) in enumerate(spec):
        w = datagen.make_quantized(bits, seed + i, n, k)
        ws_np.append(w)
        mats.append(dev_w(w))
        ys.append(torch.full((n,), float("nan"), device=DEV))
    for i, (n, k, src) in enumerate(spec):
        xs.append(ext_t[-src - 1] if src < 0 else ys[src])
        assert xs[-1].numel() == k
    ch = qg.ChainGemv(bits, mats, xs, ys, phase_sizes, flags=flags)
    ch.run()
    return ws_np, ys, ch


SMALL = [  # (n, k, src); phases [3, 2, 1, 3]
    (2048, 1024, -1), (1000, 1024, -1), (4096, 2048, -2),
    (1024, 2048, 0), (7, 4096, 2),
    (16384, 1024, 3),
    (300, 16384, 5), (1, 1024, 3), (513, 8192, -3),
]


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("flags", MODES)
def test_chain_small(bits, flags):
    ext = [datagen.normal_f32(40, 1, 1024), datagen.normal_f32(41, 1, 2048), datagen.normal_f32(42, 1, 8192)]
    ws_np, ys, _ = _run_spec(bits, SMALL, [3, 2, 1, 3], ext, flags, 300)
    refs = oracle.gemv_chain(ws_np, [s for _, _, s in SMALL], ext, _oracle_fn)
    for y, r in zip(ys, refs):
        assert_close(y.cpu().numpy().astype(np.float64), r)


PRODUCED = [  # (n, k, src); phases [3, 3, 1, 2]
    (8192, 1024, -1), (16384, 2048, -2), (300, 1024, -1),  # 0-2: short inputs
    (8192, 8192, 0), (1024, 16384, 1), (777, 8192, 0),    # 3-5: long inputs, all outputs of phase 0
    (2048, 8192, 3),                                       # 6: long input, output of phase 1
    (1024, 2048, 6), (512, 16384, 1),                      # 7-8: one input from phase 2, one from phase 0
]


@pytest.mark.parametrize("bits", [4, 6])
def test_chain_produced_images(bits):
    """Per-phase mode: a phase with long inputs that are whole outputs of the phase before
    takes its activation images from that phase, whose CTAs (their rows aligned to whole
    blocks of 32) quantise their own rows once stored.  Phase 1 takes three images from phase 0 (two of them of
    one output), phase 2 one from phase 1 (a phase whose own images were produced), phase 3
    quantises for itself (one input comes from two phases back).  Against the oracle,
    identical over repeated calls on one workspace, and bit-identical to the persistent
    kernel, which quantises every input itself."""
    ext = [datagen.normal_f32(60, 1, 1024), datagen.normal_f32(61, 1, 2048)]
    ws_np, ys, ch = _run_spec(bits, PRODUCED, [3, 3, 1, 2], ext, 0, 700)
    refs = oracle.gemv_chain(ws_np, [s for _, _, s in PRODUCED], ext, _oracle_fn)
    first = [y.cpu().numpy() for y in ys]
    for y, r in zip(first, refs):
        assert_close(y.astype(np.float64), r)
    for _ in range(2):
        for y in ys:
            y.fill_(float("nan"))
        ch.run()
        torch.cuda.synchronize()
        assert all(np.array_equal(y.cpu().numpy(), f) for y, f in zip(ys, first))
    _, ys_p, _ = _run_spec(bits, PRODUCED, [3, 3, 1, 2], ext, qg.QG_FLAG_CHAIN_PERSISTENT, 700)
    assert all(np.array_equal(y.cpu().numpy(), f) for y, f in zip(ys_p, first))
    assert qg.device_error() == 0


@pytest.mark.parametrize("flags", MODES)
def test_chain_buffer_reuse_and_repeat(flags):
    """Ping-pong buffers: phase f writes the vector phase f-1 read.  Repeated calls on one
    workspace give identical results and leave its control words zero."""
    n = 2048
    A = torch.full((n,), float("nan"), device=DEV)
    B = torch.full((n,), float("nan"), device=DEV)
    x0 = datagen.normal_f32(50, 1, n)
    X = torch.from_numpy(x0).to(DEV)
    ws_np = [datagen.make_quantized(4, 600 + i, n, n) for i in range(6)]
    mats = [dev_w(w) for w in ws_np]
    xs = [X, A, B, A, B, A]
    ys = [A, B, A, B, A, B]
    ch = qg.ChainGemv(4, mats, xs, ys, [1] * 6, flags=flags)
    refs = oracle.gemv_chain(ws_np, [-1, 0, 1, 2, 3, 4], [x0])
    prev = None
    for rep in range(3):
        A.fill_(float("nan"))
        B.fill_(float("nan"))
        ch.run()
        torch.cuda.synchronize()
        a, b = A.cpu().numpy(), B.cpu().numpy()
        assert_close(a.astype(np.float64), refs[4])
        assert_close(b.astype(np.float64), refs[5])
        if prev is not None:
            assert np.array_equal(a, prev[0]) and np.array_equal(b, prev[1])
        prev = (a, b)
        assert int(ch.ws[:qg.QG_CHAIN_CTL_BYTES].count_nonzero()) == 0
    assert qg.device_error() == 0


def test_chain_one_phase_equals_grouped():
    shapes = [(2048, 2048), (1024, 2048), (16384, 2048), (2048, 16384), (33, 1024)]
    mats, xs, ys, yg = [], [], [], []
    for i, (n, k) in enumerate(shapes):
        mats.append(dev_w(datagen.make_quantized(4, 700 + i, n, k)))
        xs.append(torch.from_numpy(datagen.normal_f32(700 + i, 1, k)).to(DEV))
        ys.append(torch.empty(n, device=DEV))
        yg.append(torch.empty(n, device=DEV))
    qg.ChainGemv(4, mats, xs, ys, [len(shapes)]).run()
    qg.qgemv_grouped(4, mats, xs, yg)
    for a, b in zip(ys, yg):
        assert torch.equal(a, b)


@pytest.fixture(scope="module")
def decode_chain():
    """The 35-layer decode chain's weights (numpy and device) and the oracle's outputs."""
    src, stages = W.decode_chain_plan(W.N_LAYERS)
    ws_np = [W.decode_projection(j // 7, j % 7)[0] for j in range(len(src))]
    mats = [dev_w(w) for w in ws_np]
    x0 = W.decode_chain_x()
    refs = oracle.gemv_chain(ws_np, src, [x0], _oracle_fn)
    return src, stages, mats, x0, refs, ws_np


def _decode_run(dc, flags, x0=None):
    src, stages, mats, x_ref, _, _ = dc
    X = torch.from_numpy(x_ref if x0 is None else x0).to(DEV)
    ys = [torch.full((W.PROJ_SHAPES[j % 7][0],), float("nan"), device=DEV) for j in range(len(src))]
    xs = [X if s < 0 else ys[s] for s in src]
    ch = qg.ChainGemv(4, mats, xs, ys, stages, flags=flags)
    ch.run()
    return ch, ys, X


def _near_tie(x, s, i):
    """Margin of element i from a rounding boundary of the int8 quantiser, in steps."""
    t = abs(float(np.float32(x[i]) / np.float32(s[i // 32])))
    return abs(t - np.floor(t) - 0.5)


@pytest.mark.parametrize("flags", MODES)
def test_decode_chain_full_size(decode_chain, flags):
    """The 35-layer decode chain (245 GEMVs, 140 phases, 2.48 GB), every output of every GEMV
    against the oracle.

    Each link is one quantised GEMV of the vector it read (Gemma WebGPU Engine,
    "Roadmap": each projection reads the buffer the previous one wrote), so every one of
    the 245 outputs is compared, at 1e-3, with the oracle's GEMV of the same weights on
    the fp32 vector the link actually read (the kernel's output of the link before, or
    the external input).

    The oracle's own end-to-end chain is a diagnostic beside it: a chain of quantised
    GEMVs is defined up to the int8 decisions of its hand-offs (fp32 sums of another
    order can move an element that sits on a rounding boundary to the other side; both
    decisions are correct), so up to the first link whose int8 input codes differ from
    the oracle chain's, every output also matches the oracle chain, and at that link
    every differing code is off by one at a near-tie of the oracle's own quantisation."""
    src, _, mats, x0, refs, ws_np = decode_chain
    _, ys, X = _decode_run(decode_chain, flags)
    torch.cuda.synchronize()
    host = [y.cpu().numpy() for y in ys]
    for j in range(len(src)):
        x_read = x0 if src[j] < 0 else host[src[j]]
        assert np.all(np.isfinite(x_read)), j
        assert_close(host[j].astype(np.float64), _oracle_fn(ws_np[j], x_read))
    checked = 0
    for j in range(len(src)):
        x_dev = X if src[j] < 0 else ys[src[j]]
        x_or = x0 if src[j] < 0 else refs[src[j]].astype(np.float32)
        gq = qg.qg_quantize_act(x_dev)[0].cpu().numpy().ravel()
        oq, os_, _ = oracle.quantize_act(x_or)
        diff = np.where(gq != oq)[0]
        if diff.size:
            for i in diff:
                assert abs(int(gq[i]) - int(oq[i])) == 1, (j, i)
                assert _near_tie(x_or, os_, i) < 1e-3, (j, i, _near_tie(x_or, os_, i))
            break
        assert_close(host[j].astype(np.float64), refs[j])
        checked += 1
    assert checked >= 14, f"only {checked} links before the first tie"  # at least two whole layers
    assert qg.device_error() == 0


def test_decode_chain_modes_identical_and_equivariant(decode_chain):
    """Both launch modes give the same bits; scaling the input by 4 scales every output
    by exactly 4, and negating it negates every output (the activation quantisation is
    per-block scale-invariant, exact under powers of two and under sign)."""
    x0 = decode_chain[3]
    ch, ys, X = _decode_run(decode_chain, 0)
    base = [y.clone() for y in ys]
    _, ys2, _ = _decode_run(decode_chain, qg.QG_FLAG_CHAIN_PERSISTENT)
    for a, b in zip(base, ys2):
        assert torch.equal(a, b)
    for factor in (4.0, -1.0):
        X.copy_(torch.from_numpy(x0 * np.float32(factor)))
        ch.run()
        for a, b in zip(base, ys):
            assert torch.equal(b, a * factor)
    assert torch.isfinite(base[-1]).all()


def test_chain_abort_word_stops_and_rearms():
    """Persistent kernel: a set abort word makes every CTA stop at its next phase boundary
    without waiting out the barrier - no output of a phase after the first is written by
    any CTA, and the device error word records the stop (16) - the workspace comes back
    zero and the next call is correct."""
    n = 2048
    ws_np = [datagen.make_quantized(4, 800 + i, n, n) for i in range(4)]
    mats = [dev_w(w) for w in ws_np]
    x0 = datagen.normal_f32(80, 1, n)
    X = torch.from_numpy(x0).to(DEV)
    ys = [torch.full((n,), float("nan"), device=DEV) for _ in range(4)]
    ch = qg.ChainGemv(4, mats, [X, ys[0], ys[1], ys[2]], ys, [1, 1, 1, 1], flags=qg.QG_FLAG_CHAIN_PERSISTENT)
    assert qg.device_error() == 0
    ctl = ch.ws[:qg.QG_CHAIN_CTL_BYTES].view(torch.int32)
    ctl[1] = 1
    torch.cuda.synchronize()
    ch.run()
    torch.cuda.synchronize()
    for y in ys[1:]:  # every CTA stopped at the first boundary
        assert bool(torch.isnan(y).all())
    assert int(ch.ws[:qg.QG_CHAIN_CTL_BYTES].count_nonzero()) == 0
    assert qg.device_error() == 16
    ch.run()
    refs = oracle.gemv_chain(ws_np, [-1, 0, 1, 2], [x0])
    for y, r in zip(ys, refs):
        assert_close(y.cpu().numpy().astype(np.float64), r)


@pytest.mark.parametrize("flags", MODES)
def test_chain_empty_descriptors_and_phases(flags):
    """Descriptors with n = 0 are skipped, and a phase made only of them adds no boundary."""
    n, k = 1024, 1024
    ws_np = [datagen.make_quantized(4, 900 + i, n, k) for i in range(3)]
    mats = [dev_w(w) for w in ws_np]
    empty = dict(mats[0])
    empty["lo"] = mats[0]["lo"][:0]
    empty["scale"] = mats[0]["scale"][:0]
    empty["min"] = mats[0]["min"][:0]
    empty["n"] = 0
    x0 = datagen.normal_f32(91, 1, k)
    X = torch.from_numpy(x0).to(DEV)
    ys = [torch.full((n,), float("nan"), device=DEV) for _ in range(3)]
    ye = [torch.empty(0, device=DEV) for _ in range(3)]
    # phases: [g0, empty] [empty] [g1, empty] [g2]
    descs = [mats[0], empty, empty, mats[1], empty, mats[2]]
    xs = [X, X, X, ys[0], ys[0], ys[1]]
    outs = [ys[0], ye[0], ye[1], ys[1], ye[2], ys[2]]
    qg.ChainGemv(4, descs, xs, outs, [2, 1, 2, 1], flags=flags).run()
    refs = oracle.gemv_chain(ws_np, [-1, 0, 1], [x0])
    for y, r in zip(ys, refs):
        assert_close(y.cpu().numpy().astype(np.float64), r)
    assert qg.device_error() == 0


@pytest.mark.parametrize("flags", MODES)
def test_chain_in_cuda_graph(flags):
    """The chain captured in a CUDA graph and replayed gives the eager call's bits."""
    spec = [(2048, 2048, -1), (2048, 2048, 0), (16384, 2048, 1), (2048, 16384, 2)]
    ext = [datagen.normal_f32(92, 1, 2048)]
    ws_np, ys, ch = _run_spec(4, spec, [1, 1, 1, 1], ext, flags, 950)
    eager = [y.clone() for y in ys]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ch.run()
    for _ in range(2):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, ys):
            assert torch.equal(a, b)
    refs = oracle.gemv_chain(ws_np, [s_ for _, _, s_ in spec], ext, _oracle_fn)
    for y, r in zip(ys, refs):
        assert_close(y.cpu().numpy().astype(np.float64), r)


def _random_reuse_chain(rng, pool_n, n_buf):
    """Phases over a pool of reused buffers: (n, k, x buffer, y buffer) per GEMV and the
    phase sizes; within a phase no output overlaps another output or an input."""
    spec, sizes = [], []
    for _ in range(rng.randint(2, 7)):
        used_out, ins, phase, inputs = [], [], [], set()
        for _ in range(rng.randint(1, 4)):
            k = rng.choice([1024, 2048, 4096, 16384])
            n = rng.choice([256, 512, 2048])
            xi = rng.choice([b for b in range(n_buf) if b not in used_out])
            if sum(kk for _, kk in inputs | {(xi, k)}) > 32768:  # distinct inputs of a phase
                break
            inputs.add((xi, k))
            outs = [b for b in range(n_buf) if b not in used_out and b not in ins and b != xi]
            if not outs:
                break
            yi = rng.choice(outs)
            ins.append(xi)
            used_out.append(yi)
            phase.append((n, k, xi, yi))
        if phase and not any(o in ins for o in used_out):
            spec += phase
            sizes.append(len(phase))
    return spec, sizes


@pytest.mark.parametrize("flags", MODES)
def test_chain_reused_buffers_match_phase_by_phase(flags):
    """Random chains whose phases read, overwrite and reuse a small pool of buffers (a
    later phase may overwrite what an earlier one read, or write where an earlier one
    wrote): the chain leaves every buffer bit-identical to running the phases one by one
    as separate qgemv_grouped calls with a device synchronisation between them."""
    import random

    rng = random.Random(77)
    pool_n, n_buf = 16384, 6
    for trial in range(16):
        spec, sizes = _random_reuse_chain(rng, pool_n, n_buf)
        init = torch.from_numpy(np.stack([datagen.normal_f32(900 + trial, b, pool_n) for b in range(n_buf)])).to(DEV)
        mats = [dev_w(datagen.make_quantized(4, 5000 + 100 * trial + i, n, k)) for i, (n, k, _, _) in enumerate(spec)]

        def views(pool):
            return ([pool[xi, :k] for (n, k, xi, yi) in spec], [pool[yi, :n] for (n, k, xi, yi) in spec])

        pa = init.clone()
        xa, ya = views(pa)
        qg.ChainGemv(4, mats, xa, ya, sizes, flags=flags).run()
        pb = init.clone()
        xb, yb = views(pb)
        off = 0
        for m in sizes:
            qg.qgemv_grouped(4, mats[off:off + m], xb[off:off + m], yb[off:off + m])
            torch.cuda.synchronize()
            off += m
        torch.cuda.synchronize()
        assert torch.equal(pa, pb), (trial, sizes)
    assert qg.device_error() == 0
