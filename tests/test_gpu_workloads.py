"""GPU parity of the five workloads at their full sizes, in the launch configurations
bench.py times (CUDA-graph replays with programmatic dependent launch), against the
CPU oracle.

* single Q4 GEMV 1024x1024, seed 0;
* the decode-layer stream (tests/test_gpu_decode_stream.py covers it: every output of
  all 245 GEMVs);
* the Q6 vocabulary projection 262144x2048, seed 2, soft-cap 30, argmax (genie-ai-runtime,
  "What Gemma 4 E2B actually is": final-logit soft-capping), and constrained selection
  over its logits;
* small-batch Q4 MMVQ 16384x2048, seed 3, B in {1, 2, 4, 8, 16} (oxinfer README,
  "Speculative decoding": the multi-token int8 kernels), with and without a workspace;
* CQ matvec, hidden 512, 8192 and 1024 rows, seed 4 (needle.js "Inference backends",
  "Pure TypeScript").

fp32 outputs: |y - ref| <= 1e-3 * max(|ref|, rms(ref)) elementwise against the fp64
oracle.  Argmax: the lowest argmax of the kernel's own logits, always, and the
oracle's wherever its top-2 margin exceeds 2e-3 * max(|l1|, rms).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_weight_gemv_gb300 as qg
from datagen import workloads as W
from tests._gpu import DEV, TOL, assert_close, dev_w, oracle_gemv_par

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from quantized_weight_gemv_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    yield
    assert qg.device_error() == 0


def _graph(fn):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    return g


def _margin_ok(ref_l):
    """True when the oracle's top-2 margin clears the tolerance, so its argmax is decided."""
    order = np.argsort(-ref_l, kind="stable")
    rms = float(np.sqrt(np.mean(ref_l ** 2)))
    return ref_l[order[0]] - ref_l[order[1]] > 2 * TOL * max(abs(ref_l[order[0]]), rms)


# ---------------------------------------------------------------- single Q4 GEMV 1024 x 1024
def test_q4_single_as_benched():
    """64 back-to-back calls with programmatic dependent launch in one graph, as timed."""
    w, x = W.q4_single()
    wd = dev_w(w)
    xt = torch.from_numpy(x).to(DEV)
    ref = oracle.gemv(w, x)
    ys = [torch.full((1024,), float("nan"), device=DEV) for _ in range(64)]
    g = _graph(lambda: [qg.qgemv_q4(wd["lo"], wd["scale"], wd["min"], xt, y=y, flags=qg.QG_FLAG_PDL) for y in ys])
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    first = ys[0].cpu().numpy()
    assert_close(first.astype(np.float64), ref)
    for y in ys[1:]:
        assert np.array_equal(y.cpu().numpy(), first)


# ---------------------------------------------------------------- Q6 vocabulary head 262144 x 2048
@pytest.fixture(scope="module")
def vocab_q6():
    w, x = W.vocab_q6()
    ref_l = oracle.softcap(oracle_gemv_par(w, x), W.SOFTCAP)
    return w, dev_w(w), x, ref_l


def test_vocab_q6_as_benched(vocab_q6):
    """Full size: 262144 rows over 304 CTAs (about 862 rows and 13 ring laps per warp),
    the 304-way argmax merge, the seed's real top-2 margin."""
    w, wd, x, ref_l = vocab_q6
    xt = torch.from_numpy(x).to(DEV)
    logits = torch.full((W.VOCAB,), float("nan"), device=DEV)
    am = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    ws = qg.vocab_workspace(DEV)
    g = _graph(lambda: qg.vocab_softcap_argmax(6, wd["lo"], wd["hi"], wd["scale"], wd["min"], xt, W.SOFTCAP,
                                               logits=logits, argmax=am, ws=ws))
    for rep in range(2):
        logits.fill_(float("nan"))
        am.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        l = logits.cpu().numpy()
        assert_close(l.astype(np.float64), ref_l)
        idx = int(am.item())
        assert idx == oracle.argmax(l), rep
        if _margin_ok(ref_l):
            assert idx == oracle.argmax(ref_l), rep
    assert int(ws[:4].view(torch.int32).item()) == 0  # the completion counter is re-armed


def test_vocab_q6_select_as_benched(vocab_q6):
    """The one-launch constrained selection at full size over the benchmark's allowed list
    (about 1 % of the ids), and the same selection over the returned logits alone."""
    w, wd, x, ref_l = vocab_q6
    xt = torch.from_numpy(x).to(DEV)
    allowed = W.select_allowed()
    at = torch.from_numpy(allowed).to(DEV)
    logits = torch.empty(W.VOCAB, device=DEV)
    tok = torch.empty(1, dtype=torch.int32, device=DEV)
    lp = torch.empty(1, dtype=torch.float32, device=DEV)
    vws = qg.vocab_select_workspace(DEV)
    qg.vocab_softcap_select(6, wd["lo"], wd["hi"], wd["scale"], wd["min"], xt, W.SOFTCAP, allowed=at, logits=logits,
                            token=tok, logprob=lp, ws=vws)
    l = logits.cpu().numpy()
    assert_close(l.astype(np.float64), ref_l)
    own_tok, _ = oracle.select(l.astype(np.float64), allowed)
    assert int(tok.item()) == own_tok
    ref_tok, ref_lp = oracle.select(ref_l, allowed)
    cand = np.sort(ref_l[allowed])
    rms = float(np.sqrt(np.mean(ref_l ** 2)))
    if cand[-1] - cand[-2] > 2 * TOL * max(abs(cand[-1]), rms):
        assert int(tok.item()) == ref_tok
    assert abs(float(lp.item()) - ref_lp) <= TOL * max(1.0, abs(ref_lp))
    tok2, lp2 = qg.qg_logits_select(logits, at, ws=qg.select_workspace(DEV), flags=qg.QG_FLAG_PDL)
    assert int(tok2.item()) == own_tok
    assert abs(float(lp2.item()) - ref_lp) <= TOL * max(1.0, abs(ref_lp))


# ---------------------------------------------------------------- small-batch MMVQ 16384 x 2048
@pytest.fixture(scope="module")
def batched_q4():
    w = W.batched_q4_weights()
    Xall = W.batched_q4_x(max(W.BATCHES))
    refs = [oracle_gemv_par(w, Xall[b]) for b in range(max(W.BATCHES))]
    return w, dev_w(w), refs


@pytest.mark.parametrize("B", W.BATCHES)
def test_batched_q4_as_benched(batched_q4, B):
    """Every column of every batch size against the oracle: eager with and without the
    workspace, and three back-to-back PDL calls on one stream in a graph (as timed)."""
    w, wd, refs = batched_q4
    X = W.batched_q4_x(B)
    for b in range(B):  # column b of batch B is column b of the largest batch
        assert np.array_equal(X[b], W.batched_q4_x(max(W.BATCHES))[b])
    Xt = torch.from_numpy(X).to(DEV)
    for ws in ("auto", None):
        Y = qg.qgemv_batched(4, wd["lo"], None, wd["scale"], wd["min"], Xt, ws=ws).cpu().numpy()
        for b in range(B):
            assert_close(Y[b].astype(np.float64), refs[b])
    Ys = [torch.full((B, W.FFN), float("nan"), device=DEV) for _ in range(3)]
    g = _graph(lambda: [qg.qgemv_batched(4, wd["lo"], None, wd["scale"], wd["min"], Xt, Y=Y, flags=qg.QG_FLAG_PDL)
                        for Y in Ys])
    for Y in Ys:
        Y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for Y in Ys:
        Yh = Y.cpu().numpy()
        for b in range(B):
            assert_close(Yh[b].astype(np.float64), refs[b])


# ---------------------------------------------------------------- CQ matvec, hidden 512
@pytest.mark.parametrize("which", [0, 1])
def test_cq_as_benched(which):
    """64 back-to-back PDL calls in one graph (as timed), plus a row range of each."""
    m = W.cq_matrix(which)
    n = W.CQ_ROWS[which]
    x = W.cq_x()
    md = dev_w(m)
    xt = torch.from_numpy(x).to(DEV)
    ref = oracle.cq_matvec(m, x, W.CQ_GROUP)
    ys = [torch.full((n,), float("nan"), device=DEV) for _ in range(64)]
    g = _graph(lambda: [qg.cq_fwht_matvec(md["idx"], md["codebook"], md["row_scale"], xt, W.CQ_GROUP, y=y,
                                          flags=qg.QG_FLAG_PDL) for y in ys])
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    first = ys[0].cpu().numpy()
    assert_close(first.astype(np.float64), ref)
    for y in ys[1:]:
        assert np.array_equal(y.cpu().numpy(), first)
    r0, cnt = n // 3, n // 2
    yr = qg.cq_fwht_matvec(md["idx"], md["codebook"], md["row_scale"], xt, W.CQ_GROUP, r0, cnt).cpu().numpy()
    assert_close(yr.astype(np.float64), ref[r0:r0 + cnt])
