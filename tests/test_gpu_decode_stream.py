"""The decode-layer stream at its full size (35 layers x 7 Q4 projections, 245 GEMVs,
2.48 GB of packed weights), in the launch configurations bench.py times: one
qgemv_grouped call (quantisation + grouped GEMV chained by programmatic dependent
launch) captured in a CUDA graph and replayed, and one qgemv_q4 call per GEMV.  Every
output of every GEMV is compared with the oracle."""
import numpy as np
import pytest
import torch

import quantized_weight_gemv_gb300 as qg
from datagen import workloads as W
from tests._gpu import DEV, assert_close, dev_w, oracle_gemv_par

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def decode_stream():
    ws_np, xs_np = [], []
    for layer in range(W.N_LAYERS):
        for proj in range(7):
            w, x = W.decode_projection(layer, proj)
            ws_np.append(w)
            xs_np.append(x)
    mats = [dev_w(w) for w in ws_np]
    xs = [torch.from_numpy(x).to(DEV) for x in xs_np]
    refs = [oracle_gemv_par(w, x) for w, x in zip(ws_np, xs_np)]
    return mats, xs, refs


def _graph(fn):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    return g


def test_decode_stream_grouped_graph(decode_stream):
    mats, xs, refs = decode_stream
    ys = [torch.full((m["n"],), float("nan"), device=DEV) for m in mats]
    grouped = qg.GroupedGemv(4, mats, xs, ys, flags=qg.QG_FLAG_PDL)
    g = _graph(grouped.run)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for y, r in zip(ys, refs):
            assert_close(y.cpu().numpy().astype(np.float64), r)
    assert qg.device_error() == 0


def test_decode_stream_per_call(decode_stream):
    mats, xs, refs = decode_stream
    ys = [torch.full((m["n"],), float("nan"), device=DEV) for m in mats]
    g = _graph(lambda: [qg.qgemv_q4(m["lo"], m["scale"], m["min"], x, y=y, flags=qg.QG_FLAG_PDL)
                        for m, x, y in zip(mats, xs, ys)])
    g.replay()
    torch.cuda.synchronize()
    for y, r in zip(ys, refs):
        assert_close(y.cpu().numpy().astype(np.float64), r)
    assert qg.device_error() == 0
