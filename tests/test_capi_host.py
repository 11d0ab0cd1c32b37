"""Host-only checks of the C ABI: the library builds and loads, exports every
declared entry point, and rejects bad arguments with the documented status
before touching the GPU."""
import ctypes
import os
import re

import pytest

import quantized_weight_gemv_gb300 as qg
from quantized_weight_gemv_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qg.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qgemv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_five_entry_points():
    names = declared_functions()
    for n in ("qgemv_q4", "qgemv_q6", "qgemv_batched", "cq_fwht_matvec", "vocab_softcap_argmax"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
        assert n in qg.SIGNATURES, n  # and the binding knows its signature


def test_status_strings_and_version(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert qg.status_string(code) not in ("", "unknown status")
    assert qg.status_string(-99) == "unknown status"
    assert lib.qg_version() >= 100
    assert 16 <= lib.qg_vocab_workspace_bytes() <= 4096  # a small fixed amount (counter and packed key)


P = ctypes.c_void_p
A16 = P(0x10000)      # a 16-byte aligned stand-in address: never dereferenced on these paths
MIS = P(0x10004)      # misaligned


def test_q4_validation(lib):
    f = lib.qgemv_q4
    assert f(A16, A16, A16, 4, 48, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG      # k % 32
    assert f(A16, A16, A16, -1, 64, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG     # n < 0
    assert f(A16, A16, A16, 4, 0, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG       # k == 0
    assert f(A16, A16, A16, 4, 65536 + 32, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(None, A16, A16, 4, 64, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(A16, A16, A16, 4, 64, None, A16, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(A16, A16, A16, 4, 64, A16, None, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(MIS, A16, A16, 4, 64, A16, A16, 0, None) == qg.QG_ERR_ALIGNMENT
    assert f(A16, A16, MIS, 4, 64, A16, A16, 0, None) == qg.QG_ERR_ALIGNMENT
    assert f(A16, A16, A16, 4, 64, MIS, A16, 0, None) == qg.QG_ERR_ALIGNMENT
    assert f(A16, A16, A16, 4, 64, A16, MIS, 0, None) == qg.QG_ERR_ALIGNMENT
    assert f(A16, A16, A16, 0, 64, A16, A16, 0, None) == qg.QG_OK                   # n == 0: nothing to do
    assert f(None, None, None, 0, 64, None, None, 0, None) == qg.QG_OK


def test_q6_and_batched_validation(lib):
    assert lib.qgemv_q6(A16, None, A16, A16, 4, 64, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG
    assert lib.qgemv_q6(A16, MIS, A16, A16, 4, 64, A16, A16, 0, None) == qg.QG_ERR_ALIGNMENT
    b = lib.qgemv_batched
    assert b(5, A16, None, A16, A16, 4, 64, 1, A16, A16, None, 0, 0, None) == qg.QG_ERR_UNSUPPORTED
    assert b(4, A16, A16, A16, A16, 4, 64, 1, A16, A16, None, 0, 0, None) == qg.QG_ERR_INVALID_ARG  # hi for Q4
    assert b(4, A16, None, A16, A16, 4, 64, 0, A16, A16, None, 0, 0, None) == qg.QG_ERR_INVALID_ARG
    assert b(4, A16, None, A16, A16, 4, 64, 17, A16, A16, None, 0, 0, None) == qg.QG_ERR_INVALID_ARG
    assert b(4, A16, None, A16, A16, 4, 16384, 16, A16, A16, None, 0, 0, None) == qg.QG_ERR_INVALID_ARG
    need = lib.qg_batched_workspace_bytes(4, 2048, 16)
    assert need > 0 and lib.qg_batched_workspace_bytes(4, 2048, 4) == 0 and lib.qg_batched_workspace_bytes(6, 2048, 16) == 0
    assert b(4, A16, None, A16, A16, 4, 2048, 16, A16, A16, A16, need - 1, 0, None) == qg.QG_ERR_WORKSPACE
    assert b(4, A16, None, A16, A16, 4, 2048, 16, A16, A16, MIS, need, 0, None) == qg.QG_ERR_ALIGNMENT


def test_cq_validation(lib):
    f = lib.cq_fwht_matvec
    assert f(A16, A16, A16, 8, 512, 100, 0, 8, A16, A16, 0, None) == qg.QG_ERR_UNSUPPORTED
    assert f(A16, A16, A16, 8, 768, 512, 0, 8, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG   # k % group
    assert f(A16, A16, A16, 8, 512, 512, 4, 5, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG   # range past n
    assert f(A16, A16, A16, 8, 512, 512, -1, 2, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(A16, A16, A16, 8, 512, 512, 0, 8, MIS, A16, 0, None) == qg.QG_ERR_ALIGNMENT
    assert f(A16, A16, A16, 8, 32768, 512, 0, 8, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(A16, A16, A16, 8, 512, 512, 3, 0, A16, A16, 0, None) == qg.QG_OK   # empty range


def test_vocab_validation(lib):
    f = lib.vocab_softcap_argmax
    ws = lib.qg_vocab_workspace_bytes()
    assert f(6, A16, A16, A16, A16, 0, 64, A16, 30.0, None, A16, A16, ws, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(6, A16, A16, A16, A16, 8, 64, A16, 30.0, None, A16, None, ws, 0, None) == qg.QG_ERR_WORKSPACE
    assert f(6, A16, A16, A16, A16, 8, 64, A16, 30.0, None, A16, A16, ws - 1, 0, None) == qg.QG_ERR_WORKSPACE
    assert f(6, A16, A16, A16, A16, 8, 64, A16, 30.0, None, None, A16, ws, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(6, A16, A16, A16, A16, 8, 64, A16, float("nan"), None, A16, A16, ws, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(6, A16, A16, A16, A16, 8, 64, A16, 30.0, MIS, A16, A16, ws, 0, None) == qg.QG_ERR_ALIGNMENT
    assert f(3, A16, A16, A16, A16, 8, 64, A16, 30.0, None, A16, A16, ws, 0, None) == qg.QG_ERR_UNSUPPORTED


def test_exposed_steps_validation(lib):
    assert lib.qg_quantize_act(A16, 48, 1, A16, A16, A16, None) == qg.QG_ERR_INVALID_ARG
    assert lib.qg_quantize_act(A16, 64, 0, A16, A16, A16, None) == qg.QG_ERR_INVALID_ARG
    assert lib.qg_quantize_act(MIS, 64, 1, A16, A16, A16, None) == qg.QG_ERR_ALIGNMENT
    assert lib.qg_blockdots(5, A16, None, 4, 64, A16, A16, None) == qg.QG_ERR_UNSUPPORTED
    assert lib.qg_blockdots(4, A16, None, 4, 64, MIS, A16, None) == qg.QG_ERR_ALIGNMENT
    assert lib.qg_blockdots(4, A16, None, 0, 64, None, None, None) == qg.QG_OK
    assert lib.qg_device_error(None) == qg.QG_ERR_INVALID_ARG


def test_binding_refuses_host_tensors():
    import torch
    t = torch.zeros(4, 32, dtype=torch.uint8)
    with pytest.raises(ValueError):
        qg.qgemv_q4(t, torch.zeros(4, 1, dtype=torch.float16), torch.zeros(4, 1, dtype=torch.float16),
                    torch.zeros(64))


def test_grouped_validation(lib):
    D = qg.GemvDesc
    ok = D(0x10000, None, 0x10000, 0x10000, 0x10000, 0x10000, 8, 2048)
    arr = (D * 2)(ok, ok)
    vp = ctypes.cast(arr, ctypes.c_void_p)
    need = lib.qg_grouped_workspace_bytes(vp, 2)
    assert need == 2 * 40 * 64
    assert lib.qg_grouped_workspace_bytes(None, 2) == 0
    f = lib.qgemv_grouped
    assert f(5, vp, 2, A16, need, 0, None) == qg.QG_ERR_UNSUPPORTED
    assert f(4, vp, 257, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(4, vp, 0, None, 0, 0, None) == qg.QG_OK
    assert f(4, None, 2, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(4, vp, 2, None, need, 0, None) == qg.QG_ERR_WORKSPACE
    assert f(4, vp, 2, A16, need - 1, 0, None) == qg.QG_ERR_WORKSPACE
    assert f(4, vp, 2, MIS, need, 0, None) == qg.QG_ERR_ALIGNMENT
    bad = (D * 1)(D(0x10000, None, 0x10000, 0x10000, 0x10000, 0x10000, 8, 1536))
    assert f(4, ctypes.cast(bad, ctypes.c_void_p), 1, A16, need, 0, None) == qg.QG_ERR_UNSUPPORTED
    bad = (D * 1)(D(0x10000, None, 0x10000, 0x10000, 0x10004, 0x10000, 8, 2048))
    assert f(4, ctypes.cast(bad, ctypes.c_void_p), 1, A16, need, 0, None) == qg.QG_ERR_ALIGNMENT
    bad = (D * 1)(D(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 8, 2048))  # hi given for Q4
    assert f(4, ctypes.cast(bad, ctypes.c_void_p), 1, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG
    empty = (D * 1)(D(None, None, None, None, None, None, 0, 2048))
    assert f(4, ctypes.cast(empty, ctypes.c_void_p), 1, None, 0, 0, None) == qg.QG_OK


def test_select_validation(lib):
    f = lib.qg_logits_select
    ws = lib.qg_select_workspace_bytes()
    assert ws >= 256 + 16 * 152
    assert f(A16, 0, None, 0, A16, A16, A16, ws, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(None, 8, None, 0, A16, A16, A16, ws, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(A16, 8, A16, -1, A16, A16, A16, ws, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(A16, 8, None, 0, A16, A16, A16, ws - 1, 0, None) == qg.QG_ERR_WORKSPACE
    assert f(A16, 8, None, 0, A16, A16, MIS, ws, 0, None) == qg.QG_ERR_ALIGNMENT
    g = lib.vocab_softcap_select
    vws = lib.qg_vocab_select_workspace_bytes()
    assert vws == lib.qg_vocab_workspace_bytes() + ws
    assert g(6, A16, A16, A16, A16, 8, 64, A16, 30.0, None, 0, None, A16, A16, A16, vws, 0, None) == qg.QG_ERR_INVALID_ARG
    assert g(6, A16, A16, A16, A16, 8, 64, A16, 30.0, None, 0, A16, A16, A16, A16, vws - 1, 0, None) == qg.QG_ERR_WORKSPACE
    assert g(3, A16, A16, A16, A16, 8, 64, A16, 30.0, None, 0, A16, A16, A16, A16, vws, 0, None) == qg.QG_ERR_UNSUPPORTED


def test_q2_validation(lib):
    f = lib.qgemv_q2
    assert f(A16, A16, 4, 48, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(MIS, A16, 4, 64, A16, A16, 0, None) == qg.QG_ERR_ALIGNMENT
    assert f(A16, None, 4, 64, A16, A16, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(None, None, 0, 64, None, None, 0, None) == qg.QG_OK
    b = lib.qgemv_batched
    assert b(2, A16, None, A16, A16, 4, 64, 1, A16, A16, None, 0, 0, None) == qg.QG_ERR_INVALID_ARG  # min given
    assert b(2, A16, A16, A16, None, 4, 64, 1, A16, A16, None, 0, 0, None) == qg.QG_ERR_INVALID_ARG  # hi given
    v = lib.vocab_softcap_argmax
    ws = lib.qg_vocab_workspace_bytes()
    assert v(2, A16, None, A16, A16, 8, 64, A16, 30.0, None, A16, A16, ws, 0, None) == qg.QG_ERR_INVALID_ARG
    assert lib.qgemv_grouped(2, A16, 1, A16, 16, 0, None) == qg.QG_ERR_UNSUPPORTED


def _chain_args(descs, sizes):
    D = qg.GemvDesc
    arr = (D * len(descs))(*descs)
    ps = (ctypes.c_int * len(sizes))(*sizes)
    return arr, ctypes.cast(arr, ctypes.c_void_p), ps, ctypes.cast(ps, ctypes.c_void_p)


def test_chain_validation(lib):
    D = qg.GemvDesc
    W = 0x10000  # weights stand-in
    X, Y1, Y2 = 0x100000, 0x200000, 0x300000
    d0 = D(W, None, W, W, X, Y1, 2048, 2048)        # phase 0 reads X
    d1 = D(W, None, W, W, Y1, Y2, 2048, 2048)       # phase 1 reads phase 0's output
    keep, vp, ps_keep, ps = _chain_args([d0, d1], [1, 1])
    need = lib.qg_chain_workspace_bytes(vp, 2, ps, 2)
    # control words and three regions of the largest phase's activation images (a phase's
    # own, and two for images produced by the phase before)
    assert need == qg.QG_CHAIN_CTL_BYTES + 3 * 40 * 64
    f = lib.qgemv_chain
    assert f(5, vp, 2, ps, 2, A16, need, 0, None) == qg.QG_ERR_UNSUPPORTED
    assert f(4, vp, 0, None, 0, None, 0, 0, None) == qg.QG_OK
    assert f(4, vp, 2, None, 2, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(4, vp, 2, ps, 0, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(4, vp, 2, ps, 3, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG     # more phases than GEMVs
    assert f(4, vp, 2, None, 2, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG
    assert f(4, vp, 2, ps, 2, None, need, 0, None) == qg.QG_ERR_WORKSPACE
    assert f(4, vp, 2, ps, 2, A16, need - 1, 0, None) == qg.QG_ERR_WORKSPACE
    assert f(4, vp, 2, ps, 2, MIS, need, 0, None) == qg.QG_ERR_ALIGNMENT
    # phase sizes must be >= 1 and sum to count
    for sizes in ([2, 0], [1, 2], [0, 2]):
        _, _, pk, p2 = _chain_args([d0, d1], sizes)
        assert f(4, vp, 2, p2, 2, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG, sizes
        assert lib.qg_chain_workspace_bytes(vp, 2, p2, 2) == 0
    # within one phase an output may not overlap an input or another output ...
    _, vp1, _, ps1 = _chain_args([d0, d1], [2])
    assert f(4, vp1, 2, ps1, 1, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG   # d1 reads d0's output
    inplace = D(W, None, W, W, X, X + 1024, 2048, 2048)  # y starts inside x
    _, vp2, _, ps2 = _chain_args([inplace], [1])
    assert f(4, vp2, 1, ps2, 1, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG
    two = [D(W, None, W, W, X, Y1, 2048, 2048), D(W, None, W, W, X, Y1 + 4096, 2048, 2048)]
    _, vp3, _, ps3 = _chain_args(two, [2])
    assert f(4, vp3, 2, ps3, 1, A16, need, 0, None) == qg.QG_ERR_INVALID_ARG   # outputs overlap
    # ... and the distinct inputs of a phase hold at most QG_CHAIN_MAX_PHASE_K values
    wide = [D(W, None, W, W, X + i * 0x20000, Y1 + i * 0x1000, 8, 16384) for i in range(3)]
    _, vp4, _, ps4 = _chain_args(wide, [3])
    big = lib.qg_chain_workspace_bytes(vp4, 3, ps4, 1)
    assert f(4, vp4, 3, ps4, 1, A16, big, 0, None) == qg.QG_ERR_UNSUPPORTED
    shared = [D(W, None, W, W, X, Y1 + i * 0x1000, 8, 16384) for i in range(3)]  # one input, three GEMVs
    _, vp5, _, ps5 = _chain_args(shared, [3])
    assert lib.qg_chain_workspace_bytes(vp5, 3, ps5, 1) == qg.QG_CHAIN_CTL_BYTES + 3 * (3 * 40 * 512)
    # descriptor rules as for qgemv_grouped
    for bad, rc in ((D(W, None, W, W, X, Y1, 8, 1536), qg.QG_ERR_UNSUPPORTED),
                    (D(W, None, W, W, X + 4, Y1, 8, 2048), qg.QG_ERR_ALIGNMENT),
                    (D(W, W, W, W, X, Y1, 8, 2048), qg.QG_ERR_INVALID_ARG),
                    (D(W, None, W, W, None, Y1, 8, 2048), qg.QG_ERR_INVALID_ARG)):
        _, vpb, _, psb = _chain_args([bad], [1])
        assert f(4, vpb, 1, psb, 1, A16, need, 0, None) == rc
    empty = D(None, None, None, None, None, None, 0, 2048)
    _, vpe, _, pse = _chain_args([empty, empty], [1, 1])
    assert f(4, vpe, 2, pse, 2, None, 0, 0, None) == qg.QG_OK
