"""The allocation-free grouped GEMV (qgemv_grouped_noalloc), called through the C ABI.

It is for callers that cannot allocate device memory: its scratch lives in a
fixed array inside the library instead of a caller workspace.  These tests check
that, on two calls in a row (the second one reusing the array the first one left
behind), its outputs agree with the allocating qgemv_grouped within the suite's
fp32 tolerance and with the CPU oracle; that two calls queued back to back with
programmatic dependent launch (the second one's quantisation overwriting the
array the first one reads) still give each group's own results; and that a group
too large for the array, or with a bad descriptor, is refused up front with the
allocating call's status.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import datagen
import oracle
import quantized_weight_gemv_gb300 as qg
from tests._gpu import DEV, TOL, assert_close, oracle_gemv_par

pytestmark = pytest.mark.gpu


def _group(bits, shapes, seed):
    mats, xs = [], []
    for i, (n, k) in enumerate(shapes):
        mats.append(qg.to_device(datagen.make_quantized(bits, seed + i, n, k), DEV))
        xs.append(torch.from_numpy(datagen.normal_f32(seed + i, 1, k)).to(DEV))
    return mats, xs


def _oracle_refs(bits, shapes, seed):
    return [oracle_gemv_par(datagen.make_quantized(bits, seed + i, n, k), datagen.normal_f32(seed + i, 1, k))
            for i, (n, k) in enumerate(shapes)]


def _descs(bits, mats, xs, ys):
    arr = (qg.GemvDesc * len(mats))()
    for i, (m, x, y) in enumerate(zip(mats, xs, ys)):
        arr[i] = qg.GemvDesc(m["lo"].data_ptr(), m["hi"].data_ptr() if bits == 6 else None, m["scale"].data_ptr(),
                             m["min"].data_ptr(), x.data_ptr(), y.data_ptr(), m["lo"].shape[0], m["lo"].shape[1] * 2)
    return arr


@pytest.fixture(scope="module", autouse=True)
def _built():
    from quantized_weight_gemv_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("bits", [4, 6])
def test_noalloc_matches_allocating_call_twice(bits):
    lib = qg.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two different groups, so that the second call runs over what the first left in the array
    for call, (shapes, seed) in enumerate((([(2048, 2048), (1024, 2048), (300, 16384), (16384, 2048)], 7000),
                                           ([(513, 8192), (2048, 1024), (77, 4096)], 7100))):
        mats, xs = _group(bits, shapes, seed)
        ref = [torch.empty(m["lo"].shape[0], device=DEV) for m in mats]
        qg.qgemv_grouped(bits, mats, xs, ref)
        ys = [torch.full((m["lo"].shape[0],), float("nan"), device=DEV) for m in mats]
        arr = _descs(bits, mats, xs, ys)
        rc = lib.qgemv_grouped_noalloc(bits, ctypes.cast(arr, ctypes.c_void_p), len(mats), 0, stream)
        assert rc == qg.QG_OK, qg.status_string(rc)
        torch.cuda.synchronize()
        for y, r, o in zip(ys, ref, _oracle_refs(bits, shapes, seed)):
            yh, rh = y.cpu().numpy().astype(np.float64), r.cpu().numpy().astype(np.float64)
            assert np.all(np.isfinite(yh)), f"call {call}: unwritten outputs"
            assert oracle.normwise_error(yh, rh) <= TOL, f"call {call}"
            assert_close(yh, o)
    assert qg.device_error() == 0


def test_noalloc_back_to_back_with_pdl():
    """Two calls on one stream with QG_FLAG_PDL: the second call's quantisation waits for
    the first call's GEMV (which reads the shared array) to finish, so each group gets its
    own activations."""
    lib = qg.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    groups = (([(16384, 2048), (2048, 16384), (1024, 2048)], 7200), ([(2048, 2048), (4096, 4096)], 7300))
    runs = []
    for shapes, seed in groups:
        mats, xs = _group(4, shapes, seed)
        ys = [torch.full((m["lo"].shape[0],), float("nan"), device=DEV) for m in mats]
        runs.append((shapes, seed, mats, xs, ys, _descs(4, mats, xs, ys)))
    torch.cuda.synchronize()
    for _, _, mats, _, _, arr in runs:
        rc = lib.qgemv_grouped_noalloc(4, ctypes.cast(arr, ctypes.c_void_p), len(mats), qg.QG_FLAG_PDL, stream)
        assert rc == qg.QG_OK, qg.status_string(rc)
    torch.cuda.synchronize()
    for shapes, seed, _, _, ys, _ in runs:
        for y, o in zip(ys, _oracle_refs(4, shapes, seed)):
            assert_close(y.cpu().numpy().astype(np.float64), o)
    assert qg.device_error() == 0


def test_noalloc_rejects_bad_descriptors_like_the_allocating_call():
    lib = qg.lib()
    arr = (qg.GemvDesc * 2)()
    ok = qg.GemvDesc(0x10000, None, 0x10000, 0x10000, 0x10000, 0x10000, 8, 2048)
    for bad, want in ((qg.GemvDesc(0x10000, None, 0x10000, 0x10000, 0x10000, 0x10000, 8, -2048),
                       qg.QG_ERR_UNSUPPORTED),
                      (qg.GemvDesc(0x10000, None, 0x10000, 0x10000, 0x10000, 0x10000, 8, 1 << 30),
                       qg.QG_ERR_UNSUPPORTED),
                      (qg.GemvDesc(0x10000, None, 0x10000, 0x10000, 0x10000, 0x10000, -1, 2048),
                       qg.QG_ERR_INVALID_ARG),
                      (qg.GemvDesc(0x10008, None, 0x10000, 0x10000, 0x10000, 0x10000, 8, 2048),
                       qg.QG_ERR_ALIGNMENT)):
        arr[0], arr[1] = ok, bad
        rc = lib.qgemv_grouped_noalloc(4, ctypes.cast(arr, ctypes.c_void_p), 2, 0, None)
        assert rc == want
        assert lib.qgemv_grouped(4, ctypes.cast(arr, ctypes.c_void_p), 2, None, 0, 0, None) == want


def test_noalloc_refuses_groups_beyond_its_array():
    lib = qg.lib()
    # 64 descriptors of k = 16384 need 64 * 20480 bytes = 1.25 MiB; 128 of them need 2.5 MiB > 2 MiB
    d = qg.GemvDesc(0x10000, None, 0x10000, 0x10000, 0x10000, 0x10000, 8, 16384)
    arr = (qg.GemvDesc * 128)(*([d] * 128))
    assert lib.qg_grouped_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), 128) > (2 << 20)
    rc = lib.qgemv_grouped_noalloc(4, ctypes.cast(arr, ctypes.c_void_p), 128, 0, None)
    assert rc == qg.QG_ERR_WORKSPACE
