"""Helpers shared by the GPU parity tests."""
import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle
import quantized_weight_gemv_gb300 as qg

# fp32 outputs: |y - ref| <= TOL * max(|ref|, rms(ref)) against the fp64 oracle
TOL = 1e-3
DEV = "cuda"


def dev_w(w):
    return qg.to_device(w, DEV)


def gpu_gemv(wd, x, flags=0):
    xt = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(DEV)
    if wd["bits"] == 2:
        y = qg.qgemv_q2(wd["lo"], wd["scale"], xt, flags=flags)
    elif wd["bits"] == 4:
        y = qg.qgemv_q4(wd["lo"], wd["scale"], wd["min"], xt, flags=flags)
    else:
        y = qg.qgemv_q6(wd["lo"], wd["hi"], wd["scale"], wd["min"], xt, flags=flags)
    return y.cpu().numpy().astype(np.float64)


def oracle_gemv_par(w, x, rows=None, threads=None):
    """The oracle over many rows, split across host threads (the C calls release the GIL)."""
    if rows is not None:
        return oracle.gemv_rows(w, x, rows)
    n = w["n"]
    threads = threads or min(32, os.cpu_count() or 1)
    bounds = [n * t // threads for t in range(threads + 1)]
    with cf.ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda t: oracle.gemv(w, x, bounds[t], bounds[t + 1] - bounds[t]), range(threads)))
    return np.concatenate(parts)


def assert_close(y, ref, tol=TOL):
    err = oracle.normwise_error(y, ref)
    assert np.all(np.isfinite(y)), "non-finite output"
    assert err <= tol, f"normwise error {err:.3e} > {tol}"
    return err
