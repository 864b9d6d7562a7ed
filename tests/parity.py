"""Parity bar shared by the GPU tests: GPU bf16 O and fp32 LSE against the fp64 oracle.

Bar: max|dO| <= 2e-2, mean|dO| <= 2e-3, max|dLSE| <= 1e-3, no NaN anywhere.
"""
import numpy as np

MAX_DO = 2e-2
MEAN_DO = 2e-3
MAX_DLSE = 1e-3


def parity_report(out_gpu, lse_gpu, out_ref, lse_ref):
    o = np.asarray(out_gpu.float().cpu().numpy() if hasattr(out_gpu, "cpu") else out_gpu,
                   dtype=np.float64)
    l = np.asarray(lse_gpu.float().cpu().numpy() if hasattr(lse_gpu, "cpu") else lse_gpu,
                   dtype=np.float64)
    do = np.abs(o - out_ref)
    dl = np.abs(l - lse_ref)
    return {
        "finite": bool(np.isfinite(o).all() and np.isfinite(l).all()),
        "max_dO": float(do.max()) if do.size else 0.0,
        "mean_dO": float(do.mean()) if do.size else 0.0,
        "max_dLSE": float(dl.max()) if dl.size else 0.0,
    }


def assert_parity(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    r = parity_report(out_gpu, lse_gpu, out_ref, lse_ref)
    assert r["finite"], f"{what}: non-finite output {r}"
    assert r["max_dO"] <= MAX_DO, f"{what}: {r}"
    assert r["mean_dO"] <= MEAN_DO, f"{what}: {r}"
    assert r["max_dLSE"] <= MAX_DLSE, f"{what}: {r}"
    return r
