"""Comparison helpers shared by the GPU parity tests."""
import numpy as np

# Attention outputs: for every (row, head), max|o_gpu - o_ref| / max|o_ref| <= REL_TOL
# (bf16 outputs with fp32 accumulation against the fp64 oracle).
REL_TOL = 1e-2
# lse: natural-log log-sum-exp in fp32
LSE_ATOL = 2e-3


def rel_err_rows(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per (row, head) relative error of [..., H, 512] outputs."""
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    den = np.where(den > 0, den, 1.0)
    return num / den


def assert_out_close(got, ref, what=""):
    e = rel_err_rows(np.asarray(got, np.float64), np.asarray(ref, np.float64))
    assert float(e.max()) <= REL_TOL, f"{what}: max relative error {e.max():.3e}"
    return float(e.max())


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: lse finiteness differs"
    d = np.abs(got[fin] - ref[fin])
    assert d.size == 0 or float(d.max()) <= LSE_ATOL * (1 + np.abs(ref[fin]).max()), \
        f"{what}: lse error {d.max():.3e}"
