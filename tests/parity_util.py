"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on
the same seeded, bf16-rounded inputs and compare with the stated tolerances.

Tolerances (from the method's accuracy targets for bf16 inputs with float32
accumulation):  O max-abs <= 1e-2, LSE max-abs <= 1e-3,
dQ/dK/dV max-abs <= 2e-2 * max|dX| (the oracle's), FP8 O max-abs <= 6e-2.
"""
import numpy as np
import torch

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_REL_TOL = 2e-2
FP8_O_TOL = 6e-2


def to64(t):
    return t.detach().to("cpu").double().numpy()


def assert_lse(gpu, ref, tol=LSE_TOL, what="lse"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ninf_g, ninf_r = np.isneginf(gpu), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), "%s: -inf pattern differs (%d vs %d rows)" % (
        what, ninf_g.sum(), ninf_r.sum())
    fin = ~ninf_r
    assert np.all(np.isfinite(gpu[fin])), "%s: non-finite values" % what
    err = np.max(np.abs(gpu[fin] - ref[fin])) if fin.any() else 0.0
    assert err <= tol, "%s max-abs error %.3e > %.1e" % (what, err, tol)
    return err


# O is written as bf16: its own rounding is up to 2^-9 |O| (half a bf16
# quantum).  Where a row averages only a few value rows (narrow sliding
# windows, the first rows of a causal mask) |O| stays near the size of single
# value rows (2 to 4 for N(0,1) data), and that rounding plus the bf16
# rounding of P can exceed the 1e-2 figure, which assumes many keys per row.
O_BF16_REL = 2.0 ** -9


def assert_o_bf16(gpu, ref, what="O"):
    """|gpu - ref| <= 1e-2 + 2^-9 |ref| element by element."""
    gpu = np.asarray(gpu, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), "%s: non-finite values" % what
    excess = np.abs(gpu - ref) - (O_TOL + O_BF16_REL * np.abs(ref))
    worst = float(np.max(excess)) if gpu.size else -1.0
    assert worst <= 0.0, "%s error exceeds 1e-2 + 2^-9|O| by %.3e" % (what, worst)
    return worst


def assert_close_abs(gpu, ref, tol, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), "%s: non-finite values" % what
    err = np.max(np.abs(gpu - ref)) if gpu.size else 0.0
    assert err <= tol, "%s max-abs error %.3e > %.3e" % (what, err, tol)
    return err


# A gradient that is identically zero in exact arithmetic (e.g. dQ with a single
# visible key) is computed on the GPU as P(dP - D) with dP from the tensor core
# and D from a float32 row sum: a ~1e-7 residue.  The relative criterion then
# degenerates, so an absolute floor of 1e-5 applies.
GRAD_ABS_FLOOR = 1e-5


def assert_grad(gpu, ref, what, tensor_maxabs=None):
    """max|gpu - ref| <= 2e-2 * (max-abs of the whole gradient tensor).

    `tensor_maxabs` is that max-abs when `ref` covers only sampled rows."""
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if tensor_maxabs is not None:
        scale = max(scale, float(tensor_maxabs))
    return assert_close_abs(gpu, ref, max(GRAD_REL_TOL * scale, GRAD_ABS_FLOOR), what)


def sample_rows(N, n, seed):
    """Sorted unique rows: the first, last and both sides of every 64/128 boundary
    near the start, plus random rows."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 63, 64, 127, 128, 129, 255, 256, N - 129, N - 128, N - 2, N - 1]
    rows = set(r for r in fixed if 0 <= r < N)
    rows.update(rng.integers(0, N, size=n).tolist())
    return sorted(rows)
