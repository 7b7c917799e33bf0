"""Shared helpers of the GPU parity tests (tolerances, transfers, oracle calls)."""
import numpy as np
import torch

import oracle
import st24_inputs as inputs

# Tolerances on max|C| (of the oracle), by input type; bf16/f16 outputs may
# also differ by one unit in the last place of the output type (rounding).
REL_TOL = {"f16": 2e-3, "bf16": 2e-3, "e4m3": 2e-2, "s8": 0.0}


def bits(t: torch.Tensor) -> np.ndarray:
    return inputs.raw(t.detach().to("cpu").contiguous()).numpy()


def ulp(x: np.ndarray, c: str) -> np.ndarray:
    """One unit in the last place of |x| in the output type (0 for f32/s32)."""
    if c not in ("bf16", "f16"):
        return np.zeros_like(x)
    mant = 7 if c == "bf16" else 10
    tiny = 2.0 ** -133 if c == "bf16" else 2.0 ** -24
    ax = np.maximum(np.abs(x), tiny)
    return np.exp2(np.floor(np.log2(ax)) - mant)


def assert_close(got: np.ndarray, ref: np.ndarray, ab: str, c: str, what: str = ""):
    """|got - ref| <= tol * max|ref| (+ 1 ulp of the output type), elementwise."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if c == "s32":
        assert np.array_equal(got, ref), f"{what}: int32 result not bit-exact"
        return
    scale = np.abs(ref).max() if ref.size else 0.0
    if ab == "s8":
        # Exact int32 sums; only the fp32 epilogue and the final rounding differ.
        tol = ulp(ref, c) + 2.0 ** -20 * scale
    else:
        tol = REL_TOL[ab] * scale + ulp(ref, c)
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        i = np.argmax(err - tol)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {np.unravel_index(i, err.shape)}"
                             f" got {got.flat[i]!r} ref {ref.flat[i]!r} tol {np.broadcast_to(tol, err.shape).flat[i]!r}")


def decode_out(Y: torch.Tensor) -> np.ndarray:
    return Y.detach().to("cpu").to(torch.float64).numpy()
