"""Tolerance rules for comparing the CUDA path with the fp64 oracle.

* fp32 outputs: |O_gpu - O_ref| <= 2e-3 (max-abs gate for 16-bit inputs with
  fp32 accumulation).
* 16-bit outputs: the same 2e-3 plus half a unit in the last place of the
  output format at |O_ref| -- the rounding of a correct result to the output
  format alone can exceed 2e-3 when |O| > 0.5 (a causal row 0 returns V[0]).
* lse: |lse_gpu - lse_ref| <= 1e-4 * max(0.1, |lse_ref|): 1e-4 relative,
  with an absolute floor of 1e-5 where |lse| < 0.1.  A purely relative gate
  is ill-posed at lse = 0 (a causal row 0 or a one-token sequence has
  lse = its single scaled score, which can be arbitrarily close to 0), and
  the fp32 evaluation m + ln l carries an absolute error of a few 1e-7 from
  m and l alone; the floor is a deliberate departure from "relative".
* E4M3 KV: 3e-2 max-abs against the oracle fed the unquantised values, and
  the 16-bit rule against the oracle fed the dequantised values.
"""
import numpy as np
import torch

ATOL = 2e-3
ATOL_FP8 = 3e-2
LSE_RTOL = 1e-4
LSE_FLOOR = 0.1  # |lse| below which the gate is absolute (LSE_RTOL * LSE_FLOOR)
_MANT = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}


def half_ulp(ref: np.ndarray, dtype) -> np.ndarray:
    if dtype == torch.float32:
        return np.zeros_like(ref)
    a = np.abs(ref)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    ulp = np.ldexp(1.0, (e - 1) - _MANT[dtype])
    if dtype == torch.float16:
        ulp = np.maximum(ulp, 2.0 ** -24)
    return np.where(a > 0, 0.5 * ulp, 0.0)


def out_errors(O_gpu: torch.Tensor, O_ref: np.ndarray, atol: float = ATOL):
    got = O_gpu.detach().float().cpu().double().numpy()
    bound = atol + half_ulp(O_ref, O_gpu.dtype)
    err = np.abs(got - O_ref)
    return err, bound


def assert_out(O_gpu, O_ref, atol: float = ATOL, what: str = "O"):
    err, bound = out_errors(O_gpu, O_ref, atol)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} elements outside the "
                             f"gate (max err {np.nanmax(err):.3e}); first bad {idx.tolist()}")
    return float(np.max(err)) if err.size else 0.0


def assert_lse(lse_gpu, lse_ref, what: str = "lse"):
    got = lse_gpu.detach().cpu().double().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: finiteness differs"
    d = np.abs(got[fin] - lse_ref[fin])
    tol = LSE_RTOL * np.maximum(LSE_FLOOR, np.abs(lse_ref[fin]))
    bad = ~(d <= tol)
    if bad.any():
        raise AssertionError(f"{what}: {int(bad.sum())} rows outside 1e-4 relative "
                             f"(max {np.max(d):.3e})")
    return float(np.max(d)) if d.size else 0.0
