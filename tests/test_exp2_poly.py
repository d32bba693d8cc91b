"""The polynomial 2^x the prefill's softmax evaluates on the FMA pipe for
part of each row's exponentials (common.cuh, ex2_poly2): the constants
committed in the kernel source are the minimax fit exp2_poly.py derives,
their fp32 evaluation stays within 3e-6 relative of 2^x, and the special
values come out exact.  On the GPU the device function is compared with the
exact values and with the SFU's ex2.approx."""
import os
import re

import numpy as np
import pytest

from exact_io_aware_106_b300 import exp2_poly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "exact_io_aware_106_b300", "csrc", "common.cuh")
BOUND = 3e-6


def committed_coefficients():
    text = open(SRC).read()
    body = text[text.index("ex2_poly2"):]
    vals = {k: float.fromhex(v.rstrip("f")) for k, v in
            re.findall(r"(kA[1-4]) = (0x[0-9a-fA-F.]+p-?\d+f)", body)}
    return [vals[f"kA{k}"] for k in range(1, 5)]


def test_committed_constants_are_the_minimax_fit():
    a, err = exp2_poly.fit()
    assert err < 3e-6
    got = committed_coefficients()
    assert np.allclose(got, [float(np.float32(v)) for v in a], rtol=0, atol=0)


def test_fp32_evaluation_error_bound_and_special_values():
    a = committed_coefficients()
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-126, 8, 400000), np.linspace(-0.5, 0.5, 10001),
                        np.arange(-126, 9, 0.5)]).astype(np.float32)
    y = exp2_poly.eval_fp32(a, x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1)
    assert rel.max() < BOUND, rel.max()
    # integers come out exact (f = 0, p = 1), -127 and below (and -inf) as +0
    ints = np.arange(-126, 9).astype(np.float32)
    assert np.array_equal(exp2_poly.eval_fp32(a, ints), np.exp2(ints))
    low = np.array([-127.0, -200.0, -1e30, -np.inf], np.float32)
    z = exp2_poly.eval_fp32(a, low)
    assert (z == 0).all() and not np.signbit(z).any()
    # between -127 and -126 the result is tiny and non-negative
    mid = np.linspace(-127, -126, 101).astype(np.float32)
    zm = exp2_poly.eval_fp32(a, mid)
    assert (zm >= 0).all() and (zm < 2.0 ** -125).all()


@pytest.mark.gpu
def test_device_polynomial_against_exact_and_sfu():
    import torch
    from exact_io_aware_106_b300 import attn
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-126, 8, 1 << 20), np.arange(-126, 9),
                        [-127.0, -300.0, -np.inf, 0.0, -0.0, 8.0]]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    yp, ys = torch.empty_like(xd), torch.empty_like(xd)
    st = attn.lib().attn_debug_exp2(attn._ptr(xd), attn._ptr(yp), attn._ptr(ys), x.size,
                                    attn._stream(None))
    assert st == attn.OK
    assert attn.last_error() == attn.OK
    yp, ys = yp.cpu().double().numpy(), ys.cpu().double().numpy()
    # the device evaluation is the simulated fp32 evaluation (at most one
    # unit in the last place apart, for an fma the simulation rounds twice)
    sim = exp2_poly.eval_fp32(committed_coefficients(), x)
    du = np.abs(yp.astype(np.float32).view(np.int32).astype(np.int64) -
                sim.view(np.int32).astype(np.int64))
    assert du.max() <= 1 and (du == 0).mean() > 0.9999
    ok = x >= -126
    exact = np.exp2(x[ok].astype(np.float64))
    assert (np.abs(yp[ok] / exact - 1) < BOUND).all()
    # and it agrees with the SFU's ex2.approx within both error bounds
    assert (np.abs(yp[ok] / ys[ok] - 1) < BOUND + 2 ** -21).all()
    assert (yp[~ok] == 0).all()
