"""Pins of the incoherent-processing oracle (random-sign Hadamard rotation
before per-head E4M3 quantisation)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import rotation as R


@pytest.mark.parametrize("d", [64, 128, 256])
def test_hadamard_is_orthogonal_and_closed_form(d):
    H = R.hadamard(d)
    assert np.array_equal(H @ H.T, d * np.eye(d, dtype=np.int64))
    i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
    pop = np.vectorize(lambda v: bin(v).count("1"))(i & j)
    assert np.array_equal(H, np.where(pop % 2 == 0, 1, -1))


def test_rotation_preserves_scores_up_to_d():
    rng = np.random.default_rng(0)
    d = 128
    q, k = rng.standard_normal((5, d)), rng.standard_normal((7, d))
    s = rng.choice([-1.0, 1.0], d)
    lhs = R.rotate(q, s) @ R.rotate(k, s).T
    assert np.allclose(lhs, d * (q @ k.T), rtol=1e-12, atol=1e-10)


def test_encode_array_matches_scalar_encoder_and_torch():
    x = np.concatenate([np.linspace(-500, 500, 2001), np.array([0.0, -0.0, 1e-9, 448.0])])
    codes = oracle.encode_e4m3(x)
    assert all(codes[i] == oracle.e4m3_encode(float(np.float32(v))) for i, v in enumerate(x))
    inr = np.abs(x) <= 448
    t = torch.from_numpy(x[inr].astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(codes[inr], t.view(torch.uint8).numpy())


def test_quantize_per_head_is_round_to_nearest_of_the_scaled_values():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 3, 40, 64)) * 3
    codes, scales = R.quantize_per_head(x)
    assert np.allclose(scales, np.abs(x.reshape(6, -1)).max(1) / 448, rtol=1e-6)
    dq = R.dequantize(codes, scales)
    # |x - deq| <= half a code step of x / scale, times the scale
    v = np.abs(x.reshape(6, -1) / scales[:, None])
    ex = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    half_step = 0.5 * np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (ex - 3))
    assert (np.abs(x.reshape(6, -1) - dq.reshape(6, -1)) <=
            half_step * scales[:, None] * (1 + 1e-6)).all()
    # the largest entry of each head maps to +-448
    for h in range(6):
        assert np.max(np.abs(dq.reshape(6, -1)[h])) == pytest.approx(448 * scales[h], rel=1e-6)


def outlier_tensor(rng, shape, frac=1e-3, mag=10.0):
    """N(0, 1) entries with a fraction `frac` replaced by N(0, mag^2)."""
    x = rng.standard_normal(shape)
    m = rng.random(shape) < frac
    x[m] = rng.standard_normal(int(m.sum())) * mag
    return x


def test_rotation_spreads_outliers():
    """The mechanism: after the rotation no component carries an outlier --
    the peak-to-RMS ratio of each head drops to that of Gaussian data."""
    rng = np.random.default_rng(3)
    x = outlier_tensor(rng, (1, 4, 256, 128))
    xr = R.rotate(x, rng.choice([-1.0, 1.0], 128))
    par = lambda a: np.abs(a).max(axis=(2, 3)) / np.sqrt((a ** 2).mean(axis=(2, 3)))  # noqa
    assert (par(xr) < 0.5 * par(x)).all()


def test_rotation_lowers_fp8_attention_error_on_outlier_data():
    """Exact attention with Q, K quantised per head to E4M3 (V too, the same
    in both arms), directly or after the rotation, on N(0,1) data with 0.1 %
    of entries drawn from N(0, 10^2): the rotated error is lower."""
    rng = np.random.default_rng(2)
    B, H, n, d = 1, 4, 256, 128
    Q, K = outlier_tensor(rng, (B, H, n, d)), outlier_tensor(rng, (B, H, n, d))
    V = rng.standard_normal((B, H, n, d))
    O, _ = oracle.sdpa(Q, K, V, True)
    vq, vs = R.quantize_per_head(V)
    Vd = R.dequantize(vq, vs)
    qn, sq = R.quantize_per_head(Q)
    kn, sk = R.quantize_per_head(K)
    On, _ = oracle.sdpa(R.dequantize(qn, sq), R.dequantize(kn, sk), Vd, True)
    s = rng.choice([-1.0, 1.0], d)
    qr, sqr = R.quantize_per_head(R.rotate(Q, s))
    kr, skr = R.quantize_per_head(R.rotate(K, s))
    Or, _ = oracle.sdpa(R.dequantize(qr, sqr), R.dequantize(kr, skr), Vd, True,
                        scale=1.0 / (d * np.sqrt(d)))
    err_naive = np.sqrt(np.mean((On - O) ** 2))
    err_rot = np.sqrt(np.mean((Or - O) ** 2))
    assert err_rot < err_naive / 1.1, (err_naive, err_rot)
