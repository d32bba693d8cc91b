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


# ------------------------------------------------- block-wise quantisation
# marketmaker.cc "Flash Attention and sequence length", FA3 item 3: the
# rotation comes before a block-wise quantisation.  Blocks of 128 rows of a
# head (the block size is this build's reading).

def test_quantize_per_block_is_round_to_nearest_of_the_block_scaled_values():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((2, 3, 300, 64)) * rng.uniform(0.5, 4, (2, 3, 300, 1))
    codes, scales = R.quantize_per_block(x, 128)
    assert scales.shape == (6, 3)  # ceil(300 / 128) blocks, the last one ragged
    dq = R.dequantize_per_block(codes, scales, 128)
    xf, df = x.reshape(6, 300, 64), dq.reshape(6, 300, 64)
    for blk in range(3):
        rows = slice(128 * blk, 128 * (blk + 1))
        sc = scales[:, blk].astype(np.float64)
        v = np.abs(xf[:, rows] / sc[:, None, None])
        ex = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
        half_step = 0.5 * np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (ex - 3))
        assert (np.abs(xf[:, rows] - df[:, rows]) <=
                half_step * sc[:, None, None] * (1 + 1e-6)).all()
        # the block's largest entry maps to the largest finite code, +-448
        for h in range(6):
            assert np.max(np.abs(df[h, rows])) == pytest.approx(448 * sc[h], rel=1e-6)


def test_quantize_per_block_codes_match_torch_cast():
    """An independent encoder: torch's float8_e4m3fn cast of the fp32
    quotient x / scale[block] gives the same codes."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((1, 2, 260, 128)) * 3
    codes, scales = R.quantize_per_block(x, 128)
    xf = x.reshape(2, 260, 128).astype(np.float32)
    sc = scales[:, np.arange(260) // 128][:, :, None]
    q = torch.from_numpy((xf / sc).astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(codes.reshape(2, 260, 128), q.view(torch.uint8).numpy())


def test_block_scales_relate_to_the_head_scale():
    """Each block's scale is at most the head's; the largest equals it; one
    block covering the whole head is per-head quantisation, bit for bit."""
    rng = np.random.default_rng(13)
    x = rng.standard_normal((2, 2, 500, 64))
    cb, sb = R.quantize_per_block(x, 128)
    ch, sh = R.quantize_per_head(x)
    assert (sb <= sh[:, None]).all()
    assert np.array_equal(sb.max(axis=1), sh)
    c1, s1 = R.quantize_per_block(x, 500)
    assert np.array_equal(c1, ch) and np.array_equal(s1[:, 0], sh)


def test_an_outlier_coarsens_only_its_own_block():
    """The property block-wise quantisation exists for: an outlier planted in
    block 1 raises that block's scale and changes that block's codes only;
    per head, it changes the codes of every block."""
    rng = np.random.default_rng(14)
    x = rng.standard_normal((1, 1, 384, 64))
    y = x.copy()
    y[0, 0, 200, 5] = 80.0
    cx, sx = R.quantize_per_block(x, 128)
    cy, sy = R.quantize_per_block(y, 128)
    assert sy[0, 1] > 10 * sx[0, 1]
    assert sy[0, 0] == sx[0, 0] and sy[0, 2] == sx[0, 2]
    assert np.array_equal(cy[..., :128, :], cx[..., :128, :])
    assert np.array_equal(cy[..., 256:, :], cx[..., 256:, :])
    hx, _ = R.quantize_per_head(x)
    hy, _ = R.quantize_per_head(y)
    assert not np.array_equal(hy[..., :128, :], hx[..., :128, :])
    # and the error of the untouched blocks stays that of clean data
    err_b = np.abs(R.dequantize_per_block(cy, sy, 128) - y)[..., :128, :].max()
    hy_c, hy_s = R.quantize_per_head(y)
    err_h = np.abs(R.dequantize(hy_c, hy_s) - y)[..., :128, :].max()
    assert err_b < err_h


def test_rotation_lowers_the_block_peak_on_outlier_data():
    """The mechanism under block-wise scales: after the rotation every
    128-row block's peak-to-RMS ratio falls by more than half."""
    rng = np.random.default_rng(15)
    x = outlier_tensor(rng, (1, 2, 512, 128))
    xr = R.rotate(x, rng.choice([-1.0, 1.0], 128))

    def par(a):
        b = a.reshape(2, 4, 128 * 128)
        return np.abs(b).max(axis=2) / np.sqrt((b ** 2).mean(axis=2))
    assert (par(xr) < 0.5 * par(x)).all()


def test_rotation_lowers_fp8_attention_error_under_block_scales():
    """Exact attention with Q, K quantised block-wise (128 rows) to E4M3,
    directly (naive) or after the rotation, V per head in both arms, on the
    outlier recipe: the rotated error is lower.  The page's 2.6x is its own
    H100 measurement on its own data and is not pinned."""
    rng = np.random.default_rng(2)
    B, H, n, d = 1, 4, 256 * 2, 128
    Q, K = outlier_tensor(rng, (B, H, n, d)), outlier_tensor(rng, (B, H, n, d))
    V = rng.standard_normal((B, H, n, d))
    O, _ = oracle.sdpa(Q, K, V, True)
    vq, vs = R.quantize_per_head(V)
    Vd = R.dequantize(vq, vs)
    deq = lambda a: R.dequantize_per_block(*R.quantize_per_block(a, 128), 128)  # noqa: E731
    On, _ = oracle.sdpa(deq(Q), deq(K), Vd, True)
    s = rng.choice([-1.0, 1.0], d)
    Or, _ = oracle.sdpa(deq(R.rotate(Q, s)), deq(R.rotate(K, s)), Vd, True,
                        scale=1.0 / (d * np.sqrt(d)))
    err_naive = np.sqrt(np.mean((On - O) ** 2))
    err_rot = np.sqrt(np.mean((Or - O) ** 2))
    assert err_rot < err_naive / 1.1, (err_naive, err_rot)
