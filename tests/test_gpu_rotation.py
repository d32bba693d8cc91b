"""Incoherent processing on the GPU: the rotate-and-quantize kernels against
the oracle's rotation and E4M3 encoder, and the fp8 prefill on rotated
codes against exact attention."""
import numpy as np
import pytest
import torch

import oracle
from oracle import rotation as R
from exact_io_aware_106_b300 import attn

pytestmark = pytest.mark.gpu


def _outliers(rng, shape, frac=1e-3, mag=10.0):
    x = rng.standard_normal(shape)
    m = rng.random(shape) < frac
    x[m] = rng.standard_normal(int(m.sum())) * mag
    return x


@pytest.mark.parametrize("d,dt", [(64, torch.bfloat16), (128, torch.float16),
                                  (256, torch.bfloat16)])
def test_rotate_quantize_matches_oracle(d, dt):
    rng = np.random.default_rng(d)
    x = torch.from_numpy(_outliers(rng, (2, 3, 100, d))).to(dt)
    signs = rng.choice([-1, 1], d).astype(np.int8)
    codes, scales = attn.rotate_quantize_e4m3(x.cuda(), torch.from_numpy(signs).cuda())
    assert attn.last_error() == attn.OK
    xr = R.rotate(x.double().numpy(), signs)
    amax = np.abs(xr.reshape(6, -1)).max(1)
    assert np.allclose(scales.cpu().numpy(), amax / 448, rtol=1e-6)
    # every code is round-to-nearest of the exact value, or its neighbour
    # when the value sits within the fp32 transform error of a boundary
    v = (xr.reshape(6, -1) / (amax / 448)[:, None]).ravel()
    lo = oracle.encode_e4m3(v * (1 - 1e-5))
    hi = oracle.encode_e4m3(v * (1 + 1e-5))
    got = codes.cpu().view(torch.uint8).numpy().ravel()
    assert ((got == lo) | (got == hi)).all()


def test_fp8_prefill_on_rotated_codes_beats_naive_on_outliers():
    rng = np.random.default_rng(5)
    B, H, n, d = 1, 4, 512, 128
    Q = _outliers(rng, (B, H, n, d))
    K = _outliers(rng, (B, H, n, d))
    V = rng.standard_normal((B, H, n, d))
    Qb, Kb, Vb = (torch.from_numpy(a).to(torch.bfloat16) for a in (Q, K, V))
    O, _ = oracle.sdpa(Qb, Kb, Vb, True)  # exact attention of the bf16 inputs
    flat = lambda t: t.reshape(B * H, n, d).contiguous()  # noqa: E731
    vq, vs = R.quantize_per_head(Vb.double().numpy())
    Vc = torch.from_numpy(vq).view(torch.float8_e4m3fn).cuda()
    vsc = torch.from_numpy(vs).cuda()
    # naive: Q, K quantised per head as they are
    qn, sqn = R.quantize_per_head(Qb.double().numpy())
    kn, skn = R.quantize_per_head(Kb.double().numpy())
    On, _ = attn.prefill(torch.from_numpy(qn).view(torch.float8_e4m3fn).cuda(),
                         torch.from_numpy(kn).view(torch.float8_e4m3fn).cuda(), Vc, True,
                         out_dtype=torch.float32, q_scale=torch.from_numpy(sqn).cuda(),
                         k_scale=torch.from_numpy(skn).cuda(), v_scale=vsc)
    # rotated on the GPU with shared signs; the scores carry a factor d
    signs = torch.from_numpy(rng.choice([-1, 1], d).astype(np.int8)).cuda()
    qr, sqr = attn.rotate_quantize_e4m3(flat(Qb).cuda(), signs)
    kr, skr = attn.rotate_quantize_e4m3(flat(Kb).cuda(), signs)
    Or, _ = attn.prefill(qr.view(B, H, n, d), kr.view(B, H, n, d), Vc, True,
                         scale=1.0 / (d * np.sqrt(d)), out_dtype=torch.float32,
                         q_scale=sqr, k_scale=skr, v_scale=vsc)
    assert attn.last_error() == attn.OK
    err_n = np.sqrt(np.mean((On.cpu().double().numpy() - O) ** 2))
    err_r = np.sqrt(np.mean((Or.cpu().double().numpy() - O) ** 2))
    print(f"fp8 attention RMSE: naive {err_n:.4e}, rotated {err_r:.4e}, ratio {err_n / err_r:.2f}")
    assert err_r < err_n / 1.1
