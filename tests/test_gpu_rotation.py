"""Incoherent processing on the GPU: the rotate-and-quantise kernels (per
head and block-wise) against the oracle's rotation and E4M3 encoder, the
E4M3 prefill with block-wise scales against the oracle, and fp8 attention
on rotated codes against naive fp8, both against exact attention."""
import numpy as np
import pytest
import torch

import oracle
from oracle import rotation as R
from exact_io_aware_106_b300 import attn
from tests.parity import ATOL_FP8, assert_lse, assert_out

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def _outliers(rng, shape, frac=1e-3, mag=10.0):
    x = rng.standard_normal(shape)
    m = rng.random(shape) < frac
    x[m] = rng.standard_normal(int(m.sum())) * mag
    return x


@pytest.mark.parametrize("d,dt,rpb", [(64, torch.bfloat16, 0), (128, torch.float16, 0),
                                      (256, torch.bfloat16, 0), (64, torch.float16, 128),
                                      (128, torch.bfloat16, 128), (256, torch.float16, 64)])
def test_rotate_quantize_matches_oracle(d, dt, rpb):
    """Rotated rows, quantised per head (rpb 0) or per block of rpb rows:
    scales equal the oracle's block amax / 448, every code is the oracle's
    round-to-nearest code or its neighbour where the exact value lies within
    the fp32 transform error of a rounding boundary."""
    rng = np.random.default_rng(d + rpb)
    x = torch.from_numpy(_outliers(rng, (2, 3, 300, d))).to(dt)
    signs = rng.choice([-1, 1], d).astype(np.int8)
    codes, scales = attn.rotate_quantize_e4m3(x.cuda(), torch.from_numpy(signs).cuda(),
                                              rows_per_block=rpb)
    assert attn.last_launch_count() == 2
    assert attn.last_error() == attn.OK
    xr = R.rotate(x.double().numpy(), signs)
    blk = rpb if rpb else 300
    _, sc_ref = R.quantize_per_block(xr, blk)
    assert np.allclose(scales.cpu().numpy().reshape(sc_ref.shape), sc_ref, rtol=1e-6)
    row_sc = sc_ref[:, np.arange(300) // blk].astype(np.float64)       # [6, 300]
    v = (xr.reshape(6, 300, d) / row_sc[:, :, None]).ravel()
    lo = oracle.encode_e4m3(v * (1 - 1e-5))
    hi = oracle.encode_e4m3(v * (1 + 1e-5))
    got = codes.cpu().view(torch.uint8).numpy().ravel()
    assert ((got == lo) | (got == hi)).all()


@pytest.mark.parametrize("d,rpb", [(64, 128), (128, 128), (256, 0), (128, 7)])
def test_quantize_without_rotation_is_bit_exact(d, rpb):
    """signs = NULL (naive fp8): no transform, so the GPU's fp32 quotient is
    the oracle's and every code and scale matches bit for bit."""
    rng = np.random.default_rng(100 + d)
    x = torch.from_numpy(_outliers(rng, (3, 257, d))).to(torch.bfloat16)
    codes, scales = attn.rotate_quantize_e4m3(x.cuda(), None, rows_per_block=rpb)
    assert attn.last_error() == attn.OK
    c_ref, s_ref = R.quantize_per_block(x.double().numpy(), rpb if rpb else 257, head_axes=1)
    assert np.array_equal(scales.cpu().numpy().reshape(s_ref.shape), s_ref)
    assert np.array_equal(codes.cpu().view(torch.uint8).numpy(), c_ref)


E4M3_BLOCK_CASES = [
    # B, Hq, Hkv, n_q, n_kv, d, causal, out
    (1, 2, 1, 300, 300, 128, True, "f32"),      # ragged last block
    (2, 4, 2, 129, 1000, 128, False, "bf16"),   # n_q past one block, 8 key blocks
    (1, 4, 1, 200, 700, 64, True, "f32"),       # n_q < n_kv, bottom-right mask
    (1, 2, 2, 333, 333, 64, False, "bf16"),
    (1, 2, 1, 257, 257, 256, True, "f32"),      # 64-key blocks: two per scale block
    (1, 4, 2, 100, 600, 256, False, "bf16"),
    (1, 1, 1, 1, 1, 128, False, "f32"),
]


def _block_inputs(case, seed, outliers=False):
    B, Hq, Hkv, nq, nkv, d, causal, outd = case
    rng = np.random.default_rng(seed)
    gen = (lambda s: _outliers(rng, s)) if outliers else rng.standard_normal
    Q = torch.from_numpy(gen((B, Hq, nq, d))).to(torch.bfloat16).double().numpy()
    K = torch.from_numpy(gen((B, Hkv, nkv, d))).to(torch.bfloat16).double().numpy()
    V = torch.from_numpy(rng.standard_normal((B, Hkv, nkv, d))).to(torch.bfloat16)
    qc, qs = R.quantize_per_block(Q, 128)
    kc, ks = R.quantize_per_block(K, 128)
    vc, vs = R.quantize_per_head(V.double().numpy())
    dev = {n: torch.from_numpy(a).cuda() for n, a in (("qs", qs), ("ks", ks), ("vs", vs))}
    f8 = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).cuda()  # noqa: E731
    return (Q, K, V.double().numpy()), (f8(qc), f8(kc), f8(vc), dev), \
        (R.dequantize_per_block(qc, qs, 128), R.dequantize_per_block(kc, ks, 128),
         R.dequantize(vc, vs))


@pytest.mark.parametrize("case", E4M3_BLOCK_CASES, ids=lambda c: "x".join(map(str, c)))
def test_prefill_e4m3_blocks_matches_oracle_on_dequantised_inputs(case):
    """Block-wise scales: every element against the oracle fed the block-wise
    dequantised inputs, under the 16-bit rule."""
    src, (Qc, Kc, Vc, sc), deq = _block_inputs(case, seed=case[3] + case[5])
    O, lse = attn.prefill_e4m3_blocks(Qc, Kc, Vc, case[6], sc["qs"], sc["ks"], sc["vs"],
                                      out_dtype=DT[case[7]])
    assert attn.last_launch_count() == 1
    assert attn.last_error() == attn.OK
    O_ref, lse_ref = oracle.sdpa(*deq, case[6])
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


@pytest.mark.parametrize("case", [E4M3_BLOCK_CASES[1], E4M3_BLOCK_CASES[5]],
                         ids=lambda c: "x".join(map(str, c)))
def test_prefill_e4m3_blocks_quantisation_budget(case):
    """Rows that average >= 512 keys against the oracle fed the unquantised
    inputs: 3e-2 max-abs."""
    src, (Qc, Kc, Vc, sc), _ = _block_inputs(case, seed=7)
    O, _ = attn.prefill_e4m3_blocks(Qc, Kc, Vc, case[6], sc["qs"], sc["ks"], sc["vs"],
                                    out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    O_src, _ = oracle.sdpa(*src, case[6])
    assert case[4] >= 512 and not case[6]
    assert_out(O, O_src, atol=ATOL_FP8)


def test_prefill_e4m3_blocks_with_equal_scales_equals_per_head_prefill():
    """One scale repeated over every block is the per-head form: outputs are
    bit-identical to attn_prefill with E4M3 inputs."""
    case = (1, 4, 2, 300, 300, 128, True, "f32")
    src, (Qc, Kc, Vc, sc), _ = _block_inputs(case, seed=3)
    qh = torch.full((4,), 0.011, device="cuda")
    kh = torch.full((2,), 0.009, device="cuda")
    O1, l1 = attn.prefill(Qc, Kc, Vc, True, out_dtype=torch.float32, q_scale=qh, k_scale=kh,
                          v_scale=sc["vs"])
    O2, l2 = attn.prefill_e4m3_blocks(Qc, Kc, Vc, True, qh.repeat_interleave(3),
                                      kh.repeat_interleave(3), sc["vs"], out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    assert torch.equal(O1, O2) and torch.equal(l1, l2)


def test_fp8_prefill_on_rotated_codes_beats_naive_on_outliers():
    """The page's comparison on the outlier recipe, every step on the GPU:
    naive fp8 (Q, K quantised block-wise as they are) against incoherent
    processing (rotated, then quantised block-wise), V per head in both arms,
    each against exact attention of the 16-bit inputs.  The per-head arms
    are reported beside them."""
    rng = np.random.default_rng(5)
    B, H, n, d = 1, 4, 512, 128
    Q = _outliers(rng, (B, H, n, d))
    K = _outliers(rng, (B, H, n, d))
    V = rng.standard_normal((B, H, n, d))
    Qb, Kb, Vb = (torch.from_numpy(a).to(torch.bfloat16) for a in (Q, K, V))
    O, _ = oracle.sdpa(Qb, Kb, Vb, True)  # exact attention of the bf16 inputs
    flat = lambda t: t.reshape(B * H, n, d).contiguous().cuda()  # noqa: E731
    vq, vs = R.quantize_per_head(Vb.double().numpy())
    Vc = torch.from_numpy(vq).view(torch.float8_e4m3fn).cuda()
    vsc = torch.from_numpy(vs).cuda()
    signs = torch.from_numpy(rng.choice([-1, 1], d).astype(np.int8)).cuda()
    errs = {}
    for arm, sg, sc in (("naive", None, 1.0 / np.sqrt(d)),
                        ("rotated", signs, 1.0 / (d * np.sqrt(d)))):
        for rpb in (0, 128):
            qc, qs = attn.rotate_quantize_e4m3(flat(Qb), sg, rows_per_block=rpb)
            kc, ks = attn.rotate_quantize_e4m3(flat(Kb), sg, rows_per_block=rpb)
            qc, kc = qc.view(B, H, n, d), kc.view(B, H, n, d)
            if rpb:
                Og, _ = attn.prefill_e4m3_blocks(qc, kc, Vc, True, qs, ks, vsc, scale=sc,
                                                 out_dtype=torch.float32)
            else:
                Og, _ = attn.prefill(qc, kc, Vc, True, scale=sc, out_dtype=torch.float32,
                                     q_scale=qs, k_scale=ks, v_scale=vsc)
            assert attn.last_error() == attn.OK
            errs[(arm, rpb)] = np.sqrt(np.mean((Og.cpu().double().numpy() - O) ** 2))
    print("fp8 attention RMSE vs exact: " + ", ".join(
        f"{a} {'block-128' if r else 'per-head'} {e:.4e}" for (a, r), e in errs.items()) +
        f"; block-wise gain {errs[('naive', 128)] / errs[('rotated', 128)]:.2f}, "
        f"per-head gain {errs[('naive', 0)] / errs[('rotated', 0)]:.2f}")
    assert errs[("rotated", 128)] < errs[("naive", 128)] / 1.1
    assert errs[("rotated", 0)] < errs[("naive", 0)] / 1.1
