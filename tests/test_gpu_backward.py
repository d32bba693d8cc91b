"""Backward pass parity: the tcgen05 backward kernels against the fp64
oracle's gradients.

Gate (per element, derived from the arithmetic): every gradient element is
a sum of terms that each pass through one 16-bit rounding on the way into
the tensor cores (P for dV, dS for dQ and dK; relative error <= 2^-9 for
bf16), accumulated in fp32.  So |g_gpu - g_ref| <= 2^-7 * sum|terms| (a 4x
margin), plus 1e-4 * (1 + max|g_ref|) for the fp32 accumulation and the
exp2 approximation, plus half a unit in the last place of a 16-bit output.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_106_b300 import attn, workloads as W
from tests.parity import half_ulp

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

CASES = [
    # B, Hq, Hkv, n_q, n_kv, d, causal, in, out
    (1, 2, 1, 128, 128, 64, False, "bf16", "f32"),
    (1, 2, 2, 300, 300, 128, True, "bf16", "f32"),
    (2, 4, 2, 200, 333, 128, False, "f16", "f32"),
    (1, 4, 1, 150, 700, 64, True, "bf16", "bf16"),   # n_q < n_kv, bottom-right, G = 4
    (1, 8, 2, 257, 257, 128, True, "bf16", "bf16"),
    (1, 2, 1, 1, 1, 64, False, "f16", "f16"),
]


def _gate(g, ref, mag, dtype, extra=0.0):
    got = g.detach().float().cpu().double().numpy()
    bound = 2.0 ** -7 * mag + 1e-4 * (1 + np.abs(ref).max()) + half_ulp(ref, dtype) + extra
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{int(bad.sum())} of {err.size} outside the gate, max err "
                           f"{err.max():.3e}, max err/mag {np.max(err / (mag + 1e-30)):.3e}")


def _round(x, dtype):
    return torch.from_numpy(x).to(dtype)


def _d_err(dO, O_err):
    """Bound on |D_i(kernel) - D_i(exact)| when the kernel's O differs from
    the exact O by at most O_err elementwise: sum_c |dO_ic| O_err_ic, plus
    the fp32 summation of d products."""
    g = np.abs(dO.double().numpy())
    return (g * O_err).sum(-1) + 1e-6 * g.sum(-1)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_backward_matches_oracle(case):
    """O and lse from the oracle: O in fp32 (D exact to fp32), then the same
    call with O rounded to the input format, gated with the oracle's bound
    on how far that rounding moves dQ and dK."""
    B, Hq, Hkv, nq, nkv, d, causal, ind, outd = case
    spec = W.PrefillSpec(B, Hq, Hkv, nq, nkv, d, causal, ind, outd)
    t = W.make_backward(spec, seed=11)
    O_ref, lse_ref = oracle.sdpa(t["Q"], t["K"], t["V"], causal)
    lse = torch.from_numpy(lse_ref).float().cuda()
    args = (t["Q"].cuda(), t["K"].cuda(), t["V"].cuda())
    O16 = _round(O_ref, DT[ind])
    d_err = _d_err(t["dO"], np.abs(O16.double().numpy() - O_ref))
    gq, gk, gv, (mq, mk, mv, sq, sk) = oracle.backward(t["Q"], t["K"], t["V"], t["dO"], causal,
                                                      magnitudes=True, d_err=d_err)
    dQ, dK, dV = attn.backward(*args, _round(O_ref, torch.float32).cuda(), t["dO"].cuda(), lse,
                               causal, out_dtype=DT[outd])
    assert attn.last_launch_count() == 3
    assert attn.last_error() == attn.OK
    _gate(dV, gv, mv, DT[outd])
    _gate(dK, gk, mk, DT[outd])
    _gate(dQ, gq, mq, DT[outd])
    dQ, dK, dV = attn.backward(*args, O16.cuda(), t["dO"].cuda(), lse, causal,
                               out_dtype=DT[outd])
    assert attn.last_error() == attn.OK
    _gate(dV, gv, mv, DT[outd])
    _gate(dK, gk, mk, DT[outd], extra=sk)
    _gate(dQ, gq, mq, DT[outd], extra=sq)


def test_backward_after_gpu_forward():
    """End to end through the library: forward, then backward from the
    forward's own O and lse."""
    spec = W.PrefillSpec(1, 4, 2, 384, 384, 128, True, "bf16", "f32")
    t = W.make_backward(spec, seed=12)
    Q, K, V, dO = (t[k].cuda() for k in ("Q", "K", "V", "dO"))
    O, lse = attn.prefill(Q, K, V, True, out_dtype=torch.bfloat16)
    dQ, dK, dV = attn.backward(Q, K, V, O, dO, lse, True, out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    # the forward's O is within its own parity bound of the exact O
    O_ref, _ = oracle.sdpa(t["Q"], t["K"], t["V"], True)
    d_err = _d_err(t["dO"], 2e-3 + half_ulp(O_ref, torch.bfloat16))
    gq, gk, gv, (mq, mk, mv, sq, sk) = oracle.backward(t["Q"], t["K"], t["V"], t["dO"], True,
                                                      magnitudes=True, d_err=d_err)
    _gate(dV, gv, mv, torch.float32)
    _gate(dK, gk, mk, torch.float32, extra=sk)
    _gate(dQ, gq, mq, torch.float32, extra=sq)


def test_backward_full_size_gqa_4k_sampled():
    """The gqa-4k shape (B4 Hq32 Hkv8 n4096 d128 causal): the gradients of
    one KV head's group, checked on the oracle restricted to that group."""
    spec = W.PREFILL_WORKLOADS["gqa-4k"]
    t = W.make_backward(spec, seed=0, device="cuda")
    O, lse = attn.prefill(t["Q"], t["K"], t["V"], True, out_dtype=torch.float32)
    dQ, dK, dV = attn.backward(t["Q"], t["K"], t["V"], O, t["dO"], lse, True,
                               out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    for b, hk in ((0, 0), (3, 7)):
        G = spec.Hq // spec.Hkv
        hs = slice(hk * G, (hk + 1) * G)
        # rows 0..n of every head of the group against keys 0..n: a causal
        # prefix of length n is the whole problem truncated to n (keys > n
        # are invisible to rows < n), so check the first 384 rows and keys
        n = 384
        Qh = t["Q"][b:b + 1, hs, :n].cpu()
        Kh = t["K"][b:b + 1, hk:hk + 1, :n].cpu()
        Vh = t["V"][b:b + 1, hk:hk + 1, :n].cpu()
        dOh = t["dO"][b:b + 1, hs, :n].cpu()
        O_ref, _ = oracle.sdpa(Qh, Kh, Vh, True)
        d_err = _d_err(dOh, np.full_like(O_ref, 2e-3))  # fp32 forward O within 2e-3
        gq, _, _, (mq, _, _, sq, _) = oracle.backward(Qh, Kh, Vh, dOh, True, magnitudes=True,
                                                      d_err=d_err)
        _gate(dQ[b:b + 1, hs, :n], gq, mq, torch.float32, extra=sq)
    assert torch.isfinite(dQ).all() and torch.isfinite(dK).all() and torch.isfinite(dV).all()
