"""Seeded random configurations against the fp64 oracle: dense prefill
(16-bit and E4M3 inputs), paged prefill, decode (16-bit and E4M3 caches),
multi-token decode and the backward, over head sizes, group sizes, lengths,
block sizes, masking and dtypes drawn together, so that combinations the
hand-picked cases do not list are exercised too.  The draws are fixed (one
generator, one seed); sizes are capped so that the oracle finishes each
case in a second or two."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_106_b300 import attn, workloads as W
from tests.parity import assert_lse, assert_out

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
_rng = np.random.RandomState(20261203)
_MAX_WORK = 1.5e9  # multiply-adds of the oracle per case (B Hq n_q n_kv d)


def _pick(xs):
    return xs[_rng.randint(len(xs))]


def _dense_cases(n):
    out = []
    while len(out) < n:
        d = _pick([64, 128, 256])
        G = _pick([1, 2, 3, 4, 8])
        Hkv = _pick([1, 2])
        B = _pick([1, 2])
        causal = bool(_rng.randint(2))
        n_q = int(_rng.randint(1, 600))
        n_kv = n_q + int(_rng.randint(0, 900)) if causal else int(_rng.randint(1, 1200))
        ind = _pick(["bf16", "f16"])
        outd = _pick(["f32", ind])
        if B * Hkv * G * n_q * n_kv * d > _MAX_WORK:
            continue
        out.append((B, Hkv * G, Hkv, n_q, n_kv, d, causal, ind, outd))
    return out


def _paged_cases(n):
    out = []
    while len(out) < n:
        d = _pick([64, 128, 256])
        G = _pick([1, 2, 4, 8])
        Hkv = _pick([1, 2])
        B = int(_rng.randint(1, 6))
        bs = _pick([16, 32, 64])
        causal = bool(_rng.randint(2))
        n_q = int(_rng.randint(1, 300))
        lens = [n_q + int(_rng.randint(0, 1500)) for _ in range(B)]
        ind = _pick(["bf16", "f16"])
        if sum(lens) * Hkv * G * n_q * d > _MAX_WORK:
            continue
        out.append((B, Hkv * G, Hkv, n_q, d, lens, bs, causal, ind))
    return out


def _decode_cases(n):
    out = []
    while len(out) < n:
        d = _pick([64, 128, 256])
        G = _pick([1, 2, 3, 4, 5, 8, 16])
        Hkv = _pick([1, 2, 4])
        S = int(_rng.randint(1, 9))
        T = _pick([1, 1, 2, 3, 4, 8])
        if G * T > 64:
            continue
        bs = _pick([16, 32, 64])
        lens = [max(T, int(_rng.randint(1, 3000))) for _ in range(S)]
        kv = _pick(["bf16", "f16"])
        out.append((S, Hkv * G, Hkv, T, d, lens, bs, kv))
    return out


DENSE = _dense_cases(24)
PAGED = _paged_cases(16)
DECODE = _decode_cases(24)


@pytest.mark.parametrize("i", range(len(DENSE)), ids=[f"r{i}" for i in range(len(DENSE))])
def test_random_prefill(i):
    B, Hq, Hkv, n_q, n_kv, d, causal, ind, outd = DENSE[i]
    spec = W.PrefillSpec(B, Hq, Hkv, n_q, n_kv, d, causal, ind, outd)
    t = W.make_prefill(spec, seed=100 + i)
    O, lse = attn.prefill(t["Q"].cuda(), t["K"].cuda(), t["V"].cuda(), causal,
                          out_dtype=DT[outd])
    assert attn.last_error() == attn.OK
    O_ref, lse_ref = oracle.sdpa(t["Q"], t["K"], t["V"], causal)
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


@pytest.mark.parametrize("i", range(len(PAGED)), ids=[f"r{i}" for i in range(len(PAGED))])
def test_random_prefill_paged(i):
    B, Hq, Hkv, n_q, d, lens, bs, causal, ind = PAGED[i]
    spec = W.PagedPrefillSpec(B, Hq, Hkv, n_q, d, 1, max(lens), bs, causal, ind, "f32")
    t = W.make_paged_prefill(spec, seed=200 + i, lens=lens)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    O, lse = attn.prefill_paged(g["Q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                                max_seq_len=max(lens), causal=causal, out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    O_ref, lse_ref = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"],
                                          t["seq_lens"], causal)
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


@pytest.mark.parametrize("i", range(len(DECODE)), ids=[f"r{i}" for i in range(len(DECODE))])
def test_random_decode(i):
    S, Hq, Hkv, T, d, lens, bs, kv = DECODE[i]
    g_out = DT[kv]
    if T == 1:
        spec = W.DecodeSpec(S, Hq, Hkv, d, 1, max(lens), bs, kv, kv, kv)
        t = W.make_decode(spec, seed=300 + i, lens=lens)
        g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
        O, lse = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                             max_seq_len=max(lens), out_dtype=g_out)
        O_ref, lse_ref = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                             t["seq_lens"])
    else:
        spec = W.PagedPrefillSpec(S, Hq, Hkv, T, d, 1, max(lens), bs, True, kv, kv)
        t = W.make_paged_prefill(spec, seed=300 + i, lens=lens)
        g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
        O, lse = attn.decode_tokens(g["Q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                                    max_seq_len=max(lens), out_dtype=g_out)
        O_ref, lse_ref = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"],
                                              t["seq_lens"], True)
    assert attn.last_error() == attn.OK
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


def _e4m3_prefill_cases(n):
    out = []
    while len(out) < n:
        d = _pick([64, 128, 256])
        G = _pick([1, 2, 4, 8])
        Hkv = _pick([1, 2])
        causal = bool(_rng.randint(2))
        n_q = int(_rng.randint(1, 500))
        n_kv = n_q + int(_rng.randint(0, 700)) if causal else int(_rng.randint(1, 1000))
        if Hkv * G * n_q * n_kv * d > _MAX_WORK:
            continue
        out.append((1, Hkv * G, Hkv, n_q, n_kv, d, causal, _pick(["f32", "bf16", "f16"])))
    return out


def _e4m3_decode_cases(n):
    out = []
    while len(out) < n:
        d = _pick([64, 128, 256])
        G = _pick([1, 2, 4, 8, 16, 32])
        Hkv = _pick([1, 2])
        S = int(_rng.randint(1, 7))
        bs = _pick([16, 32, 64])
        lens = [int(_rng.randint(1, 3000)) for _ in range(S)]
        out.append((S, Hkv * G, Hkv, d, lens, bs))
    return out


E4M3_PREFILL = _e4m3_prefill_cases(12)
E4M3_DECODE = _e4m3_decode_cases(12)


@pytest.mark.parametrize("i", range(len(E4M3_PREFILL)),
                         ids=[f"r{i}" for i in range(len(E4M3_PREFILL))])
def test_random_prefill_e4m3(i):
    # against the oracle fed the dequantised inputs (code * per-head scale),
    # under the 16-bit rules
    B, Hq, Hkv, n_q, n_kv, d, causal, outd = E4M3_PREFILL[i]
    spec = W.PrefillSpec(B, Hq, Hkv, n_q, n_kv, d, causal, "bf16", outd)
    t = W.make_prefill(spec, seed=400 + i)
    qz = W.quantize_prefill_e4m3(t)
    g = {k: v.cuda() for k, v in qz.items()}
    O, lse = attn.prefill(g["Q"], g["K"], g["V"], causal, out_dtype=DT[outd],
                          q_scale=g["q_scale"], k_scale=g["k_scale"], v_scale=g["v_scale"])
    assert attn.last_error() == attn.OK
    deq = {n: oracle.dequantize_e4m3(qz[n], qz[n.lower() + "_scale"], 1) for n in "QKV"}
    O_ref, lse_ref = oracle.sdpa(deq["Q"], deq["K"], deq["V"], causal)
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


@pytest.mark.parametrize("i", range(len(E4M3_DECODE)),
                         ids=[f"r{i}" for i in range(len(E4M3_DECODE))])
def test_random_decode_e4m3(i):
    S, Hq, Hkv, d, lens, bs = E4M3_DECODE[i]
    spec = W.DecodeSpec(S, Hq, Hkv, d, 1, max(lens), bs, "bf16", "e4m3", "bf16")
    t = W.make_decode(spec, seed=500 + i, lens=lens)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    O, lse = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                         max_seq_len=max(lens), k_scale=g["k_scale"], v_scale=g["v_scale"],
                         out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    O_ref, lse_ref = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                         t["seq_lens"], k_scale=t["k_scale"],
                                         v_scale=t["v_scale"])
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


def _backward_cases(n):
    out = []
    while len(out) < n:
        d = _pick([64, 128])
        G = _pick([1, 2, 4])
        Hkv = _pick([1, 2])
        B = _pick([1, 2])
        causal = bool(_rng.randint(2))
        n_q = int(_rng.randint(1, 400))
        n_kv = n_q + int(_rng.randint(0, 300)) if causal else int(_rng.randint(1, 500))
        ind = _pick(["bf16", "f16"])
        outd = _pick(["f32", ind])
        out.append((B, Hkv * G, Hkv, n_q, n_kv, d, causal, ind, outd))
    return out


BACKWARD = _backward_cases(10)


@pytest.mark.parametrize("i", range(len(BACKWARD)), ids=[f"r{i}" for i in range(len(BACKWARD))])
def test_random_backward(i):
    # the backward tests' own check (fp32 and 16-bit O, gated per element by
    # the bound derived from the 16-bit rounding of P and dS)
    from tests import test_gpu_backward as bw
    bw.test_backward_matches_oracle(BACKWARD[i])
