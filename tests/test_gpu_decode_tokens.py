"""Multi-token decode (several new tokens per sequence, e.g. speculative
drafts): the split-KV tensor-core decode with G * n_new query rows per KV
head, against the oracle's paged prefill with n_q = n_new."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_106_b300 import attn, workloads as W
from tests.parity import assert_lse, assert_out

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

CASES = [
    # S, Hq, Hkv, T, d, lens, block, dtype
    (4, 8, 2, 4, 128, [4, 17, 300, 2000], 16, "bf16"),
    (3, 4, 4, 16, 64, [16, 100, 999], 32, "f16"),
    (2, 16, 2, 2, 256, [2, 5000], 16, "bf16"),
    (3, 6, 2, 5, 128, [5, 64, 77], 64, "bf16"),       # G = 3, T = 5: 15 rows
    (3, 16, 2, 4, 128, [4, 333, 4000], 16, "bf16"),   # G = 8, T = 4: two 16-row tiles
    (2, 4, 1, 5, 256, [5, 700], 16, "bf16"),          # G = 4, T = 5: 20 rows, ragged tile
    (2, 16, 1, 4, 64, [4, 1000], 32, "f16"),          # G = 16, T = 4: four tiles
]


def _dev(t):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{c[0]}-Hq{c[1]}-Hkv{c[2]}-T{c[3]}-"
                         f"d{c[4]}-bs{c[6]}-{c[7]}")
def test_decode_tokens_matches_paged_oracle(case):
    S, Hq, Hkv, T, d, lens, bs, dt = case
    spec = W.PagedPrefillSpec(S, Hq, Hkv, T, d, 1, max(lens), bs, True, dt, "f32")
    t = W.make_paged_prefill(spec, seed=7, lens=lens)
    g = _dev(t)
    O_ref, lse_ref = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"],
                                          t["seq_lens"], True)
    for out in (torch.float32, DT[dt]):
        O, lse = attn.decode_tokens(g["Q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                                    max_seq_len=max(lens), out_dtype=out)
        assert attn.last_launch_count() == 2
        assert attn.last_error() == attn.OK
        assert_out(O, O_ref)
        assert_lse(lse, lse_ref)


@pytest.mark.parametrize("Hq", [8, 16], ids=["12rows", "24rows"])
def test_decode_tokens_e4m3_cache(Hq):
    S, Hkv, T, d, lens, bs = 3, 2, 3, 128, [3, 200, 1500], 16
    spec = W.PagedPrefillSpec(S, Hq, Hkv, T, d, 1, max(lens), bs, True, "bf16", "f32")
    t = W.make_paged_prefill(spec, seed=8, lens=lens)
    kq, ks = W.quantize_e4m3_per_head(t["Kc"], 1)
    vq, vs = W.quantize_e4m3_per_head(t["Vc"], 1)
    nb = t["Kc"].shape[0]
    Kd = torch.from_numpy(oracle.dequantize_e4m3(kq, ks.repeat(nb), 1))
    Vd = torch.from_numpy(oracle.dequantize_e4m3(vq, vs.repeat(nb), 1))
    O_ref, lse_ref = oracle.prefill_paged(t["Q"].double(), Kd, Vd, t["block_table"],
                                          t["seq_lens"], True)
    O, lse = attn.decode_tokens(t["Q"].cuda(), kq.cuda(), vq.cuda(), t["block_table"].cuda(),
                                t["seq_lens"].cuda(), max_seq_len=max(lens), k_scale=ks.cuda(),
                                v_scale=vs.cuda(), out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


def test_decode_tokens_one_token_equals_decode():
    S, Hq, Hkv, d, lens = 3, 8, 2, 128, [1, 33, 700]
    spec = W.PagedPrefillSpec(S, Hq, Hkv, 1, d, 1, max(lens), 16, True, "bf16", "f32")
    t = _dev(W.make_paged_prefill(spec, seed=9, lens=lens))
    O1, l1 = attn.decode_tokens(t["Q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                                max_seq_len=max(lens), out_dtype=torch.float32)
    O2, l2 = attn.decode(t["Q"][:, :, 0].contiguous(), t["Kc"], t["Vc"], t["block_table"],
                         t["seq_lens"], max_seq_len=max(lens), out_dtype=torch.float32)
    assert torch.equal(O1[:, :, 0], O2) and torch.equal(l1[:, :, 0], l2)


def test_decode_tokens_short_sequence_is_reported():
    S, Hq, Hkv, T, d, lens = 2, 4, 2, 4, 64, [4, 90]
    spec = W.PagedPrefillSpec(S, Hq, Hkv, T, d, 1, max(lens), 16, True, "bf16", "f32")
    t = _dev(W.make_paged_prefill(spec, seed=10, lens=lens))
    t["seq_lens"][0] = T - 1
    O, lse = attn.decode_tokens(t["Q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                                max_seq_len=max(lens), out_dtype=torch.float32)
    assert attn.last_error() == attn.ERR_INVALID
    assert (O[0] == 0).all() and torch.isnan(lse[0]).all()
    assert torch.isfinite(O[1]).all()
