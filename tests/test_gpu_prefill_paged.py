"""Prefill over a block-paged cache (prefix caching / chunked prefill):
the tcgen05 kernels with K/V gathered block by block through the block
table, against the fp64 oracle's paged prefill."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_106_b300 import attn, workloads as W
from tests.parity import assert_lse, assert_out

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

CASES = [
    # B, Hq, Hkv, n_q, d, lens, block, causal, in, out
    (3, 4, 2, 77, 128, [77, 300, 1000], 16, True, "bf16", "f32"),
    (2, 8, 8, 300, 64, [300, 333], 32, True, "f16", "f16"),
    (2, 4, 1, 1, 128, [1, 500], 16, True, "bf16", "bf16"),       # one new token (decode shape)
    (2, 2, 2, 129, 256, [129, 700], 64, True, "bf16", "f32"),
    (2, 4, 2, 64, 128, [100, 2000], 16, False, "bf16", "f32"),   # non-causal
    (1, 16, 1, 256, 64, [4100], 16, True, "f16", "f32"),         # G = 16
    (2, 4, 2, 200, 256, [205, 1333], 16, True, "f16", "bf16"),
    # the CTAs take the sequences longest first: equal lengths, and more
    # sequences than one warp ranks in one pass
    (37, 2, 1, 16, 64, [16 + 9 * ((3 * i) % 20) for i in range(37)], 16, True, "bf16", "f32"),
    (33, 2, 2, 40, 256, [40 + 11 * ((7 * i) % 12) for i in range(33)], 32, True, "bf16", "f32"),
    # more sequences than are ranked: the given order
    (70, 2, 2, 8, 128, [8 + 7 * ((5 * i) % 33) for i in range(70)], 16, True, "f16", "f32"),
    # one TMA box per cache block: 32- and 64-token boxes, sequence ends inside them
    (3, 4, 2, 100, 128, [100, 777, 1301], 64, True, "bf16", "f32"),
    (2, 8, 2, 64, 128, [64, 999], 32, True, "f16", "bf16"),
    (2, 4, 4, 130, 64, [130, 2049], 64, True, "bf16", "f32"),
    # d = 256: V by one box per cache block into a unit-major stage, K by two
    # warps; 20 key blocks, sequence ends inside a block
    (2, 4, 2, 300, 256, [1203, 2501], 16, True, "bf16", "bf16"),
    (2, 4, 2, 300, 256, [1203, 2501], 64, False, "f16", "f32"),
    # d = 256 with 16-token blocks (4-D V boxes): non-causal; no cached prefix
    # (n_q = length) with the end inside the first key block; equal lengths
    (3, 2, 1, 97, 256, [97, 300, 2048], 16, False, "bf16", "f32"),
    (2, 2, 2, 77, 256, [77, 77], 16, True, "f16", "f32"),
    (4, 4, 4, 64, 256, [640, 640, 641, 639], 16, True, "bf16", "bf16"),
]


def _dev(t):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


def _run(case, seed=0, poison=False):
    B, Hq, Hkv, nq, d, lens, bs, causal, ind, outd = case
    spec = W.PagedPrefillSpec(B, Hq, Hkv, nq, d, 1, max(lens), bs, causal, ind, outd)
    t = W.make_paged_prefill(spec, seed=seed, lens=lens)
    if poison:
        # slots past every sequence end hold NaN: they must not reach O
        for b, L in enumerate(lens):
            if L % bs:
                blk = int(t["block_table"][b, (L - 1) // bs])
                t["Kc"][blk, :, L % bs:] = float("nan")
                t["Vc"][blk, :, L % bs:] = float("nan")
    g = _dev(t)
    O, lse = attn.prefill_paged(g["Q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                                max_seq_len=max(lens), causal=causal, out_dtype=DT[outd])
    assert attn.last_launch_count() == 1
    return t, O, lse


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-Hq{c[1]}-Hkv{c[2]}-nq{c[3]}-"
                         f"d{c[4]}-bs{c[6]}-{'c' if c[7] else 'nc'}-{c[8]}-{c[9]}")
def test_prefill_paged_small(case):
    t, O, lse = _run(case)
    assert attn.last_error() == attn.OK
    O_ref, lse_ref = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"],
                                          t["seq_lens"], case[7])
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


@pytest.mark.parametrize("d,bs", [(64, 16), (128, 16), (256, 16), (128, 64), (256, 32)])
def test_prefill_paged_stale_slots_do_not_leak(d, bs):
    # at d = 256 the sequence-end V unit is copied by two warps, panel by panel
    case = (3, 4, 2, 77, d, [77, 301, 999], bs, True, "bf16", "f32")
    t, O, lse = _run(case, seed=1, poison=True)
    assert attn.last_error() == attn.OK
    assert torch.isfinite(O).all()
    O_ref, lse_ref = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"],
                                          t["seq_lens"], True)
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


def test_prefill_paged_bad_block_is_reported():
    case = (3, 4, 2, 64, 128, [64, 200, 300], 16, True, "bf16", "f32")
    B, Hq, Hkv, nq, d, lens, bs, causal, ind, outd = case
    spec = W.PagedPrefillSpec(B, Hq, Hkv, nq, d, 1, max(lens), bs, causal, ind, outd)
    t = W.make_paged_prefill(spec, seed=2, lens=lens)
    g = _dev(t)
    g["seq_lens"][1] = nq - 1  # causal: shorter than its new tokens
    O, lse = attn.prefill_paged(g["Q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                                max_seq_len=max(lens), causal=True, out_dtype=torch.float32)
    assert attn.last_error() == attn.ERR_INVALID
    assert (O[1] == 0).all() and torch.isnan(lse[1]).all()
    keep = torch.tensor([True, False, True])
    O_ref, lse_ref = oracle.prefill_paged(t["Q"][keep], t["Kc"], t["Vc"],
                                          t["block_table"][keep], t["seq_lens"][keep], True)
    assert_out(O[keep], O_ref)
    assert attn.last_error() == attn.OK


def test_prefill_paged_full_size_sampled_rows():
    spec = W.PAGED_PREFILL_WORKLOADS["paged-prefill"]
    t = W.make_paged_prefill(spec, seed=0, device="cuda")
    O, lse = attn.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                                max_seq_len=spec.len_hi, causal=spec.causal,
                                out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    for lo, hi in ((0, 2), (127, 129), (spec.n_q - 2, spec.n_q)):
        O_ref, lse_ref = oracle.prefill_paged(host["Q"], host["Kc"], host["Vc"],
                                              host["block_table"], host["seq_lens"],
                                              spec.causal, rows=(lo, hi))
        assert_out(O[:, :, lo:hi], O_ref, what=f"rows {lo}:{hi}")
        assert_lse(lse[:, :, lo:hi], lse_ref, what=f"rows {lo}:{hi}")
    assert torch.isfinite(O).all()
