"""Paged split-KV decode parity against the fp64 oracle, plus KV append
bit-exactness and the device-side index checks."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_106_b300 import attn, workloads as W
from tests.parity import ATOL_FP8, assert_lse, assert_out

pytestmark = pytest.mark.gpu


def _dev(t):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


CASES = [
    # num_seqs, Hq, Hkv, d, block, lens, kv
    (5, 8, 2, 128, 16, [1, 15, 16, 17, 300], "bf16"),
    (3, 4, 4, 64, 16, [33, 1000, 2], "bf16"),
    (4, 16, 1, 128, 32, [64, 65, 700, 3], "bf16"),
    (2, 32, 2, 64, 64, [1500, 129], "bf16"),
    (3, 12, 4, 256, 16, [40, 600, 2049], "bf16"),
    (4, 8, 8, 128, 16, [5, 4096, 300, 1], "f16"),
    (2, 16, 8, 256, 16, [70, 9], "f16"),
    (6, 6, 2, 128, 16, [1, 2, 3, 250, 251, 1300], "bf16"),   # G = 3
    (3, 32, 1, 128, 16, [1, 777, 3000], "bf16"),             # MQA, G = 32: two row tiles
    (3, 32, 1, 64, 16, [1, 777, 3000], "bf16"),              # d = 64, G = 32: one CTA, two tiles
    (2, 40, 1, 64, 32, [100, 2500], "f16"),                  # G = 40: three tiles, last ragged
    (2, 64, 1, 256, 16, [17, 1200], "bf16"),                 # G = 64: four tiles
    (2, 32, 1, 128, 16, [900, 33], "f16"),                   # f16, two consumer groups
    (2, 48, 2, 128, 16, [31, 2222], "bf16"),                 # G = 24: two tiles, 8-row tail
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{c[0]}-Hq{c[1]}-Hkv{c[2]}-d{c[3]}-"
                         f"bs{c[4]}-{c[6]}")
def test_decode_small(case):
    S, Hq, Hkv, d, bs, lens, kv = case
    spec = W.DecodeSpec(S, Hq, Hkv, d, 1, max(lens), bs, kv, kv, kv)
    t = W.make_decode(spec, seed=1, lens=lens)
    O_ref, lse_ref = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                         t["seq_lens"])
    g = _dev(t)
    for out in (torch.float32, W.DTYPES[kv]):
        O, lse = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                             max_seq_len=max(lens), out_dtype=out)
        assert attn.last_launch_count() == 2
        assert attn.last_error() == attn.OK
        assert_out(O, O_ref)
        assert_lse(lse, lse_ref)


@pytest.mark.parametrize("d,G", [(d, G) for d in (64, 128, 256) for G in (1, 4, 8, 16)] +
                         [(64, 32),    # d = 64, G = 32: one warp serving two row tiles
                          (128, 32),   # two consumer groups, one row tile each
                          (256, 32)])
def test_decode_e4m3(d, G):
    spec = W.DecodeSpec(3, 2 * G, 2, d, 1, 2000, 16, "bf16", "e4m3", "bf16")
    t = W.make_decode(spec, seed=2, lens=[2000, 1500, 37], keep_unquantised=True)
    g = _dev(t)
    O, lse = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                         max_seq_len=2000, k_scale=g["k_scale"], v_scale=g["v_scale"],
                         out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    # the kernel's arithmetic, against the oracle fed the dequantised cache
    O_dq, lse_dq = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                       t["seq_lens"], k_scale=t["k_scale"],
                                       v_scale=t["v_scale"])
    assert_out(O, O_dq)
    assert_lse(lse, lse_dq)
    # the quantisation budget, against the oracle fed the unquantised cache
    O_src, _ = oracle.decode_paged(t["q"], t["Kc_src"], t["Vc_src"], t["block_table"],
                                   t["seq_lens"])
    long_rows = [0, 1]  # long sequences average the per-element quantisation error
    assert_out(O[long_rows], O_src[long_rows], atol=ATOL_FP8)


def _rising_cache(t, spec, rise=40.0, noise=0.1, seed=0):
    """Rewrite a decode case so that the scores climb along each sequence:
    q components about 1, the key of logical token p about r_p (r rising
    linearly to a log2-domain score of `rise` at the longest sequence's
    end).  Each row's reference max then goes stale unit after unit."""
    g = torch.Generator().manual_seed(seed)
    S, d, bs = spec.num_seqs, spec.d, spec.block_size
    t["q"] = (1.0 + noise * torch.randn(S, spec.Hq, d, generator=g)).to(t["q"].dtype)
    r_max = rise / (1.4426950408889634 * d ** 0.5)
    K = noise * torch.randn(t["Vc"].shape, generator=g)
    lens = t["seq_lens"].tolist()
    for s_i, n in enumerate(lens):
        for b in range((n + bs - 1) // bs):
            pos = torch.arange(b * bs, b * bs + bs, dtype=torch.float32)
            K[int(t["block_table"][s_i, b])] += (r_max * pos / max(lens)).view(1, bs, 1)
    return K


@pytest.mark.parametrize("kv,d,G", [("e4m3", 64, 4), ("e4m3", 64, 32), ("e4m3", 128, 8),
                                    ("e4m3", 256, 16), ("bf16", 128, 4)])
def test_decode_rising_scores_move_the_reference(kv, d, G):
    """Units are computed against each row's current reference max and kept
    while no partial row sum of p exceeds the kernel's limit; climbing
    scores exercise kept units (p far above 1) and units redone from a new
    row max."""
    lens = [2000, 1500, 600, 37]
    spec = W.DecodeSpec(len(lens), 2 * G, 2, d, 1, max(lens), 16, "bf16", kv, "bf16")
    t = W.make_decode(spec, seed=5, lens=lens)
    K = _rising_cache(t, spec, seed=d + G)
    if kv == "e4m3":
        t["Kc"], t["k_scale"] = W.quantize_e4m3_per_head(K.to(torch.bfloat16), 1)
    else:
        t["Kc"] = K.to(torch.bfloat16)
    g = _dev(t)
    O, lse = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                         max_seq_len=max(lens), k_scale=g["k_scale"], v_scale=g["v_scale"],
                         out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    O_ref, lse_ref = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                         t["seq_lens"], k_scale=t["k_scale"],
                                         v_scale=t["v_scale"])
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


def test_decode_empty_and_boundary_lengths():
    lens = [0, 16, 32, 1, 0]
    spec = W.DecodeSpec(5, 4, 2, 128, 1, 32, 16, "bf16", "bf16", "bf16")
    t = W.make_decode(spec, seed=3, lens=[max(x, 1) for x in lens])
    t["seq_lens"] = torch.tensor(lens, dtype=torch.int32)
    O_ref, lse_ref = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                         t["seq_lens"])
    g = _dev(t)
    O, lse = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                         max_seq_len=32, out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    assert (O[0] == 0).all() and (O[4] == 0).all()
    assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[4]).all()
    assert_out(O, O_ref)
    assert_lse(lse, lse_ref)


def test_decode_bad_block_index_is_reported_not_read():
    spec = W.DecodeSpec(3, 4, 2, 128, 1, 64, 16, "bf16", "bf16", "bf16")
    t = W.make_decode(spec, seed=4, lens=[64, 20, 33])
    g = _dev(t)
    g["block_table"][1, 1] = t["num_blocks"] + 5  # out of range
    O, lse = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                         max_seq_len=64, out_dtype=torch.float32)
    assert attn.last_error() == attn.ERR_INVALID
    assert (O[1] == 0).all() and torch.isnan(lse[1]).all()
    O_ref, _ = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                                   seq_subset=[0, 2])
    assert_out(O[[0, 2]], O_ref[[0, 2]])
    assert attn.last_error() == attn.OK  # the error word was cleared


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_decode_full_size_sampled_sequences(out):
    """The 64-sequence paged-decode workload in the launch configuration the
    benchmark times (bf16 output there), on sampled sequences: the shortest,
    the longest and six others."""
    spec = W.DECODE_WORKLOADS["paged-decode"]
    t = W.make_decode(spec, seed=0, device="cuda")
    lens = t["seq_lens"].cpu()
    O, lse = attn.decode(t["q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                         max_seq_len=spec.len_hi, out_dtype=W.DTYPES[out])
    assert attn.last_error() == attn.OK
    order = torch.argsort(lens)
    pick = sorted({int(order[0]), int(order[-1]), 7, 40, 3, 21, 55, 63})
    # gather the sampled sequences' blocks into a compact cache for the oracle
    bt = t["block_table"].cpu()
    rows, phys = [], []
    for s in pick:
        nblk = (int(lens[s]) + spec.block_size - 1) // spec.block_size
        phys.append(bt[s, :nblk])
    allb = torch.cat(phys).long()
    Kc = t["Kc"][allb.cuda()].cpu()
    Vc = t["Vc"][allb.cuda()].cpu()
    table = torch.full((len(pick), bt.shape[1]), -1, dtype=torch.int32)
    off = 0
    for i, p in enumerate(phys):
        table[i, :len(p)] = torch.arange(off, off + len(p), dtype=torch.int32)
        off += len(p)
    O_ref, lse_ref = oracle.decode_paged(t["q"][pick].cpu(), Kc, Vc, table, lens[pick])
    assert_out(O[pick], O_ref)
    assert_lse(lse[pick], lse_ref)
    assert torch.isfinite(O).all()


# every cell of the G x d x cache-format sweep (code-journey.com "Attention
# co-design", Group Size (G) x Head Dimension (Hsz)): 32 sequences x 8192
SWEEP_DECODE = [W.sweep_decode(G, d, kv) for kv in ("bf16", "e4m3") for G in (1, 4, 8, 16)
                for d in (64, 128, 256)]


@pytest.mark.parametrize("spec", SWEEP_DECODE, ids=lambda s: s.name)
def test_decode_sweep_full_size_sampled_sequences(spec):
    """The G x d sweep at full size (32 sequences x 8192 tokens, every split
    busy, several CTAs per SM), checked on sampled sequences."""
    t = W.make_decode(spec, seed=0, device="cuda")
    O, lse = attn.decode(t["q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                         max_seq_len=spec.len_hi, k_scale=t["k_scale"], v_scale=t["v_scale"],
                         out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    pick = [0, 13, spec.num_seqs - 1]
    bt = t["block_table"].cpu()
    nblk = (spec.len_hi + spec.block_size - 1) // spec.block_size
    phys = torch.cat([bt[s, :nblk] for s in pick]).long()
    Kc, Vc = t["Kc"][phys.cuda()].cpu(), t["Vc"][phys.cuda()].cpu()
    table = torch.arange(len(pick) * nblk, dtype=torch.int32).view(len(pick), nblk)
    ks = None if t["k_scale"] is None else t["k_scale"].cpu()
    vs = None if t["v_scale"] is None else t["v_scale"].cpu()
    O_ref, lse_ref = oracle.decode_paged(t["q"][pick].cpu(), Kc, Vc, table,
                                         t["seq_lens"][pick].cpu(), k_scale=ks, v_scale=vs)
    assert_out(O[pick], O_ref)
    assert_lse(lse[pick], lse_ref)
    assert torch.isfinite(O).all()
    # the bf16 output the benchmark writes: the same call rounded once
    O16, _ = attn.decode(t["q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                         max_seq_len=spec.len_hi, k_scale=t["k_scale"], v_scale=t["v_scale"],
                         out_dtype=torch.bfloat16)
    assert attn.last_error() == attn.OK
    assert torch.equal(O16, O.to(torch.bfloat16))


# ----------------------------------------------------------------- append

@pytest.mark.parametrize("kv,d", [("bf16", 128), ("f16", 64), ("e4m3", 128), ("e4m3", 256)])
def test_kv_append_bit_exact(kv, d):
    src = "bf16" if kv == "e4m3" else kv
    spec = W.DecodeSpec(4, 8, 2, d, 1, 100, 16, src, kv, src)
    t = W.make_decode(spec, seed=5, lens=[100, 48, 17, 64], extra_blocks=4)
    T = 9
    kn, vn = W.make_append(T, 2, d, src, seed=5)
    seq_ids = torch.tensor([0, 1, 1, 2, 3, 3, 3, 0, 2], dtype=torch.int32)
    positions = torch.tensor([99, 0, 47, 16, 63, 62, 5, 3, 10], dtype=torch.int32)
    Ko, Vo = oracle.kv_append(kn, vn, t["Kc"], t["Vc"], t["block_table"], seq_ids, positions,
                              t["k_scale"], t["v_scale"])
    g = _dev(t)
    attn.kv_append(kn.cuda(), vn.cuda(), g["Kc"], g["Vc"], g["block_table"], seq_ids.cuda(),
                   positions.cuda(), g["k_scale"], g["v_scale"])
    assert attn.last_launch_count() == 1
    assert attn.last_error() == attn.OK
    assert np.array_equal(oracle._as_np(g["Kc"].cpu()), Ko)
    assert np.array_equal(oracle._as_np(g["Vc"].cpu()), Vo)


def test_kv_append_rejects_bad_entries_on_device():
    spec = W.DecodeSpec(2, 4, 2, 128, 1, 32, 16, "bf16", "bf16", "bf16")
    t = W.make_decode(spec, seed=6, lens=[32, 16])
    kn, vn = W.make_append(3, 2, 128, "bf16", seed=6)
    seq_ids = torch.tensor([0, 5, 1], dtype=torch.int32)       # seq 5 does not exist
    positions = torch.tensor([3, 0, 40], dtype=torch.int32)    # pos 40 is past the table
    g = _dev(t)
    before_k = g["Kc"].clone()
    attn.kv_append(kn.cuda(), vn.cuda(), g["Kc"], g["Vc"], g["block_table"], seq_ids.cuda(),
                   positions.cuda())
    assert attn.last_error() == attn.ERR_INVALID
    Ko, _ = oracle.kv_append(kn[:1], vn[:1], t["Kc"], t["Vc"], t["block_table"], seq_ids[:1],
                             positions[:1])
    assert np.array_equal(oracle._as_np(g["Kc"].cpu()), Ko)
    assert not torch.equal(before_k, g["Kc"])


def test_append_then_decode_sees_new_token():
    """Append one token per sequence at position len, then decode with len+1:
    the result equals the oracle over the extended sequences."""
    spec = W.DecodeSpec(3, 8, 2, 128, 1, 64, 16, "bf16", "bf16", "bf16")
    lens = [31, 32, 5]
    t = W.make_decode(spec, seed=7, lens=[x + 1 for x in lens])
    kn, vn = W.make_append(3, 2, 128, "bf16", seed=7)
    seq_ids = torch.arange(3, dtype=torch.int32)
    positions = torch.tensor(lens, dtype=torch.int32)
    Ko, Vo = oracle.kv_append(kn, vn, t["Kc"], t["Vc"], t["block_table"], seq_ids, positions)
    Ko_t = torch.from_numpy(Ko.view(np.int16)).view(torch.bfloat16)
    Vo_t = torch.from_numpy(Vo.view(np.int16)).view(torch.bfloat16)
    O_ref, _ = oracle.decode_paged(t["q"], Ko_t, Vo_t, t["block_table"], t["seq_lens"])
    g = _dev(t)
    attn.kv_append(kn.cuda(), vn.cuda(), g["Kc"], g["Vc"], g["block_table"], seq_ids.cuda(),
                   positions.cuda())
    O, _ = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                       max_seq_len=64, out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    assert_out(O, O_ref)
