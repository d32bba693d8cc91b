"""Pins of the fp64 oracle against what the pages and mathematics fix.

None of these compares the oracle with a retyped copy of itself: each check
uses a library routine (torch SDPA in float64, scipy softmax / logsumexp,
torch's float8/bfloat16 casts, numpy float16), a closed form, an invariant
the pages state, or an exact special case.
"""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
from exact_io_aware_106_b300 import workloads as W


def _rand(shape, seed, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64).to(dtype)


def _torch_ref(Q, K, V, causal, scale):
    """torch SDPA in float64 with KV heads repeated per group and a
    bottom-right causal mask."""
    Q, K, V = Q.double(), K.double(), V.double()
    G = Q.shape[1] // K.shape[1]
    K = K.repeat_interleave(G, dim=1)
    V = V.repeat_interleave(G, dim=1)
    nq, nkv = Q.shape[2], K.shape[2]
    mask = None
    if causal:
        i = torch.arange(nq)[:, None]
        j = torch.arange(nkv)[None, :]
        mask = j <= i + (nkv - nq)
    return torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                            scale=scale)


# ------------------------------------------------------------- element formats

def test_bf16_decode_all_patterns():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_decode(b) for b in range(1 << 16)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_f16_decode_all_patterns():
    ref = np.arange(0, 1 << 16, dtype=np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_decode(b) for b in range(1 << 16)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_e4m3_decode_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range_and_saturates():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x.clamp(-448.0, 448.0).float()
    # every exact midpoint between neighbouring codes exercises ties-to-even
    vals = torch.arange(0, 127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = vals.float()
    mids = (vals[1:] + vals[:-1]) / 2
    x = torch.cat([x, mids, -mids])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in x.numpy()], dtype=np.uint8)
    assert (got == ref).all()
    for v in (448.0, 449.0, 464.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F


# ------------------------------------------------------------ the definition

@pytest.mark.parametrize("B,Hq,Hkv,nq,nkv,d,causal", [
    (1, 1, 1, 7, 7, 8, False),
    (2, 4, 2, 9, 13, 16, True),
    (1, 6, 3, 16, 16, 32, True),
    (2, 2, 2, 5, 21, 4, False),
    (1, 8, 1, 3, 40, 8, True),
])
def test_sdpa_matches_torch_sdpa_fp64(B, Hq, Hkv, nq, nkv, d, causal):
    Q = _rand((B, Hq, nq, d), 1)
    K = _rand((B, Hkv, nkv, d), 2)
    V = _rand((B, Hkv, nkv, d), 3)
    scale = 1.0 / np.sqrt(d)
    O, lse = oracle.sdpa(Q, K, V, causal, scale)
    ref = _torch_ref(Q, K, V, causal, scale).numpy()
    assert np.abs(O - ref).max() < 1e-12
    # lse against scipy's logsumexp over the masked scaled scores
    Kr = K.repeat_interleave(Hq // Hkv, dim=1).numpy()
    S = np.einsum("bhid,bhjd->bhij", Q.numpy(), Kr) * scale
    if causal:
        i = np.arange(nq)[:, None]
        j = np.arange(nkv)[None, :]
        S = np.where(j <= i + (nkv - nq), S, -np.inf)
    assert np.abs(lse - scipy.special.logsumexp(S, axis=-1)).max() < 1e-12


def test_low_precision_inputs_are_decoded_exactly():
    spec = W.PrefillSpec(1, 2, 1, 9, 9, 16, True, "bf16", "bf16")
    t = W.make_prefill(spec, seed=5)
    O, lse = oracle.sdpa(t["Q"], t["K"], t["V"], True)
    ref = _torch_ref(t["Q"], t["K"], t["V"], True, 0.25).numpy()
    assert np.abs(O - ref).max() < 1e-12
    spec = W.PrefillSpec(1, 1, 1, 6, 6, 8, False, "f16", "f32")
    t = W.make_prefill(spec, seed=6)
    O, _ = oracle.sdpa(t["Q"], t["K"], t["V"], False)
    ref = _torch_ref(t["Q"], t["K"], t["V"], False, 1 / np.sqrt(8)).numpy()
    assert np.abs(O - ref).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_rows_are_probabilities(causal):
    """With V = identity (n_kv = d) the output rows are the softmax rows:
    non-negative, summing to 1, equal to scipy's softmax of the scores."""
    n = 12
    Q = _rand((1, 1, n, n), 11)
    K = _rand((1, 1, n, n), 12)
    V = torch.eye(n, dtype=torch.float64).reshape(1, 1, n, n)
    P, _ = oracle.sdpa(Q, K, V, causal, 0.7)
    assert (P >= 0).all()
    assert np.abs(P.sum(-1) - 1.0).max() < 1e-12
    S = (Q[0, 0] @ K[0, 0].T).numpy() * 0.7
    if causal:
        S = np.where(np.tril(np.ones((n, n), bool)), S, -np.inf)
    assert np.abs(P[0, 0] - scipy.special.softmax(S, axis=-1)).max() < 1e-12


@pytest.mark.parametrize("c", [-1000.0, -3.5, 0.25, 1000.0])
def test_max_shift_invariance(c):
    """Adding the same constant to every score of a row leaves the
    probabilities (hence O) unchanged and shifts lse by that constant; the
    shift by +1000 would overflow a naive exp in fp64."""
    n, d = 10, 6
    Q = _rand((1, 2, n, d), 21)
    K = _rand((1, 2, n, d), 22)
    V = _rand((1, 2, n, d), 23)
    scale = 0.5
    O, lse = oracle.sdpa(Q, K, V, True, scale)
    Q2 = torch.cat([Q, torch.full((1, 2, n, 1), c / scale, dtype=torch.float64)], -1)
    K2 = torch.cat([K, torch.ones((1, 2, n, 1), dtype=torch.float64)], -1)
    V2 = torch.cat([V, torch.zeros((1, 2, n, 1), dtype=torch.float64)], -1)
    O2, lse2 = oracle.sdpa(Q2, K2, V2, True, scale)
    assert np.isfinite(O2).all()
    assert np.abs(O2[..., :d] - O).max() < 1e-12
    assert np.abs(lse2 - (lse + c)).max() < 1e-9 * max(1.0, abs(c))
    with np.errstate(over="ignore"):
        assert not np.isfinite(np.exp(np.float64(1000.0)))


def test_equal_scores_give_mean_of_V():
    n, d = 9, 5
    Q = torch.zeros((1, 1, n, d), dtype=torch.float64)
    K = _rand((1, 1, n, d), 31)
    V = _rand((1, 1, n, d), 32)
    O, lse = oracle.sdpa(Q, K, V, False, 1.0)
    assert np.abs(O[0, 0] - V[0, 0].numpy().mean(0)[None, :]).max() < 1e-13
    assert np.abs(lse - np.log(n)).max() < 1e-13
    O, _ = oracle.sdpa(Q, K, V, True, 1.0)
    for i in range(n):
        assert np.abs(O[0, 0, i] - V[0, 0, :i + 1].numpy().mean(0)).max() < 1e-13


def test_causal_row0_is_V0_and_prefix_equals_truncated_noncausal():
    spec = W.PrefillSpec(1, 2, 1, 11, 11, 8, True, "bf16", "bf16")
    t = W.make_prefill(spec, seed=9)
    O, lse = oracle.sdpa(t["Q"], t["K"], t["V"], True)
    V = t["V"].double().numpy()
    assert np.array_equal(O[0, :, 0], np.repeat(V[0, :1, 0], 2, axis=0))
    for i in range(11):
        Oi, _ = oracle.sdpa(t["Q"][:, :, i:i + 1], t["K"][:, :, :i + 1], t["V"][:, :, :i + 1],
                            False)
        assert np.abs(Oi[:, :, 0] - O[:, :, i]).max() < 1e-13
    # bottom-right alignment: n_q < n_kv, last query sees every key
    Ob, _ = oracle.sdpa(t["Q"][:, :, -3:], t["K"], t["V"], True)
    assert np.abs(Ob - O[:, :, -3:]).max() < 1e-13


def test_gqa_equals_mha_with_repeated_kv_and_g1_is_mha():
    Q = _rand((2, 6, 7, 8), 41)
    K = _rand((2, 2, 7, 8), 42)
    V = _rand((2, 2, 7, 8), 43)
    O, lse = oracle.sdpa(Q, K, V, True)
    Or, lser = oracle.sdpa(Q, K.repeat_interleave(3, 1), V.repeat_interleave(3, 1), True)
    assert np.abs(O - Or).max() == 0.0 and np.abs(lse - lser).max() == 0.0
    # head h uses KV head h // G: moving KV head 1 changes only heads 3..5
    K2 = K.clone()
    K2[:, 1] *= 2.0
    O2, _ = oracle.sdpa(Q, K2, V, True)
    assert np.abs(O2[:, :3] - O[:, :3]).max() == 0.0
    assert np.abs(O2[:, 3:] - O[:, 3:]).max() > 1e-3


def test_rows_variant_equals_full():
    Q = _rand((2, 4, 10, 8), 51)
    K = _rand((2, 2, 14, 8), 52)
    V = _rand((2, 2, 14, 8), 53)
    O, lse = oracle.sdpa(Q, K, V, True)
    rows = [(b, h, i) for b in range(2) for h in range(4) for i in (0, 3, 9)]
    Or, lr = oracle.sdpa_rows(Q, K, V, rows, True)
    for r, (b, h, i) in enumerate(rows):
        assert np.abs(Or[r] - O[b, h, i]).max() < 1e-14
        assert abs(lr[r] - lse[b, h, i]) < 1e-14


def test_operation_counts():
    """Softmax exp count and multiply-add count the oracle performs match the
    pages' counting (non-causal prefill, decode)."""
    B, Hq, Hkv, n, d = 2, 4, 2, 12, 8
    Q = _rand((B, Hq, n, d), 61)
    K = _rand((B, Hkv, n, d), 62)
    V = _rand((B, Hkv, n, d), 63)
    _, _, (macs, exps) = oracle.sdpa(Q, K, V, False, return_counts=True)
    assert exps == B * Hq * n * n
    assert macs == 2 * B * Hq * n * n * d


# ------------------------------------------------------------------- decode

@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_decode_paged_equals_sdpa_on_gathered_cache(kv):
    spec = W.DecodeSpec(5, 8, 2, 16, 1, 70, 16, "bf16", kv, "bf16")
    t = W.make_decode(spec, seed=4, lens=[1, 15, 16, 17, 70])
    O, lse = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                                 k_scale=t["k_scale"], v_scale=t["v_scale"])
    for s in range(5):
        L = int(t["seq_lens"][s])
        idx = torch.arange(L)
        blk = t["block_table"][s, idx // 16].long()
        Ks = t["Kc"][blk, :, idx % 16].double()  # [L, Hkv, d]
        Vs = t["Vc"][blk, :, idx % 16].double()
        if kv == "e4m3":
            Ks = t["Kc"][blk, :, idx % 16].float().double() * t["k_scale"].double()[None, :, None]
            Vs = t["Vc"][blk, :, idx % 16].float().double() * t["v_scale"].double()[None, :, None]
        q = t["q"][s].double()[None, :, None, :]
        ref = _torch_ref(q, Ks.permute(1, 0, 2)[None], Vs.permute(1, 0, 2)[None], False,
                         1 / np.sqrt(16))
        assert np.abs(O[s] - ref[0, :, 0].numpy()).max() < 1e-12


def test_decode_empty_sequence_and_subset():
    spec = W.DecodeSpec(3, 4, 1, 8, 1, 20, 16, "bf16", "bf16", "bf16")
    t = W.make_decode(spec, seed=2, lens=[0, 5, 20])
    O, lse = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"])
    assert (O[0] == 0).all() and np.isneginf(lse[0]).all()
    Os, ls = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                                 seq_subset=[2])
    assert np.array_equal(Os[2], O[2]) and (Os[1] == 0).all()


def test_decode_rejects_bad_block_index():
    spec = W.DecodeSpec(2, 2, 1, 8, 16, 16, 16, "bf16", "bf16", "bf16")
    t = W.make_decode(spec, seed=2)
    bt = t["block_table"].clone()
    bt[1, 0] = t["num_blocks"]
    with pytest.raises(ValueError):
        oracle.decode_paged(t["q"], t["Kc"], t["Vc"], bt, t["seq_lens"])


# -------------------------------------------------------------- kv append

@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_kv_append_writes_slot(kv):
    spec = W.DecodeSpec(3, 4, 2, 16, 5, 40, 16, "bf16", kv, "bf16")
    t = W.make_decode(spec, seed=8, lens=[5, 16, 40])
    kn, vn = W.make_append(3, 2, 16, "bf16", seed=8)
    pos = torch.tensor([5, 16, 39], dtype=torch.int32)
    sid = torch.tensor([0, 1, 2], dtype=torch.int32)
    # the block table must cover position 16 of sequence 1
    bt = torch.cat([t["block_table"], torch.full((3, 1), -1, dtype=torch.int32)], 1)
    extra = t["num_blocks"]
    Kc = torch.cat([t["Kc"], t["Kc"][:1]], 0)
    Vc = torch.cat([t["Vc"], t["Vc"][:1]], 0)
    bt[1, 1] = extra
    Ko, Vo = oracle.kv_append(kn, vn, Kc, Vc, bt, sid, pos, t["k_scale"], t["v_scale"])
    Kraw = oracle._as_np(Kc)
    changed = np.argwhere((Ko != Kraw).reshape(Ko.shape[0], Ko.shape[1], Ko.shape[2], -1)
                          .any(-1))
    for r in range(3):
        blk = int(bt[sid[r], pos[r] // 16])
        slot = int(pos[r] % 16)
        for h in range(2):
            if kv == "bf16":
                assert np.array_equal(Ko[blk, h, slot], oracle._as_np(kn[r, h]))
                assert np.array_equal(Vo[blk, h, slot], oracle._as_np(vn[r, h]))
            else:
                # torch casts out-of-range values to NaN; the cache format
                # saturates, so clamp first (RN of a clamped 448 is 448)
                ref_k = (kn[r, h].float() / t["k_scale"][h]).clamp(-448, 448)
                ref_v = (vn[r, h].float() / t["v_scale"][h]).clamp(-448, 448)
                ref_k = ref_k.to(torch.float8_e4m3fn)
                ref_v = ref_v.to(torch.float8_e4m3fn)
                assert np.array_equal(Ko[blk, h, slot], ref_k.view(torch.uint8).numpy())
                assert np.array_equal(Vo[blk, h, slot], ref_v.view(torch.uint8).numpy())
    # nothing outside the three written slots changed
    for b, h, s in changed:
        assert any(b == int(bt[sid[r], pos[r] // 16]) and s == int(pos[r] % 16)
                   for r in range(3))


def test_dequantize_e4m3_per_head_matches_torch_cast():
    """The oracle's per-head E4M3 dequantisation (its own bit-level decoder)
    equals torch's decode of the same codes times the per-head scale."""
    x = torch.randn(2, 3, 5, 8, generator=torch.Generator().manual_seed(11)) * 3
    codes = (x / 0.05).to(torch.float8_e4m3fn)
    scale = torch.linspace(0.5, 2.0, 6)
    got = oracle.dequantize_e4m3(codes, scale, 1)
    want = (codes.to(torch.float64) * scale.double().view(2, 3, 1, 1)).numpy()
    assert np.array_equal(got, want)



# ------------------------------------------------------------ paged prefill

def _gather(Kc, bt, lens, b):
    """Dense [1, Hkv, len, d] copy of sequence b's cache (data movement)."""
    bs = Kc.shape[2]
    L = int(lens[b])
    blocks = bt[b, :(L + bs - 1) // bs].long()
    x = Kc[blocks]                                   # [nblk, Hkv, bs, d]
    x = x.permute(1, 0, 2, 3).reshape(Kc.shape[1], -1, Kc.shape[3])[:, :L]
    return x.unsqueeze(0).contiguous()


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_paged_equals_sdpa_on_gathered_cache(causal):
    spec = W.PagedPrefillSpec(3, 4, 2, 21, 16, 21, 70, 16, causal, "bf16", "f32")
    t = W.make_paged_prefill(spec, seed=3)
    O, lse = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                                  causal)
    for b in range(spec.B):
        K = _gather(t["Kc"], t["block_table"], t["seq_lens"], b)
        V = _gather(t["Vc"], t["block_table"], t["seq_lens"], b)
        Ob, lb = oracle.sdpa(t["Q"][b:b + 1], K, V, causal)
        assert np.allclose(O[b], Ob[0], rtol=0, atol=1e-12)
        assert np.allclose(lse[b], lb[0], rtol=0, atol=1e-12)


def test_prefill_paged_one_query_equals_decode():
    spec = W.PagedPrefillSpec(4, 8, 2, 1, 32, 1, 90, 16, True, "f16", "f32")
    t = W.make_paged_prefill(spec, seed=4)
    O, lse = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"],
                                  True)
    Od, ld = oracle.decode_paged(t["Q"][:, :, 0], t["Kc"], t["Vc"], t["block_table"],
                                 t["seq_lens"])
    assert np.allclose(O[:, :, 0], Od, rtol=0, atol=1e-12)
    assert np.allclose(lse[:, :, 0], ld, rtol=0, atol=1e-12)


def test_prefill_paged_row_range_and_validation():
    spec = W.PagedPrefillSpec(2, 2, 1, 40, 16, 40, 100, 32, True, "bf16", "f32")
    t = W.make_paged_prefill(spec, seed=5)
    O, lse = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"], True)
    Os, ls = oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"], t["seq_lens"], True,
                                  rows=(7, 19))
    assert np.array_equal(Os, O[:, :, 7:19]) and np.array_equal(ls, lse[:, :, 7:19])
    # the last query of a causal row sees every key: equal to the full row
    bt = t["block_table"].clone()
    bt[0, 0] = t["num_blocks"] + 3
    with pytest.raises(ValueError):
        oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], bt, t["seq_lens"], True)
    short = t["seq_lens"].clone()
    short[1] = spec.n_q - 1                      # causal needs len >= n_q
    with pytest.raises(ValueError):
        oracle.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"], short, True)
