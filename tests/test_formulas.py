"""The pages' closed forms, pinned against their printed values and against
first-principles counts (oracle operation counts, bytes of real tensors)."""
import json
import os

import numpy as np
import torch

import oracle
from oracle import formulas as F
from exact_io_aware_106_b300 import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")))
MiB, GiB = 2 ** 20, 2 ** 30


def test_score_bytes_printed_table():
    g = GOLD["score_bytes_fp32_one_head"]
    for n, mib in zip(g["n"], g["MiB"]):
        assert F.score_bytes(n) == mib * MiB
        assert np.zeros((n, n), np.float32).nbytes == mib * MiB
    # doubling the length quadruples the term
    assert F.score_bytes(2048) == 4 * F.score_bytes(1024)


def test_fig2_scores_vs_kv_cache():
    g = GOLD["fig2_8192_tokens"]
    assert F.score_bytes(g["tokens"], heads=g["score_heads"], layers=g["score_layers"],
                         bytes_per=g["score_bytes_per_scalar"]) == g["score_GiB"] * GiB
    # the page leaves d_h out; 1 GiB needs d_h = 128
    dh = [d for d in (32, 64, 96, 128, 256)
          if F.kv_cache_bytes(g["kv_layers"], g["tokens"], g["kv_heads"], d,
                              g["kv_bytes_per_scalar"]) == g["kv_GiB"] * GiB]
    assert dh == [128]


def test_kv_cache_formula_equals_allocated_cache():
    """2*L*n*h_kv*d_h*b equals the bytes of the K and V caches the harness
    allocates (L = 1, n = total tokens, block-aligned lengths)."""
    for kv, b in (("bf16", 2), ("e4m3", 1)):
        spec = W.DecodeSpec(4, 8, 2, 32, 16, 64, 16, "bf16", kv, "bf16")
        t = W.make_decode(spec, seed=1, lens=[16, 32, 48, 64])
        n = int(t["seq_lens"].sum())
        allocated = t["Kc"].numel() * t["Kc"].element_size() + \
            t["Vc"].numel() * t["Vc"].element_size()
        assert allocated == F.kv_cache_bytes(1, n, 2, 32, b)


def test_arithmetic_intensity_decode_first_principles_and_printed():
    """Decode AI = FLOPs / bytes at 1 B per element: FLOPs from the oracle's
    own multiply-adds (2 flops each), bytes = q + K + V + O of one KV head."""
    for G, KVSL in ((1, 64), (4, 96), (8, 40)):
        d = 8
        spec = W.DecodeSpec(1, G, 1, d, KVSL, KVSL, 16, "bf16", "bf16", "bf16")
        t = W.make_decode(spec, seed=3)
        _, _, (macs, _) = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                              t["seq_lens"], return_counts=True)
        flops = 2 * macs
        nbytes = (G * d) + (KVSL * d) + (KVSL * d) + (G * d)
        assert abs(flops / nbytes - F.ai_decode(G, KVSL)) < 1e-12
    for G, KVSL, printed in GOLD["ai_decode_printed"]["cases"]:
        assert abs(F.ai_decode(G, KVSL) - printed) < 0.01


def test_arithmetic_intensity_prefill_first_principles_and_printed_discrepancy():
    for G, ISL in ((1, 16), (4, 24), (8, 12)):
        d = 8
        Q = torch.randn(1, G, ISL, d, dtype=torch.float64)
        K = torch.randn(1, 1, ISL, d, dtype=torch.float64)
        _, _, (macs, _) = oracle.sdpa(Q, K, K, False, return_counts=True)
        nbytes = (G * ISL * d) * 2 + (ISL * d) * 2  # Q and O; K and V
        assert abs(2 * macs / nbytes - F.ai_prefill(G, ISL)) < 1e-9
    g = GOLD["ai_prefill_printed"]
    (G1, L1, p1), (G2, L2, p2) = g["cases"]
    a1, a2 = F.ai_prefill(G1, L1), F.ai_prefill(G2, L2)
    assert abs(a1 - 58254.2) < 0.1 and abs(a2 - 61680.9) < 0.1
    assert abs(a1 - p1) > 1000 and abs(a2 - p2) > 1000  # printed values are wrong
    assert a2 / a1 - 1 < g["claim_improvement_below"]  # "<6%" still holds


def test_softmax_operation_counts_from_oracle():
    PB, QH, ISL, d = 2, 3, 10, 4
    Q = torch.randn(PB, QH, ISL, d, dtype=torch.float64)
    K = torch.randn(PB, QH, ISL, d, dtype=torch.float64)
    _, _, (_, exps) = oracle.sdpa(Q, K, K, False, return_counts=True)
    assert exps == F.softmax_ops_prefill(PB, QH, ISL)
    # the count does not depend on the head size
    Q2 = torch.randn(PB, QH, ISL, 4 * d, dtype=torch.float64)
    K2 = torch.randn(PB, QH, ISL, 4 * d, dtype=torch.float64)
    _, _, (_, exps2) = oracle.sdpa(Q2, K2, K2, False, return_counts=True)
    assert exps2 == exps
    spec = W.DecodeSpec(3, 4, 2, 8, 33, 33, 16, "bf16", "bf16", "bf16")
    t = W.make_decode(spec, seed=5)
    _, _, (_, dexps) = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                           t["seq_lens"], return_counts=True)
    assert dexps == F.softmax_ops_decode(3, 4, 33)


def test_trading_day_figure_is_recorded_inconsistent():
    g = GOLD["trading_day_scores"]
    b = F.score_bytes(g["steps"], heads=g["heads"], bytes_per=g["bytes_per_scalar"])
    assert b == 13_141_440_000
    assert abs(b / 1e9 - g["printed_GB"]) > 0.2 and abs(b / GiB - g["printed_GB"]) > 0.6
