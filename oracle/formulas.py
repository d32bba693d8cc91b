"""Closed forms the pages print -- TEST INFRASTRUCTURE ONLY.

Each function restates one counting formula; the tests pin them against the
values printed on the pages and against first-principles counts taken from
the oracle itself (multiply-adds and exp evaluations it performs, bytes of
the tensors it is given), never against a retyped copy of the formula.
"""
from __future__ import annotations


def score_bytes(n: int, heads: int = 1, layers: int = 1, bytes_per: int = 4) -> int:
    """Explicitly stored score matrices: n x n per head and layer
    (auturnal.com "From attention to IO-aware execution", §4 and §6)."""
    return n * n * bytes_per * heads * layers


def kv_cache_bytes(L: int, n: int, h_kv: int, d_h: int, b: int) -> int:
    """KV cache of L layers, n positions, h_kv KV heads of size d_h, b bytes
    per scalar: 2*L*n*h_kv*d_h*b (same page, §9; excludes weights, workspace
    and allocator fragmentation)."""
    return 2 * L * n * h_kv * d_h * b


def ai_prefill(G: int, ISL: int) -> float:
    """Prefill arithmetic intensity with 1-byte elements (code-journey.com
    "Attention co-design", Group Size): 2*G*ISL/(G+1)."""
    return 2.0 * G * ISL / (G + 1)


def ai_decode(G: int, KVSL: int) -> float:
    """Decode arithmetic intensity with 1-byte elements: 2*G*KVSL/(G+KVSL)."""
    return 2.0 * G * KVSL / (G + KVSL)


def softmax_ops_prefill(PB: int, QH: int, ISL: int) -> int:
    """Softmax exponentials in prefill, independent of the head size
    (same page, Head Dimension): PB*QH*ISL^2."""
    return PB * QH * ISL ** 2


def softmax_ops_decode(DB: int, QH: int, KVSL: int) -> int:
    """Softmax exponentials in one decode step: DB*QH*KVSL."""
    return DB * QH * KVSL
