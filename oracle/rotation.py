"""Incoherent processing for fp8 attention -- TEST INFRASTRUCTURE ONLY.

marketmaker.cc "Flash Attention and sequence length", FA3: before fp8
quantisation Q and K are multiplied by the same random orthogonal matrix, so
that a few large entries (outliers) are spread over all d components and the
per-head scale (amax / 448) no longer has to cover them; Q K^T is unchanged
because the matrix is orthogonal.

The matrix used here is diag(s) H_d with random signs s_i = +-1 and H_d the
Sylvester Hadamard matrix (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]),
entries +-1, H_d H_d^T = d I.  It is left unnormalised, so
(Q diag(s) H)(K diag(s) H)^T = d Q K^T: the attention scale becomes
scale / d (exact for d a power of two).
"""
from __future__ import annotations

import numpy as np

from . import dequantize_e4m3, encode_e4m3


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (a power of two), int64 +-1."""
    assert d > 0 and d & (d - 1) == 0
    H = np.ones((1, 1), np.int64)
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def rotate(x, signs) -> np.ndarray:
    """x [..., d] (fp64) times diag(signs) H_d."""
    x = np.asarray(x, np.float64)
    s = np.asarray(signs, np.float64)
    return (x * s) @ hadamard(x.shape[-1]).astype(np.float64)


def quantize_per_head(xr: np.ndarray, head_axes: int = 2):
    """Per-head E4M3 quantisation of a rotated tensor [B, H, n, d]: scale =
    amax/448 over each (b, h), codes = e4m3_rn_satfinite(x / scale) with the
    division rounded to fp32 (the oracle's encoder).  Returns (codes,
    scales[B*H])."""
    lead = int(np.prod(xr.shape[:head_axes]))
    flat = xr.reshape(lead, -1)
    amax = np.abs(flat).max(axis=1)
    scale = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32)
    q = (flat.astype(np.float32) / scale[:, None]).astype(np.float32)
    return encode_e4m3(q).reshape(xr.shape), scale


def dequantize(codes, scales, head_axes: int = 2) -> np.ndarray:
    return dequantize_e4m3(codes, scales, head_axes - 1)
