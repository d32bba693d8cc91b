"""Incoherent processing for fp8 attention -- TEST INFRASTRUCTURE ONLY.

marketmaker.cc "Flash Attention and sequence length", FA3 (item 3): before
the block-wise fp8 quantisation, Q and K are multiplied by the same random
orthogonal matrix, so that a few large entries (outliers) are spread over
all d components; Q K^T is unchanged because the matrix is orthogonal.

Block-wise quantisation: each block of `rows_per_block` consecutive rows of
one head gets its own scale, amax / 448 over the block (448 is the largest
finite E4M3 value), so an outlier only coarsens its own block.  The page
names the granularity ("block-wise") but not the block size; 128 rows is
the reading here (one query tile / key block of the attention kernel).
quantize_per_head is the same rule with one block per head.

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


def quantize_per_block(x: np.ndarray, rows_per_block: int = 128, head_axes: int = 2):
    """Block-wise E4M3 quantisation of x [..., n, d] (the leading `head_axes`
    axes index heads): rows r of a head belong to block r // rows_per_block;
    scale[h, blk] = amax / 448 over the block's values (1 where the block is
    all zero), codes = e4m3_rn_satfinite(x / scale) with the division rounded
    to fp32 (the oracle's encoder).  Returns (codes like x, scales
    [heads, ceil(n / rows_per_block)] fp32)."""
    x = np.asarray(x, np.float64)
    n, d = x.shape[-2], x.shape[-1]
    lead = int(np.prod(x.shape[:head_axes]))
    flat = x.reshape(lead, n, d)
    nb = -(-n // rows_per_block)
    scales = np.ones((lead, nb), np.float32)
    codes = np.zeros((lead, n, d), np.uint8)
    for b in range(nb):
        blk = flat[:, b * rows_per_block:(b + 1) * rows_per_block]
        amax = np.abs(blk).reshape(lead, -1).max(axis=1)
        sc = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32)
        scales[:, b] = sc
        q = (blk.astype(np.float32) / sc[:, None, None]).astype(np.float32)
        codes[:, b * rows_per_block:(b + 1) * rows_per_block] = encode_e4m3(q)
    return codes.reshape(x.shape), scales


def dequantize_per_block(codes, scales, rows_per_block: int = 128,
                         head_axes: int = 2) -> np.ndarray:
    """fp64 values of block-wise E4M3 codes: the oracle's bit-level decoder
    times the scale of each row's block."""
    c = np.asarray(codes)
    n, d = c.shape[-2], c.shape[-1]
    lead = int(np.prod(c.shape[:head_axes]))
    v = dequantize_e4m3(c.reshape(lead, n * d), np.ones(lead), 0).reshape(lead, n, d)
    sc = np.asarray(scales, np.float64).reshape(lead, -1)
    row_scale = sc[:, np.arange(n) // rows_per_block]
    return (v * row_scale[:, :, None]).reshape(c.shape)
