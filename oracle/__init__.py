"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

The numerical work lives in ``attn_oracle.c`` (plain C, fp64, materialised
score matrices); this module compiles it with gcc and wraps it with ctypes.
``recurrence.py`` restates the blockwise online-softmax recurrence and the
split combine for the invariant tests, and ``formulas.py`` holds the closed
forms the pages print (score bytes, KV-cache bytes, arithmetic intensity,
softmax operation counts).

Sources (page title, section):
  auturnal.com "From attention to IO-aware execution" §2 (SDPA), §8 (max
  subtraction, (m, l, u) statistics), §9 (KV-cache size);
  papanda925.com "Transformer complexity strategies", standard-attention
  pseudocode and KV-cache concept;
  code-journey.com "Attention co-design for long-context inference", Group
  Size (G);
  marketmaker.cc "Flash Attention and sequence length", causal masking.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# element-format codes shared with attn_oracle.c (its own enum)
F16, BF16, F32, E4M3, F64 = 0, 1, 2, 3, 4

_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so (gcc -O2 -fopenmp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.oracle_sdpa.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                  i32, f64, i32, vp]
        L.oracle_sdpa.restype = i32
        L.oracle_sdpa_rows.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, i32, i32, i32,
                                       i32, i32, i32, f64, i32]
        L.oracle_sdpa_rows.restype = i32
        L.oracle_decode_paged.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp,
                                          i32, i32, i32, i32, i32, i32, i32, f64, vp, i32,
                                          i32, vp]
        L.oracle_decode_paged.restype = i32
        L.oracle_backward.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      i32, i32, i32, i32, i32, i32, i32, f64, i32]
        L.oracle_backward.restype = i32
        L.oracle_prefill_paged.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, vp, i32, i32,
                                           i32, i32, i32, i32, i32, i32, i32, f64, i32, i32,
                                           i32]
        L.oracle_prefill_paged.restype = i32
        L.oracle_kv_append.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, i32,
                                       i32, i32, i32, i32, i32, i32]
        L.oracle_kv_append.restype = i32
        L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_f64.restype = f64
        L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f64.restype = f64
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_f64.restype = f64
        L.oracle_encode_e4m3_array.argtypes = [vp, vp, ctypes.c_longlong]
        L.oracle_encode_e4m3_array.restype = None
        L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
        L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        _lib = L
    return _lib


# ------------------------------------------------------------------ helpers

def _as_np(x):
    """Host array view of a CPU torch tensor or numpy array (no copy of data
    values: torch half/bfloat16/float8 tensors are viewed as raw bits)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            assert x.device.type == "cpu", "oracle inputs live on the host"
            x = x.contiguous()
            if x.dtype in (torch.float16, torch.bfloat16):
                return x.view(torch.int16).numpy().view(np.uint16)
            if x.dtype == torch.float8_e4m3fn:
                return x.view(torch.uint8).numpy()
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x)


def dtype_code(x) -> int:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32,
                    torch.float8_e4m3fn: E4M3, torch.float64: F64}[x.dtype]
    except ImportError:  # pragma: no cover
        pass
    return {np.dtype(np.float32): F32, np.dtype(np.float64): F64,
            np.dtype(np.uint8): E4M3}[np.asarray(x).dtype]


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


# ------------------------------------------------------------- public calls

def sdpa(Q, K, V, causal: bool, scale: float | None = None, nthreads: int = 0,
         return_counts: bool = False):
    """Exact attention.  Q [B,Hq,nq,d], K/V [B,Hkv,nkv,d] (same element type).
    Returns (O [B,Hq,nq,d] fp64, lse [B,Hq,nq] fp64[, (macs, exps)])."""
    code = dtype_code(Q)
    assert dtype_code(K) == code and dtype_code(V) == code
    q, k, v = _as_np(Q), _as_np(K), _as_np(V)
    B, Hq, nq, d = q.shape
    _, Hkv, nkv, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.zeros((B, Hq, nq, d), np.float64)
    lse = np.zeros((B, Hq, nq), np.float64)
    counts = np.zeros(2, np.int64)
    rc = lib().oracle_sdpa(_p(q), _p(k), _p(v), code, _p(O), _p(lse), B, Hq, Hkv, nq, nkv,
                           d, int(causal), float(scale), nthreads, _p(counts))
    if rc != 0:
        raise ValueError("oracle_sdpa: invalid arguments")
    if return_counts:
        return O, lse, (int(counts[0]), int(counts[1]))
    return O, lse


def sdpa_rows(Q, K, V, rows, causal: bool, scale: float | None = None, nthreads: int = 0):
    """Selected rows (b, h, i) of exact attention; returns (O [r,d], lse [r])."""
    code = dtype_code(Q)
    q, k, v = _as_np(Q), _as_np(K), _as_np(V)
    B, Hq, nq, d = q.shape
    _, Hkv, nkv, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.ascontiguousarray(np.asarray(rows, np.int64).reshape(-1, 3))
    O = np.zeros((rows.shape[0], d), np.float64)
    lse = np.zeros(rows.shape[0], np.float64)
    rc = lib().oracle_sdpa_rows(_p(q), _p(k), _p(v), code, _p(rows), rows.shape[0], _p(O),
                                _p(lse), B, Hq, Hkv, nq, nkv, d, int(causal), float(scale),
                                nthreads)
    if rc != 0:
        raise ValueError("oracle_sdpa_rows: invalid arguments")
    return O, lse


def decode_paged(q, Kc, Vc, block_table, seq_lens, scale: float | None = None,
                 k_scale=None, v_scale=None, seq_subset=None, nthreads: int = 0,
                 return_counts: bool = False):
    """One-token attention over a block-paged cache [num_blocks,Hkv,bs,d].
    Returns (O [S,Hq,d], lse [S,Hq]) in fp64 (rows outside seq_subset are 0)."""
    qc, kc = dtype_code(q), dtype_code(Kc)
    qn, Kn, Vn = _as_np(q), _as_np(Kc), _as_np(Vc)
    bt = np.ascontiguousarray(_as_np(block_table).astype(np.int32))
    sl = np.ascontiguousarray(_as_np(seq_lens).astype(np.int32))
    S, Hq, d = qn.shape
    num_blocks, Hkv, bs, _ = Kn.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    ks = None if k_scale is None else np.ascontiguousarray(_as_np(k_scale).astype(np.float32))
    vs = None if v_scale is None else np.ascontiguousarray(_as_np(v_scale).astype(np.float32))
    sub = None if seq_subset is None else np.ascontiguousarray(np.asarray(seq_subset, np.int32))
    O = np.zeros((S, Hq, d), np.float64)
    lse = np.zeros((S, Hq), np.float64)
    counts = np.zeros(2, np.int64)
    rc = lib().oracle_decode_paged(_p(qn), qc, _p(Kn), _p(Vn), kc, _p(ks), _p(vs), _p(bt),
                                   _p(sl), _p(O), _p(lse), S, Hq, Hkv, d, bs, bt.shape[1],
                                   num_blocks, float(scale), _p(sub),
                                   0 if sub is None else len(sub), nthreads, _p(counts))
    if rc != 0:
        raise ValueError("oracle_decode_paged: invalid arguments")
    if return_counts:
        return O, lse, (int(counts[0]), int(counts[1]))
    return O, lse


def backward(Q, K, V, dO, causal: bool, scale: float | None = None, nthreads: int = 0,
             magnitudes: bool = False, d_err=None):
    """Gradients of exact attention for upstream gradient dO [B,Hq,nq,d]:
    returns (dQ [B,Hq,nq,d], dK, dV [B,Hkv,nkv,d]) in fp64, plus (with
    magnitudes=True) the per-element sums of |terms| (mag_q, mag_k, mag_v).
    With d_err [B,Hq,nq] (a bound on a perturbation of each row's D_i), the
    magnitudes tuple also carries the resulting bounds on the change of dQ
    and dK (dsens_q, dsens_k)."""
    code = dtype_code(Q)
    assert dtype_code(K) == code and dtype_code(V) == code and dtype_code(dO) == code
    q, k, v, go = _as_np(Q), _as_np(K), _as_np(V), _as_np(dO)
    B, Hq, nq, d = q.shape
    _, Hkv, nkv, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dQ = np.zeros(q.shape, np.float64)
    dK = np.zeros(k.shape, np.float64)
    dV = np.zeros(k.shape, np.float64)
    mq = np.zeros(q.shape, np.float64) if magnitudes else None
    mk = np.zeros(k.shape, np.float64) if magnitudes else None
    mv = np.zeros(k.shape, np.float64) if magnitudes else None
    de = None if d_err is None else np.ascontiguousarray(np.asarray(d_err, np.float64))
    sq = np.zeros(q.shape, np.float64) if de is not None else None
    sk = np.zeros(k.shape, np.float64) if de is not None else None
    rc = lib().oracle_backward(_p(q), _p(k), _p(v), _p(go), code, _p(dQ), _p(dK), _p(dV),
                               _p(mq), _p(mk), _p(mv), _p(de), _p(sq), _p(sk), B, Hq, Hkv, nq,
                               nkv, d, int(causal), float(scale), nthreads)
    if rc != 0:
        raise ValueError("oracle_backward: invalid arguments")
    if magnitudes:
        mags = (mq, mk, mv) if de is None else (mq, mk, mv, sq, sk)
        return dQ, dK, dV, mags
    return dQ, dK, dV


def prefill_paged(Q, Kc, Vc, block_table, seq_lens, causal: bool, scale: float | None = None,
                  rows=None, nthreads: int = 0):
    """n_q query rows per sequence against its block-paged cache (the new
    tokens are the sequence's last n_q).  Q [B,Hq,n_q,d]; caches
    [num_blocks,Hkv,bs,d]; rows = (lo, hi) limits the query rows computed.
    Returns (O [B,Hq,hi-lo,d], lse [B,Hq,hi-lo]) in fp64."""
    qn, Kn, Vn = _as_np(Q), _as_np(Kc), _as_np(Vc)
    bt = np.ascontiguousarray(_as_np(block_table).astype(np.int32))
    sl = np.ascontiguousarray(_as_np(seq_lens).astype(np.int32))
    B, Hq, n_q, d = qn.shape
    num_blocks, Hkv, bs, _ = Kn.shape
    lo, hi = (0, n_q) if rows is None else rows
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.zeros((B, Hq, hi - lo, d), np.float64)
    lse = np.zeros((B, Hq, hi - lo), np.float64)
    rc = lib().oracle_prefill_paged(_p(qn), dtype_code(Q), _p(Kn), _p(Vn), dtype_code(Kc),
                                    _p(bt), _p(sl), _p(O), _p(lse), B, Hq, Hkv, n_q, d, bs,
                                    bt.shape[1], num_blocks, int(causal), float(scale), lo, hi,
                                    nthreads)
    if rc != 0:
        raise ValueError("oracle_prefill_paged: invalid arguments")
    return O, lse


def kv_append(k_new, v_new, Kc, Vc, block_table, seq_ids, positions, k_scale=None,
              v_scale=None):
    """Returns updated copies (numpy, raw bits) of the K and V caches."""
    sc = dtype_code(k_new)
    kc = dtype_code(Kc)
    kn, vn = _as_np(k_new), _as_np(v_new)
    Kout, Vout = _as_np(Kc).copy(), _as_np(Vc).copy()
    bt = np.ascontiguousarray(_as_np(block_table).astype(np.int32))
    sid = np.ascontiguousarray(_as_np(seq_ids).astype(np.int32))
    pos = np.ascontiguousarray(_as_np(positions).astype(np.int32))
    ks = None if k_scale is None else np.ascontiguousarray(_as_np(k_scale).astype(np.float32))
    vs = None if v_scale is None else np.ascontiguousarray(_as_np(v_scale).astype(np.float32))
    T, Hkv, d = kn.shape
    num_blocks, _, bs, _ = Kout.shape
    rc = lib().oracle_kv_append(_p(kn), _p(vn), sc, _p(Kout), _p(Vout), kc, _p(ks), _p(vs),
                                _p(bt), _p(sid), _p(pos), T, Hkv, d, bs, bt.shape[1],
                                bt.shape[0], num_blocks)
    if rc != 0:
        raise ValueError("oracle_kv_append: invalid arguments")
    return Kout, Vout


_E4M3_LUT = None


def dequantize_e4m3(codes, scale, head_dim: int = 1) -> np.ndarray:
    """fp64 values of E4M3 codes times a per-head scale: code -> value by the
    oracle's own bit-level decoder (all 256 codes), multiplied by
    scale[head] along axis `head_dim` after flattening the axes before it
    (scale has one entry per (leading index, head) pair, in order)."""
    global _E4M3_LUT
    if _E4M3_LUT is None:
        _E4M3_LUT = np.array([e4m3_decode(i) for i in range(256)], np.float64)
    c = _as_np(codes)
    v = _E4M3_LUT[c]
    sc = np.asarray(_as_np(scale), np.float64).reshape(-1)
    lead = int(np.prod(c.shape[:head_dim + 1]))
    assert sc.size == lead, "one scale per head"
    return (v.reshape(lead, -1) * sc[:, None]).reshape(c.shape)


def encode_e4m3(x) -> np.ndarray:
    """E4M3 codes (round to nearest even, saturating) of fp32 values, by the
    oracle's own encoder."""
    a = np.ascontiguousarray(np.asarray(x, np.float32))
    out = np.zeros(a.shape, np.uint8)
    lib().oracle_encode_e4m3_array(_p(a), _p(out), a.size)
    return out


def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_to_f64(code))


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_f32_to_e4m3(x))


def f16_decode(bits: int) -> float:
    return float(lib().oracle_f16_to_f64(bits))


def bf16_decode(bits: int) -> float:
    return float(lib().oracle_bf16_to_f64(bits))
