"""ctypes binding of libattn.so (include/attn.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks that tensors live on the GPU, passes their device pointers, sizes and
the current CUDA stream, and turns non-zero status codes into exceptions.
There is no fallback: if the library or a GPU is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
_DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2, torch.float8_e4m3fn: 3}

EXPORTS = ("attn_prefill", "attn_prefill_from_host", "attn_prefill_from_host_heads_per_chunk",
           "attn_prefill_paged", "attn_decode_workspace_bytes", "attn_decode",
           "attn_decode_tokens", "attn_kv_append", "attn_backward",
           "attn_backward_workspace_bytes", "attn_rotate_quantize_e4m3",
           "attn_prefill_e4m3_blocks", "attn_last_error", "attn_status_str",
           "attn_last_launch_count", "attn_decode_static_ws", "attn_debug_prefill_timeout",
           "attn_debug_set_hooks")

# Rows per E4M3 scale block in prefill_e4m3_blocks (ATTN_E4M3_SCALE_BLOCK).
E4M3_SCALE_BLOCK = 128

# Scratch size compiled into the library for attn_decode_static_ws.
DECODE_STATIC_WS_BYTES = 16 << 20


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_str(status)} ({status})")


_lib = None


def lib():
    """Load libattn.so (raises OSError if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: run `python -m exact_io_aware_106_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.attn_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                   i32, i32, vp, vp, vp, vp]
        L.attn_prefill.restype = i32
        L.attn_prefill_from_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                             i32, i32, i32, i32, i32, f32, i32, i32, vp, vp, vp,
                                             i32, vp]
        L.attn_prefill_from_host.restype = i32
        L.attn_prefill_from_host_heads_per_chunk.argtypes = [i32] * 7
        L.attn_prefill_from_host_heads_per_chunk.restype = i32
        L.attn_prefill_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                         i32, i32, i32, i32, i32, f32, i32, i32, vp]
        L.attn_prefill_paged.restype = i32
        L.attn_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.attn_decode_workspace_bytes.restype = sz
        L.attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                  i32, f32, i32, i32, i32, vp, vp, vp, sz, vp]
        L.attn_decode.restype = i32
        L.attn_decode_tokens.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                         i32, i32, i32, i32, f32, i32, i32, i32, vp, vp, vp, sz,
                                         vp]
        L.attn_decode_tokens.restype = i32
        L.attn_kv_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                     i32, i32, i32, vp, vp, vp]
        L.attn_kv_append.restype = i32
        L.attn_backward_workspace_bytes.argtypes = [i32, i32, i32]
        L.attn_backward_workspace_bytes.restype = sz
        L.attn_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                    i32, i32, f32, i32, i32, i32, vp, sz, vp]
        L.attn_backward.restype = i32
        L.attn_rotate_quantize_e4m3.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                vp]
        L.attn_rotate_quantize_e4m3.restype = i32
        L.attn_prefill_e4m3_blocks.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                               i32, i32, f32, i32, vp, vp, vp, vp]
        L.attn_prefill_e4m3_blocks.restype = i32
        L.attn_debug_prefill_timeout.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                 i32, i32, f32, i32, i32, ctypes.c_uint, vp]
        L.attn_debug_prefill_timeout.restype = i32
        L.attn_debug_set_hooks.argtypes = [ctypes.c_uint, ctypes.c_uint, vp]
        L.attn_debug_set_hooks.restype = i32
        L.attn_last_error.argtypes = [vp]
        L.attn_last_error.restype = i32
        L.attn_status_str.argtypes = [i32]
        L.attn_status_str.restype = ctypes.c_char_p
        L.attn_decode_static_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                            i32, i32, i32, i32, f32, i32, i32, i32, vp, vp, vp]
        L.attn_decode_static_ws.restype = i32
        L.attn_last_launch_count.argtypes = []
        L.attn_last_launch_count.restype = i32
        _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().attn_status_str(s).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensor must live on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("tensor must be contiguous")


def _check(fn, st):
    if st != OK:
        raise AttnError(fn, st)


def last_launch_count() -> int:
    return lib().attn_last_launch_count()


def last_error(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device error status."""
    return lib().attn_last_error(_stream(stream))


# Test hooks of attn_debug_set_hooks (ATTN_HOOK_*).
HOOK_WITHHOLD_Q = 1
HOOK_WITHHOLD_KV = 2


def debug_set_hooks(wait_limit_us: int, hooks: int, stream=None) -> int:
    """Failure-path tests only: set the kernels' wait limit (microseconds,
    0 = default) and test hooks for every later call; (0, 0) clears them."""
    return lib().attn_debug_set_hooks(wait_limit_us, hooks, _stream(stream))


def prefill(Q, K, V, causal: bool, scale: float | None = None, out_dtype=None, O=None,
            lse=None, want_lse: bool = True, q_scale=None, k_scale=None, v_scale=None,
            stream=None):
    """O = softmax(scale Q K^T [causal]) V for Q [B,Hq,n_q,d], K/V [B,Hkv,n_kv,d].
    E4M3 inputs take per-head fp32 scales q_scale [B*Hq], k_scale/v_scale
    [B*Hkv] (value = code * scale).  Returns (O, lse) with lse [B,Hq,n_q]
    fp32 (None if want_lse is False)."""
    _cuda(Q, K, V, q_scale, k_scale, v_scale)
    B, Hq, nq, d = Q.shape
    _, Hkv, nkv, _ = K.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype is None:
        out_dtype = torch.bfloat16 if Q.dtype == torch.float8_e4m3fn else Q.dtype
    if O is None:
        O = torch.empty((B, Hq, nq, d), dtype=out_dtype, device=Q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, nq), dtype=torch.float32, device=Q.device)
    _cuda(O, lse)
    st = lib().attn_prefill(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), B, Hq, Hkv, nq, nkv,
                            d, int(bool(causal)), float(scale), _DT[Q.dtype], _DT[O.dtype],
                            _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _stream(stream))
    _check("attn_prefill", st)
    return O, lse


def _host(*ts):
    for t in ts:
        if t is not None:
            if t.is_cuda:
                raise ValueError("tensor must live in host memory")
            if not t.is_contiguous():
                raise ValueError("tensor must be contiguous")


def prefill_from_host(hQ, hK, hV, causal: bool, scale: float | None = None, out_dtype=None,
                      hO=None, hlse=None, want_lse: bool = True, Q=None, K=None, V=None,
                      O=None, lse=None, q_scale=None, k_scale=None, v_scale=None,
                      chunks: int = 0, device=None, stream=None):
    """prefill() for host-resident hQ [B,Hq,n_q,d], hK/hV [B,Hkv,n_kv,d]: the
    copies in and out are overlapped with the attention kernels, chunk by
    chunk of heads.  Host tensors should be pinned.  Device buffers Q, K, V,
    O, lse are allocated on `device` (default: the current one) when not
    given.  Returns (hO, hlse); they are complete once `stream` has been
    synchronised."""
    _host(hQ, hK, hV, hO, hlse)
    B, Hq, nq, d = hQ.shape
    _, Hkv, nkv, _ = hK.shape
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype is None:
        out_dtype = torch.bfloat16 if hQ.dtype == torch.float8_e4m3fn else hQ.dtype
    if hO is None:
        hO = torch.empty((B, Hq, nq, d), dtype=out_dtype, pin_memory=True)
    if hlse is None and want_lse:
        hlse = torch.empty((B, Hq, nq), dtype=torch.float32, pin_memory=True)
    Q = torch.empty(hQ.shape, dtype=hQ.dtype, device=device) if Q is None else Q
    K = torch.empty(hK.shape, dtype=hK.dtype, device=device) if K is None else K
    V = torch.empty(hV.shape, dtype=hV.dtype, device=device) if V is None else V
    O = torch.empty(hO.shape, dtype=hO.dtype, device=device) if O is None else O
    if hlse is not None and lse is None:
        lse = torch.empty(hlse.shape, dtype=torch.float32, device=device)
    _cuda(Q, K, V, O, lse, q_scale, k_scale, v_scale)
    for h, t in ((hQ, Q), (hK, K), (hV, V), (hO, O), (hlse, lse)):
        if (h is None) != (t is None) or (h is not None and (h.shape != t.shape or
                                                               h.dtype != t.dtype)):
            raise ValueError("host and device buffers differ in shape or dtype")
    st = lib().attn_prefill_from_host(
        _ptr(hQ), _ptr(hK), _ptr(hV), _ptr(hO), _ptr(hlse), _ptr(Q), _ptr(K), _ptr(V), _ptr(O),
        _ptr(lse), B, Hq, Hkv, nq, nkv, d, int(bool(causal)), float(scale), _DT[hQ.dtype],
        _DT[hO.dtype], _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), int(chunks),
        _stream(stream))
    _check("attn_prefill_from_host", st)
    return hO, hlse


def prefill_from_host_heads_per_chunk(B, Hq, Hkv, n_q, d, chunks=0, sms=148) -> int:
    """Heads per chunk attn_prefill_from_host uses (host arithmetic only)."""
    return lib().attn_prefill_from_host_heads_per_chunk(B, Hq, Hkv, n_q, d, chunks, sms)


def prefill_paged(Q, Kc, Vc, block_table, seq_lens, max_seq_len: int, causal: bool = True,
                  scale: float | None = None, out_dtype=None, O=None, lse=None,
                  want_lse: bool = True, stream=None):
    """n_q new tokens per sequence (the last n_q of each sequence, already in
    the cache) against the whole block-paged cache [num_blocks,Hkv,bs,d].
    Q [B,Hq,n_q,d]; returns (O [B,Hq,n_q,d], lse [B,Hq,n_q])."""
    _cuda(Q, Kc, Vc, block_table, seq_lens)
    B, Hq, nq, d = Q.shape
    num_blocks, Hkv, bs, _ = Kc.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype is None:
        out_dtype = Q.dtype
    if O is None:
        O = torch.empty((B, Hq, nq, d), dtype=out_dtype, device=Q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, nq), dtype=torch.float32, device=Q.device)
    _cuda(O, lse)
    st = lib().attn_prefill_paged(_ptr(Q), _ptr(Kc), _ptr(Vc), _ptr(block_table),
                                  _ptr(seq_lens), _ptr(O), _ptr(lse), B, Hq, Hkv, nq, d, bs,
                                  block_table.shape[1], num_blocks, int(max_seq_len),
                                  int(bool(causal)), float(scale), _DT[Q.dtype], _DT[O.dtype],
                                  _stream(stream))
    _check("attn_prefill_paged", st)
    return O, lse


def backward(Q, K, V, O, dO, lse, causal: bool, scale: float | None = None, out_dtype=None,
             dQ=None, dK=None, dV=None, workspace=None, stream=None):
    """Gradients (dQ, dK, dV) of O = softmax(scale Q K^T [causal]) V for the
    upstream gradient dO, given the forward's O (16-bit or fp32) and lse."""
    _cuda(Q, K, V, O, dO, lse)
    B, Hq, nq, d = Q.shape
    _, Hkv, nkv, _ = K.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype is None:
        out_dtype = Q.dtype
    dQ = torch.empty(Q.shape, dtype=out_dtype, device=Q.device) if dQ is None else dQ
    dK = torch.empty(K.shape, dtype=out_dtype, device=Q.device) if dK is None else dK
    dV = torch.empty(V.shape, dtype=out_dtype, device=Q.device) if dV is None else dV
    need = int(lib().attn_backward_workspace_bytes(B, Hq, nq))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=Q.device)
    _cuda(dQ, dK, dV, workspace)
    st = lib().attn_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(lse), _ptr(dQ),
                             _ptr(dK), _ptr(dV), B, Hq, Hkv, nq, nkv, d, int(bool(causal)),
                             float(scale), _DT[Q.dtype], _DT[O.dtype], _DT[dQ.dtype],
                             _ptr(workspace), workspace.numel(), _stream(stream))
    _check("attn_backward", st)
    return dQ, dK, dV


def rotate_quantize_e4m3(X, signs=None, rows_per_block: int = 0, stream=None):
    """Rows of X [..., n, d] times diag(signs) H_d (no rotation when signs is
    None), quantised to E4M3 with one scale per block of rows_per_block rows
    of a head (0: one per head; all leading dims but the last two flattened
    into heads).  Returns (codes like X in float8_e4m3fn, scales
    [heads, ceil(n / rows_per_block)] fp32, or [heads] for per-head)."""
    _cuda(X, signs)
    d = X.shape[-1]
    n = X.shape[-2]
    heads = X.numel() // (n * d)
    rpb = n if rows_per_block <= 0 or rows_per_block > n else rows_per_block
    nb = -(-n // rpb)
    codes = torch.empty(X.shape, dtype=torch.float8_e4m3fn, device=X.device)
    scales = torch.empty((heads, nb), dtype=torch.float32, device=X.device)
    ws = torch.empty(heads * nb, dtype=torch.int32, device=X.device)
    st = lib().attn_rotate_quantize_e4m3(_ptr(X), _ptr(signs), _ptr(codes), _ptr(scales),
                                         _ptr(ws), heads, n, d, int(rows_per_block),
                                         _DT[X.dtype], _stream(stream))
    _check("attn_rotate_quantize_e4m3", st)
    return codes, (scales.view(heads) if rows_per_block <= 0 else scales)


def prefill_e4m3_blocks(Q, K, V, causal: bool, q_scale, k_scale, v_scale,
                        scale: float | None = None, out_dtype=torch.bfloat16, O=None, lse=None,
                        want_lse: bool = True, stream=None):
    """prefill() for E4M3 Q [B,Hq,n_q,d], K/V [B,Hkv,n_kv,d] with block-wise
    scales: q_scale [B*Hq, ceil(n_q/128)], k_scale [B*Hkv, ceil(n_kv/128)]
    (one per 128 rows of a head), v_scale [B*Hkv].  Returns (O, lse)."""
    _cuda(Q, K, V, q_scale, k_scale, v_scale)
    B, Hq, nq, d = Q.shape
    _, Hkv, nkv, _ = K.shape
    bq, bk = -(-nq // E4M3_SCALE_BLOCK), -(-nkv // E4M3_SCALE_BLOCK)
    if q_scale.numel() != B * Hq * bq or k_scale.numel() != B * Hkv * bk or \
            v_scale.numel() != B * Hkv:
        raise ValueError("scale arrays do not match the block-wise layout")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty((B, Hq, nq, d), dtype=out_dtype, device=Q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, nq), dtype=torch.float32, device=Q.device)
    _cuda(O, lse)
    st = lib().attn_prefill_e4m3_blocks(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), B, Hq,
                                        Hkv, nq, nkv, d, int(bool(causal)), float(scale),
                                        _DT[O.dtype], _ptr(q_scale), _ptr(k_scale),
                                        _ptr(v_scale), _stream(stream))
    _check("attn_prefill_e4m3_blocks", st)
    return O, lse


def decode_workspace_bytes(num_seqs: int, Hq: int, d: int, max_seq_len: int) -> int:
    return int(lib().attn_decode_workspace_bytes(num_seqs, Hq, d, max_seq_len))


def decode(q, Kc, Vc, block_table, seq_lens, max_seq_len: int, scale: float | None = None,
           k_scale=None, v_scale=None, out_dtype=None, O=None, lse=None, workspace=None,
           want_lse: bool = True, stream=None):
    """One query token per sequence against a paged cache [num_blocks,Hkv,bs,d].
    Returns (O [S,Hq,d], lse [S,Hq])."""
    _cuda(q, Kc, Vc, block_table, seq_lens, k_scale, v_scale)
    S, Hq, d = q.shape
    num_blocks, Hkv, bs, _ = Kc.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype is None:
        out_dtype = q.dtype
    if O is None:
        O = torch.empty((S, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((S, Hq), dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(S, Hq, d, max_seq_len)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _cuda(O, lse, workspace)
    st = lib().attn_decode(_ptr(q), _ptr(Kc), _ptr(Vc), _ptr(block_table), _ptr(seq_lens),
                           _ptr(O), _ptr(lse), S, Hq, Hkv, d, bs, block_table.shape[1],
                           num_blocks, int(max_seq_len), float(scale), _DT[q.dtype],
                           _DT[Kc.dtype], _DT[O.dtype], _ptr(k_scale), _ptr(v_scale),
                           _ptr(workspace), workspace.numel(), _stream(stream))
    _check("attn_decode", st)
    return O, lse


def decode_tokens(q, Kc, Vc, block_table, seq_lens, max_seq_len: int, scale: float | None = None,
                  k_scale=None, v_scale=None, out_dtype=None, O=None, lse=None, workspace=None,
                  want_lse: bool = True, stream=None):
    """n_new new tokens per sequence (its last n_new, already in the cache):
    q [S,Hq,n_new,d] against the paged cache.  Returns (O [S,Hq,n_new,d],
    lse [S,Hq,n_new])."""
    _cuda(q, Kc, Vc, block_table, seq_lens, k_scale, v_scale)
    S, Hq, T, d = q.shape
    num_blocks, Hkv, bs, _ = Kc.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out_dtype is None:
        out_dtype = q.dtype
    if O is None:
        O = torch.empty((S, Hq, T, d), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((S, Hq, T), dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(S * T, Hq, d, max_seq_len)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _cuda(O, lse, workspace)
    st = lib().attn_decode_tokens(_ptr(q), _ptr(Kc), _ptr(Vc), _ptr(block_table),
                                  _ptr(seq_lens), _ptr(O), _ptr(lse), S, T, Hq, Hkv, d, bs,
                                  block_table.shape[1], num_blocks, int(max_seq_len),
                                  float(scale), _DT[q.dtype], _DT[Kc.dtype], _DT[O.dtype],
                                  _ptr(k_scale), _ptr(v_scale), _ptr(workspace),
                                  workspace.numel(), _stream(stream))
    _check("attn_decode_tokens", st)
    return O, lse


def kv_append(k_new, v_new, Kc, Vc, block_table, seq_ids, positions, k_scale=None,
              v_scale=None, stream=None):
    """Write k_new/v_new [T,Hkv,d] into the paged caches in place."""
    _cuda(k_new, v_new, Kc, Vc, block_table, seq_ids, positions, k_scale, v_scale)
    T, Hkv, d = k_new.shape
    num_blocks, _, bs, _ = Kc.shape
    st = lib().attn_kv_append(_ptr(k_new), _ptr(v_new), _ptr(Kc), _ptr(Vc), _ptr(block_table),
                              _ptr(seq_ids), _ptr(positions), T, block_table.shape[0], Hkv, d,
                              bs, block_table.shape[1], num_blocks, _DT[k_new.dtype],
                              _DT[Kc.dtype], _ptr(k_scale), _ptr(v_scale), _stream(stream))
    _check("attn_kv_append", st)
