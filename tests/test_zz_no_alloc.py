"""attn_decode_static_ws: decode for callers that may not allocate device
memory (a host framework that owns every allocation, or a latency-critical
thread that cannot pay for cudaMalloc).  It keeps its split-KV scratch in an
array compiled into the library, so these tests check that its results match
attn_decode with a caller-provided workspace, on two calls in a row (the
second call finds the first call's leftovers in the shared array), and that
sizes beyond the array are refused before anything runs.

This file is collected last on purpose: a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_106_b300 import attn, workloads as W
from tests.parity import assert_lse, assert_out

_DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2, torch.float8_e4m3fn: 3}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _static_ws_decode(g, max_seq_len, out_dtype):
    """Call the C entry point directly with device pointers (no workspace)."""
    S, Hq, d = g["q"].shape
    num_blocks, Hkv, bs, _ = g["Kc"].shape
    O = torch.empty((S, Hq, d), dtype=out_dtype, device="cuda")
    lse = torch.empty((S, Hq), dtype=torch.float32, device="cuda")
    st = attn.lib().attn_decode_static_ws(
        _p(g["q"]), _p(g["Kc"]), _p(g["Vc"]), _p(g["block_table"]), _p(g["seq_lens"]), _p(O),
        _p(lse), S, Hq, Hkv, d, bs, g["block_table"].shape[1], num_blocks, max_seq_len,
        1.0 / np.sqrt(d), _DT[g["q"].dtype], _DT[g["Kc"].dtype], _DT[out_dtype],
        _p(g["k_scale"]), _p(g["v_scale"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, O, lse


@pytest.mark.gpu
def test_static_ws_decode_matches_workspace_decode_twice():
    calls = [
        (W.DecodeSpec(6, 16, 4, 128, 1, 3000, 16, "bf16", "bf16", "f32"),
         [3000, 1, 17, 2048, 999, 64], 11),
        (W.DecodeSpec(4, 8, 2, 64, 1, 5000, 32, "bf16", "bf16", "bf16"),
         [5000, 33, 4096, 2], 12),
    ]
    for spec, lens, seed in calls:  # two calls in a row share the scratch array
        t = W.make_decode(spec, seed=seed, lens=lens)
        g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
        out_dt = W.DTYPES[spec.out_dtype]
        st, O, lse = _static_ws_decode(g, spec.len_hi, out_dt)
        assert st == attn.OK, attn.status_str(st)
        assert attn.last_launch_count() == 2
        assert attn.last_error() == attn.OK
        O_ref, lse_ref = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"],
                                     g["seq_lens"], max_seq_len=spec.len_hi, out_dtype=out_dt)
        assert attn.last_error() == attn.OK
        assert_out(O, O_ref.double().cpu().numpy(), what="static-ws O")
        assert_lse(lse, lse_ref.double().cpu().numpy(), what="static-ws lse")
        # and against the fp64 oracle directly
        O_or, lse_or = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                           t["seq_lens"])
        assert_out(O, O_or, what="static-ws O vs oracle")
        assert_lse(lse, lse_or, what="static-ws lse vs oracle")


@pytest.mark.gpu
def test_static_ws_decode_allocates_no_device_memory():
    """The entry point's promise: once its kernels are loaded (a first call),
    a call leaves the device's free memory exactly where it was."""
    spec = W.DecodeSpec(5, 16, 4, 128, 1, 4000, 16, "bf16", "bf16", "bf16")
    t = W.make_decode(spec, seed=13, lens=[4000, 7, 1234, 16, 2500])
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    st, O, lse = _static_ws_decode(g, spec.len_hi, torch.bfloat16)  # loads the kernels
    assert st == attn.OK
    torch.cuda.synchronize()
    S, Hq, d = g["q"].shape
    num_blocks, Hkv, bs, _ = g["Kc"].shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        st = attn.lib().attn_decode_static_ws(
            _p(g["q"]), _p(g["Kc"]), _p(g["Vc"]), _p(g["block_table"]), _p(g["seq_lens"]),
            _p(O), _p(lse), S, Hq, Hkv, d, bs, g["block_table"].shape[1], num_blocks,
            spec.len_hi, 1.0 / np.sqrt(d), 1, 1, 1, None, None, stream)
        assert st == attn.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert attn.last_error() == attn.OK


def test_static_ws_decode_refuses_sizes_beyond_its_scratch():
    """64 sequences x 32 heads x d=128 up to 32768 tokens need ~32 MiB of
    split-KV scratch, more than the 16 MiB compiled in: refused on the host,
    before any CUDA call (fake pointers are never dereferenced)."""
    from exact_io_aware_106_b300 import build
    build.build()
    need = attn.decode_workspace_bytes(64, 32, 128, 32768)
    assert need > attn.DECODE_STATIC_WS_BYTES
    fake = ctypes.c_void_p(1 << 20)
    st = attn.lib().attn_decode_static_ws(fake, fake, fake, fake, fake, fake, None, 64, 32, 8,
                                          128, 16, 2048, 70000, 32768, 0.1, 1, 1, 1, None, None,
                                          None)
    assert st == attn.ERR_UNSUPPORTED
    assert attn.last_launch_count() == 0
