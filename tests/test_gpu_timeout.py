"""The bounded-wait failure path on the GPU, made to happen in the allowed
form: attn_debug_prefill_timeout shortens every wait's limit to a few
hundred microseconds and has the prefill's producer withhold its Q copy, so
the MMA issuer's first wait runs out.  The call must return, the error word
must read ATTN_ERR_TIMEOUT, the CTA's rows must be O = 0 / lse = NaN, and the
next ordinary call on the same stream must match the oracle (tensor memory
was freed, nothing was left behind)."""
import time

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_106_b300 import attn, workloads as W
from tests.parity import assert_lse, assert_out

pytestmark = pytest.mark.gpu


def _p(t):
    import ctypes
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("d", [64, 128, 256])
def test_expired_wait_is_reported_and_the_device_stays_usable(d):
    spec = W.PrefillSpec(1, 1, 1, 128, 128, d, True, "bf16", "f32")
    t = W.make_prefill(spec, seed=31 + d)
    Q, K, V = (t[n].cuda() for n in "QKV")
    O = torch.full((1, 1, 128, d), float("nan"), device="cuda")
    lse = torch.zeros((1, 1, 128), device="cuda")
    assert attn.last_error() == attn.OK
    stream = torch.cuda.current_stream()
    import ctypes
    t0 = time.perf_counter()
    st = attn.lib().attn_debug_prefill_timeout(
        _p(Q), _p(K), _p(V), _p(O), _p(lse), 1, 1, 1, 128, 128, d, 1, 1.0 / np.sqrt(d),
        1, 2, 300, ctypes.c_void_p(stream.cuda_stream))
    wall = time.perf_counter() - t0
    assert st == attn.OK, attn.status_str(st)
    assert attn.last_error() == attn.ERR_TIMEOUT
    assert (O == 0).all()
    assert torch.isnan(lse).all()
    assert wall < 1.0, wall  # the short limit, not the 2 s default, was used
    assert attn.last_error() == attn.OK  # cleared by the read
    # the next ordinary call on the same stream matches the oracle
    O2, lse2 = attn.prefill(Q, K, V, True, out_dtype=torch.float32)
    assert attn.last_error() == attn.OK
    O_ref, lse_ref = oracle.sdpa(t["Q"], t["K"], t["V"], True)
    assert_out(O2, O_ref)
    assert_lse(lse2, lse_ref)


@pytest.mark.parametrize("d,kv", [(128, "bf16"), (64, "e4m3")])
def test_expired_decode_wait_is_reported_and_the_device_stays_usable(d, kv):
    # the decode split kernel's producer issues no copy, so its consumers'
    # first wait runs out; the split partials are marked unusable and the
    # combine writes O = 0, lse = NaN
    lens = [1, 300, 2500]
    spec = W.DecodeSpec(3, 8, 2, d, 1, max(lens), 16, "bf16", kv, "bf16")
    t = W.make_decode(spec, seed=5, lens=lens)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    kw = {}
    if kv == "e4m3":
        kw = dict(k_scale=g["k_scale"], v_scale=g["v_scale"])
    assert attn.last_error() == attn.OK
    assert attn.debug_set_hooks(300, attn.HOOK_WITHHOLD_KV) == attn.OK
    try:
        t0 = time.perf_counter()
        O, lse = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                             max_seq_len=max(lens), out_dtype=torch.float32, **kw)
        status = attn.last_error()
        wall = time.perf_counter() - t0
    finally:
        assert attn.debug_set_hooks(0, 0) == attn.OK
    assert status == attn.ERR_TIMEOUT
    assert (O == 0).all()
    assert torch.isnan(lse).all()
    assert wall < 1.0, wall
    # the next ordinary call matches the oracle
    O2, lse2 = attn.decode(g["q"], g["Kc"], g["Vc"], g["block_table"], g["seq_lens"],
                           max_seq_len=max(lens), out_dtype=torch.float32, **kw)
    assert attn.last_error() == attn.OK
    O_ref, lse_ref = oracle.decode_paged(t["q"], t["Kc"], t["Vc"], t["block_table"],
                                         t["seq_lens"], k_scale=t.get("k_scale"),
                                         v_scale=t.get("v_scale"))
    assert_out(O2, O_ref)  # E4M3: against the oracle fed the dequantised cache
    assert_lse(lse2, lse_ref)
