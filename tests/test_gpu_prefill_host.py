"""Prefill from host buffers (attn_prefill_from_host): the chunked,
copy-overlapped path gives exactly the bits of the device-resident prefill
(every chunk is the same kernel on the same data), and the oracle's result
within the usual gates.  Chunk plans cover whole KV-head groups, parts of a
group, several batches, E4M3 inputs, and lse on and off."""
import pytest
import torch

import oracle
from exact_io_aware_106_b300 import attn, workloads as W
from tests.parity import assert_lse, assert_out

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, n_q, n_kv, d, causal, in, out, chunks
    (1, 8, 2, 300, 300, 128, True, "bf16", "bf16", 0),      # one chunk (small)
    (1, 8, 2, 300, 300, 128, True, "bf16", "bf16", 2),      # one group per chunk
    (1, 8, 2, 300, 300, 128, True, "bf16", "f32", 8),       # one head per chunk
    (2, 4, 1, 200, 700, 64, True, "f16", "f16", 4),         # parts of a group, 2 batches
    (3, 6, 3, 129, 129, 128, False, "bf16", "bf16", 5),     # 2 groups per chunk, last has 1
    (1, 4, 2, 257, 257, 256, True, "bf16", "f32", 3),       # d = 256, one head per chunk
    (1, 6, 3, 257, 257, 256, True, "f16", "bf16", 2),       # d = 256, chunks of 4 and 2 heads
]


def _spec(c):
    B, Hq, Hkv, nq, nkv, d, causal, ind, outd, _ = c
    return W.PrefillSpec(B, Hq, Hkv, nq, nkv, d, causal, ind, outd)


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_prefill_from_host_equals_device_prefill_and_oracle(case):
    spec, chunks = _spec(case), case[-1]
    t = W.make_prefill(spec, seed=11)
    hQ, hK, hV = (t[k].pin_memory() for k in ("Q", "K", "V"))
    out = W.DTYPES[spec.out_dtype]
    hO, hlse = attn.prefill_from_host(hQ, hK, hV, spec.causal, out_dtype=out, chunks=chunks)
    torch.cuda.synchronize()
    assert attn.last_error() == attn.OK
    F = spec.B * spec.Hq
    hpc = attn.prefill_from_host_heads_per_chunk(spec.B, spec.Hq, spec.Hkv, spec.n_q, spec.d,
                                                 chunks,
                                                 torch.cuda.get_device_properties(0)
                                                 .multi_processor_count)
    assert attn.last_launch_count() == -(-F // hpc)
    Od, lsed = attn.prefill(hQ.cuda(), hK.cuda(), hV.cuda(), spec.causal, out_dtype=out)
    torch.cuda.synchronize()
    assert torch.equal(hO.view(torch.uint8), Od.cpu().view(torch.uint8))
    assert torch.equal(hlse, lsed.cpu())
    O_ref, lse_ref = oracle.sdpa(t["Q"], t["K"], t["V"], spec.causal)
    assert_out(hO, O_ref)
    assert_lse(hlse, lse_ref)


def test_prefill_from_host_without_lse_and_given_device_buffers():
    spec = W.PrefillSpec(2, 4, 2, 384, 384, 128, True, "bf16", "bf16")
    t = W.make_prefill(spec, seed=12)
    hQ, hK, hV = (t[k].pin_memory() for k in ("Q", "K", "V"))
    dev = {k: torch.full(t[k].shape, float("nan"), dtype=t[k].dtype, device="cuda")
           for k in ("Q", "K", "V")}
    O = torch.empty(t["Q"].shape, dtype=torch.bfloat16, device="cuda")
    hO, hlse = attn.prefill_from_host(hQ, hK, hV, True, want_lse=False, Q=dev["Q"], K=dev["K"],
                                      V=dev["V"], O=O, chunks=4)
    torch.cuda.synchronize()
    assert hlse is None and attn.last_error() == attn.OK
    # the device buffers now hold the inputs and the output
    for k in ("Q", "K", "V"):
        assert torch.equal(dev[k].cpu().view(torch.uint8), t[k].view(torch.uint8))
    assert torch.equal(O.cpu().view(torch.uint8), hO.view(torch.uint8))
    O_ref, _ = oracle.sdpa(t["Q"], t["K"], t["V"], True)
    assert_out(hO, O_ref)


def test_prefill_from_host_e4m3():
    spec = W.PrefillSpec(1, 8, 2, 256, 256, 128, True, "e4m3", "bf16")
    t = W.make_prefill(spec, seed=13)
    kw = W.quantize_prefill_e4m3(t)
    Q8, K8, V8 = kw.pop("Q"), kw.pop("K"), kw.pop("V")
    sc = {k: v.cuda() for k, v in kw.items()}
    hO, hlse = attn.prefill_from_host(Q8.pin_memory(), K8.pin_memory(), V8.pin_memory(), True,
                                      chunks=8, **sc)
    torch.cuda.synchronize()
    assert attn.last_error() == attn.OK
    Od, lsed = attn.prefill(Q8.cuda(), K8.cuda(), V8.cuda(), True, **sc)
    torch.cuda.synchronize()
    assert torch.equal(hO.view(torch.uint8), Od.cpu().view(torch.uint8))
    assert torch.equal(hlse, lsed.cpu())


def test_prefill_from_host_is_ordered_on_the_stream():
    """Back-to-back calls on one stream, each overwriting the previous call's
    device buffers: every call's host output is its own problem's result."""
    spec = W.PrefillSpec(1, 8, 2, 1024, 1024, 128, True, "bf16", "bf16")
    Q = K = V = O = lse = None
    outs, refs = [], []
    for seed in (21, 22, 23):
        t = W.make_prefill(spec, seed=seed)
        hQ, hK, hV = (t[k].pin_memory() for k in ("Q", "K", "V"))
        if Q is None:
            Q, K, V = (torch.empty(x.shape, dtype=x.dtype, device="cuda") for x in (hQ, hK, hV))
            O = torch.empty(hQ.shape, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(hQ.shape[:3], dtype=torch.float32, device="cuda")
        outs.append(attn.prefill_from_host(hQ, hK, hV, True, Q=Q, K=K, V=V, O=O, lse=lse,
                                           chunks=8))
        refs.append(t)
    torch.cuda.synchronize()
    assert attn.last_error() == attn.OK
    for (hO, hlse), t in zip(outs, refs):
        Od, lsed = attn.prefill(t["Q"].cuda(), t["K"].cuda(), t["V"].cuda(), True)
        torch.cuda.synchronize()
        assert torch.equal(hO.view(torch.uint8), Od.cpu().view(torch.uint8))
        assert torch.equal(hlse, lsed.cpu())
    O_ref, lse_ref = oracle.sdpa(refs[-1]["Q"], refs[-1]["K"], refs[-1]["V"], True)
    assert_out(outs[-1][0], O_ref)
    assert_lse(outs[-1][1], lse_ref)
