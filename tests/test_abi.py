"""The C-ABI library loads, exports every symbol include/attn.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed:
these paths return before any CUDA call)."""
import ctypes
import os
import re

import pytest

from exact_io_aware_106_b300 import attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from exact_io_aware_106_b300 import build
    build.build()
    return attn.lib()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("attn_prefill", "attn_decode", "attn_kv_append", "attn_decode_workspace_bytes",
              "attn_last_error", "attn_status_str"):
        assert s in syms


def test_library_exports_every_declared_symbol(L):
    for s in declared_symbols():
        assert hasattr(L, s), s
        assert s in attn.EXPORTS


def test_status_strings(L):
    assert attn.status_str(0) == "ATTN_OK"
    assert attn.status_str(4) == "ATTN_ERR_TIMEOUT"
    assert attn.status_str(99) == "ATTN_UNKNOWN_STATUS"


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced by the host checks


def _prefill(L, **kw):
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, lse=None, B=1, Hq=4, Hkv=2, nq=128, nkv=128, d=128,
             causal=1, scale=0.1, ind=1, outd=1, qs=None, ks=None, vs=None)
    a.update(kw)
    return L.attn_prefill(a["Q"], a["K"], a["V"], a["O"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                          a["nq"], a["nkv"], a["d"], a["causal"], a["scale"], a["ind"], a["outd"],
                          a["qs"], a["ks"], a["vs"], None)


def test_prefill_host_validation(L):
    assert _prefill(L, Q=None) == attn.ERR_INVALID
    assert _prefill(L, Hq=3, Hkv=2) == attn.ERR_INVALID
    assert _prefill(L, nq=0) == attn.ERR_INVALID
    assert _prefill(L, nq=200, nkv=100) == attn.ERR_INVALID           # causal, n_q > n_kv
    assert _prefill(L, Q=ctypes.c_void_p((1 << 20) + 8)) == attn.ERR_INVALID  # alignment
    assert _prefill(L, scale=float("nan")) == attn.ERR_INVALID
    assert _prefill(L, d=96) == attn.ERR_UNSUPPORTED
    assert _prefill(L, ind=2) == attn.ERR_UNSUPPORTED                 # fp32 inputs
    assert _prefill(L, outd=3) == attn.ERR_UNSUPPORTED
    assert _prefill(L, ind=3) == attn.ERR_INVALID                     # E4M3 without scales
    assert _prefill(L, ind=3, qs=FAKE, ks=FAKE, vs=None) == attn.ERR_INVALID
    assert L.attn_last_launch_count() == 0


def test_prefill_e4m3_blocks_host_validation(L):
    def call(**kw):
        a = dict(Q=FAKE, B=1, Hq=4, Hkv=2, nq=128, nkv=128, d=128, causal=1, outd=1, qs=FAKE,
                 ks=FAKE, vs=FAKE)
        a.update(kw)
        return L.attn_prefill_e4m3_blocks(a["Q"], FAKE, FAKE, FAKE, None, a["B"], a["Hq"],
                                          a["Hkv"], a["nq"], a["nkv"], a["d"], a["causal"], 0.1,
                                          a["outd"], a["qs"], a["ks"], a["vs"], None)
    assert call(Q=None) == attn.ERR_INVALID
    assert call(qs=None) == attn.ERR_INVALID                          # scales required
    assert call(ks=None) == attn.ERR_INVALID
    assert call(nq=300, nkv=200) == attn.ERR_INVALID                  # causal, n_q > n_kv
    assert call(d=80) == attn.ERR_UNSUPPORTED
    assert call(outd=3) == attn.ERR_UNSUPPORTED                       # E4M3 output
    assert L.attn_last_launch_count() == 0


def test_debug_prefill_timeout_host_validation(L):
    def call(limit=300, d=128, ind=1):
        return L.attn_debug_prefill_timeout(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 128, 128, d,
                                            1, 0.1, ind, 2, limit, None)
    assert call(limit=0) == attn.ERR_INVALID
    assert call(limit=2000000) == attn.ERR_INVALID
    assert call(d=96) == attn.ERR_UNSUPPORTED                          # head sizes 64/128/256
    assert call(ind=3) == attn.ERR_UNSUPPORTED                         # 16-bit inputs only
    assert L.attn_last_launch_count() == 0


def test_debug_set_hooks_host_validation(L):
    assert L.attn_debug_set_hooks(2000000, 0, None) == attn.ERR_INVALID   # limit above 1 s
    assert L.attn_debug_set_hooks(300, 4, None) == attn.ERR_INVALID       # unknown hook bit
    assert L.attn_last_launch_count() == 0


def test_rotate_quantize_host_validation(L):
    def call(**kw):
        a = dict(X=FAKE, heads=2, rows=100, d=128, rpb=128, ind=1)
        a.update(kw)
        return L.attn_rotate_quantize_e4m3(a["X"], None, FAKE, FAKE, FAKE, a["heads"], a["rows"],
                                           a["d"], a["rpb"], a["ind"], None)
    assert call(X=None) == attn.ERR_INVALID
    assert call(rpb=-1) == attn.ERR_INVALID
    assert call(rows=0) == attn.ERR_INVALID
    assert call(d=32) == attn.ERR_UNSUPPORTED
    assert call(ind=3) == attn.ERR_UNSUPPORTED                        # E4M3 input
    assert L.attn_last_launch_count() == 0


def _prefill_paged(L, **kw):
    a = dict(B=2, Hq=4, Hkv=2, nq=64, d=128, bs=16, mb=8, nb=32, msl=128, causal=1, scale=0.1,
             ind=1, outd=1, bt=FAKE)
    a.update(kw)
    return L.attn_prefill_paged(FAKE, FAKE, FAKE, a["bt"], FAKE, FAKE, None, a["B"], a["Hq"],
                                a["Hkv"], a["nq"], a["d"], a["bs"], a["mb"], a["nb"], a["msl"],
                                a["causal"], a["scale"], a["ind"], a["outd"], None)


def test_prefill_paged_host_validation(L):
    assert _prefill_paged(L, bt=None) == attn.ERR_INVALID
    assert _prefill_paged(L, Hq=6, Hkv=4) == attn.ERR_INVALID
    assert _prefill_paged(L, msl=8 * 16 + 1) == attn.ERR_INVALID       # longer than the table
    assert _prefill_paged(L, nq=200) == attn.ERR_INVALID               # causal, n_q > max length
    assert _prefill_paged(L, ind=3) == attn.ERR_UNSUPPORTED            # E4M3 cache
    assert _prefill_paged(L, d=80) == attn.ERR_UNSUPPORTED
    assert _prefill_paged(L, bs=8, msl=64) == attn.ERR_UNSUPPORTED
    assert L.attn_last_launch_count() == 0


def _decode(L, **kw):
    a = dict(S=4, Hq=8, Hkv=2, d=128, bs=16, mb=8, nb=32, msl=128, scale=0.1, qd=1, kvd=1,
             od=1, ks=None, vs=None, ws=FAKE, wsb=1 << 30, bt=FAKE)
    a.update(kw)
    return L.attn_decode(FAKE, FAKE, FAKE, a["bt"], FAKE, FAKE, None, a["S"], a["Hq"], a["Hkv"],
                         a["d"], a["bs"], a["mb"], a["nb"], a["msl"], a["scale"], a["qd"],
                         a["kvd"], a["od"], a["ks"], a["vs"], a["ws"], a["wsb"], None)


def test_decode_host_validation(L):
    assert _decode(L, bt=None) == attn.ERR_INVALID
    assert _decode(L, Hq=6, Hkv=4) == attn.ERR_INVALID
    assert _decode(L, msl=8 * 16 + 1) == attn.ERR_INVALID              # longer than the table
    assert _decode(L, wsb=16) == attn.ERR_INVALID                      # workspace too small
    assert _decode(L, kvd=3, ks=None) == attn.ERR_INVALID              # fp8 without scales
    assert _decode(L, d=80) == attn.ERR_UNSUPPORTED
    assert _decode(L, bs=8, msl=64) == attn.ERR_UNSUPPORTED
    assert _decode(L, Hq=130, Hkv=2) == attn.ERR_UNSUPPORTED           # G > 64
    assert _decode(L, kvd=0) == attn.ERR_UNSUPPORTED                   # f16 cache, bf16 query
    assert _decode(L, ws=ctypes.c_void_p((1 << 20) + 16)) == attn.ERR_INVALID


def test_decode_tokens_host_validation(L):
    def call(**kw):
        a = dict(S=4, T=4, Hq=8, Hkv=2, d=128, msl=128, wsb=1 << 30)
        a.update(kw)
        return L.attn_decode_tokens(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, a["S"], a["T"],
                                    a["Hq"], a["Hkv"], a["d"], 16, 8, 32, a["msl"], 0.1, 1, 1, 1,
                                    None, None, FAKE, a["wsb"], None)
    assert call(T=0) == attn.ERR_INVALID
    assert call(T=17) == attn.ERR_UNSUPPORTED                          # G * T = 68 > 64
    assert call(T=4, msl=3) == attn.ERR_INVALID                        # shorter than its new tokens
    assert call(wsb=1024) == attn.ERR_INVALID                          # workspace too small
    assert L.attn_last_launch_count() == 0


def test_decode_workspace_size_is_monotone(L):
    a = attn.decode_workspace_bytes(64, 32, 128, 32768)
    b = attn.decode_workspace_bytes(64, 32, 128, 1024)
    assert a >= b > 0
    assert attn.decode_workspace_bytes(0, 32, 128, 1024) == 0


def test_kv_append_host_validation(L):
    f = L.attn_kv_append
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 2, 128, 16, 4, 8, 1, 1, None, None,
             None) == attn.OK                                          # nothing to do
    assert f(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3, 2, 2, 128, 16, 4, 8, 1, 1, None, None,
             None) == attn.ERR_INVALID
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3, 2, 2, 128, 16, 4, 8, 1, 3, None, None,
             None) == attn.ERR_INVALID                                 # fp8 without scales
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3, 2, 2, 100, 16, 4, 8, 1, 1, None, None,
             None) == attn.ERR_UNSUPPORTED


def _from_host(L, **kw):
    a = dict(hQ=FAKE, hK=FAKE, hV=FAKE, hO=FAKE, hl=None, Q=FAKE, K=FAKE, V=FAKE, O=FAKE,
             lse=None, B=1, Hq=4, Hkv=2, nq=128, nkv=128, d=128, causal=1, scale=0.1, ind=1,
             outd=1, chunks=0)
    a.update(kw)
    return L.attn_prefill_from_host(a["hQ"], a["hK"], a["hV"], a["hO"], a["hl"], a["Q"], a["K"],
                                    a["V"], a["O"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["nq"],
                                    a["nkv"], a["d"], a["causal"], a["scale"], a["ind"],
                                    a["outd"], None, None, None, a["chunks"], None)


def test_prefill_from_host_validation(L):
    assert _from_host(L, hQ=None) == attn.ERR_INVALID
    assert _from_host(L, hO=None) == attn.ERR_INVALID
    assert _from_host(L, hl=FAKE) == attn.ERR_INVALID          # lse on one side only
    assert _from_host(L, lse=FAKE) == attn.ERR_INVALID
    assert _from_host(L, chunks=-1) == attn.ERR_INVALID
    assert _from_host(L, Q=None) == attn.ERR_INVALID           # the device-side checks
    assert _from_host(L, Hq=3) == attn.ERR_INVALID
    assert _from_host(L, d=96) == attn.ERR_UNSUPPORTED
    assert _from_host(L, ind=3) == attn.ERR_INVALID            # E4M3 without scales
    assert L.attn_last_launch_count() == 0


def _hpc(B, Hq, Hkv, n, d, chunks, sms=148):
    return attn.prefill_from_host_heads_per_chunk(B, Hq, Hkv, n, d, chunks, sms)


def test_prefill_from_host_chunk_plan(L):
    # 64 query heads over 8 KV heads, 32768 rows (128 CTAs per head): 32 chunks
    # of a quarter group by default, whole groups when 8 are asked for
    assert _hpc(1, 64, 8, 32768, 128, 0) == 2
    assert _hpc(1, 64, 8, 32768, 128, 16) == 4
    assert _hpc(1, 64, 8, 32768, 128, 8) == 8
    assert _hpc(1, 64, 8, 32768, 128, 1) == 64
    assert _hpc(1, 64, 8, 32768, 128, 3) == 24          # ceil(8/3) = 3 groups per chunk
    # a small problem (2 CTAs per head) stays in one chunk by default
    assert _hpc(1, 4, 2, 300, 128, 0) == 4
    # 8 query heads of 16 CTAs each (4096 rows): 148 SMs need 10 heads, so one chunk
    assert _hpc(1, 8, 2, 4096, 128, 0) == 8
    # more chunks than groups: the smallest divisor m of G with groups*m >= want
    assert _hpc(1, 12, 1, 4096, 128, 5) == 2            # m = 6
    # never more than 64 chunks
    assert _hpc(40, 2, 1, 4096, 128, 64) == 2           # 80 would be needed: whole groups
    assert _hpc(1, 4, 3, 128, 128, 0) == 0              # Hq % Hkv != 0
    assert _hpc(1, 4, 2, 128, 128, -1) == 0


def test_prefill_from_host_chunk_plan_is_always_valid(L):
    import itertools
    for B, Hkv, G, n, d, want in itertools.product((1, 2, 3), (1, 2, 8), (1, 2, 3, 4, 8, 16),
                                                   (1, 300, 4096, 65536), (64, 128, 256),
                                                   (0, 1, 2, 5, 16, 64, 100)):
        Hq = Hkv * G
        h = _hpc(B, Hq, Hkv, n, d, want)
        assert h >= 1
        assert h % G == 0 or G % h == 0, (B, Hq, Hkv, h)     # whole groups or a part of one
        F = B * Hq
        assert h <= max(F, G) and -(-F // h) <= 64
        if h % G == 0 and h > G:
            assert F % G == 0
