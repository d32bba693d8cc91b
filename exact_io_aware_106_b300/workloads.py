"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and lays them out; it contains none of
the attention arithmetic, so both the CUDA path and the fp64 oracle can be
fed from it.  Values are iid N(0,1) drawn in fp32 and cast once (round to
nearest even) to the storage type.  Generation on a CUDA device uses the
device generator (Philox), generation on the host uses the CPU generator, so
the same seed gives different values on the two; the structure (sequence
lengths, block table) is always drawn on the host and is identical.

Workload shapes (sizes as given for each workload):
  single-head:   B=1, H=1, n=512, d=64, fp16, non-causal, fp32 output
  gqa-4k:        B=4, Hq=32, Hkv=8, d=128, n=4096, bf16, causal
  long-23k:      B=1, H=12 (MHA), d=64, n=23400, fp16, causal
  long-32k:      B=1, Hq=64, Hkv=8, d=128, n=32768, bf16, causal
  paged-decode:  64 sequences, Hq=32, Hkv=8, d=128, lengths U[1024, 32768],
                 bf16 cache in 16-token blocks, block table = a seeded random
                 permutation of the blocks dealt to the sequences in order
  sweep:         decode batch 32 x KVSL 8192 and prefill B=1 ISL 8192, Hkv=8,
                 Hq=8G for G in {1,4,8,16}, d in {64,128,256}, bf16 or
                 fp8-E4M3 KV with per-head scale amax/448
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
          "e4m3": torch.float8_e4m3fn}


@dataclass(frozen=True)
class PrefillSpec:
    B: int
    Hq: int
    Hkv: int
    n_q: int
    n_kv: int
    d: int
    causal: bool
    dtype: str = "bf16"
    out_dtype: str = "bf16"
    name: str = ""


@dataclass(frozen=True)
class DecodeSpec:
    num_seqs: int
    Hq: int
    Hkv: int
    d: int
    len_lo: int
    len_hi: int
    block_size: int = 16
    q_dtype: str = "bf16"
    kv_dtype: str = "bf16"
    out_dtype: str = "bf16"
    name: str = ""


@dataclass(frozen=True)
class PagedPrefillSpec:
    """n_q new query tokens per sequence attending to the sequence's whole
    block-paged cache (prefix + the new tokens, length U[len_lo, len_hi])."""
    B: int
    Hq: int
    Hkv: int
    n_q: int
    d: int
    len_lo: int
    len_hi: int
    block_size: int = 16
    causal: bool = True
    dtype: str = "bf16"
    out_dtype: str = "bf16"
    name: str = ""


PREFILL_WORKLOADS = {
    "single-head": PrefillSpec(1, 1, 1, 512, 512, 64, False, "f16", "f32", "single-head"),
    "gqa-4k": PrefillSpec(4, 32, 8, 4096, 4096, 128, True, "bf16", "bf16", "gqa-4k"),
    "long-23k": PrefillSpec(1, 12, 12, 23400, 23400, 64, True, "f16", "f16", "long-23k"),
    "long-32k": PrefillSpec(1, 64, 8, 32768, 32768, 128, True, "bf16", "bf16", "long-32k"),
}

PAGED_PREFILL_WORKLOADS = {
    # chunked prefill over cached prefixes: 8 sequences x 1024 new tokens,
    # total lengths U[4096, 16384], GQA 32/8, d 128, bf16, 16-token blocks
    "paged-prefill": PagedPrefillSpec(8, 32, 8, 1024, 128, 4096, 16384, 16, True, "bf16", "bf16",
                                      "paged-prefill"),
}

# multi-token decode: the paged-decode workload with 4 new tokens per
# sequence (e.g. speculative drafts), G * 4 = 16 query rows per KV head
DECODE_TOKENS_WORKLOADS = {
    "spec-decode-4": (4, None),
    # 8 new tokens: G * 8 = 32 query rows per KV head, two 16-row tiles
    "spec-decode-8": (8, None),
}

DECODE_WORKLOADS = {
    "paged-decode": DecodeSpec(64, 32, 8, 128, 1024, 32768, 16, "bf16", "bf16", "bf16",
                               "paged-decode"),
}


def sweep_prefill(G: int, d: int, kv: str = "bf16") -> PrefillSpec:
    """kv: "bf16", "e4m3" (one scale per head) or "e4m3b" (E4M3 with Q / K
    scales per 128-row block, the block-wise form; values drawn as bf16)."""
    return PrefillSpec(1, 8 * G, 8, 8192, 8192, d, True, kv, "bf16",
                       f"sweep-prefill-G{G}-d{d}-{kv}")


def sweep_decode(G: int, d: int, kv: str = "bf16") -> DecodeSpec:
    return DecodeSpec(32, 8 * G, 8, d, 8192, 8192, 16, "bf16", kv, "bf16",
                      f"sweep-decode-G{G}-d{d}-{kv}")


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, dtype, g, device):
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(dtype)


def make_prefill(spec: PrefillSpec, seed: int = 0, device="cpu"):
    """Q [B,Hq,n_q,d], K/V [B,Hkv,n_kv,d] in the spec's storage type, drawn in
    the order Q, K, V from one generator."""
    g = _gen(device, seed)
    dt = DTYPES["bf16" if spec.dtype.startswith("e4m3") else spec.dtype]
    Q = _randn((spec.B, spec.Hq, spec.n_q, spec.d), dt, g, device)
    K = _randn((spec.B, spec.Hkv, spec.n_kv, spec.d), dt, g, device)
    V = _randn((spec.B, spec.Hkv, spec.n_kv, spec.d), dt, g, device)
    return {"Q": Q, "K": K, "V": V}


def make_seq_structure(num_seqs, len_lo, len_hi, block_size, seed, extra_blocks=0,
                       lens=None):
    """Sequence lengths ~ U{len_lo..len_hi} and a block table dealing a
    seeded random permutation of the physical blocks to the sequences in
    order.  The table is wide enough for len_hi tokens per sequence; unused
    entries are -1.  Always drawn on the host."""
    g = _gen("cpu", seed + 7919)
    if lens is None:
        lens = torch.randint(len_lo, len_hi + 1, (num_seqs,), generator=g, dtype=torch.int64)
    else:
        lens = torch.as_tensor(lens, dtype=torch.int64)
    nblk = (lens + block_size - 1) // block_size
    num_blocks = int(nblk.sum()) + extra_blocks
    max_blocks = max(1, (len_hi + block_size - 1) // block_size,
                     int(nblk.max()) if num_seqs else 1)
    perm = torch.randperm(max(num_blocks, 1), generator=g, dtype=torch.int64)[:num_blocks]
    table = torch.full((num_seqs, max_blocks), -1, dtype=torch.int32)
    off = 0
    for s in range(num_seqs):
        k = int(nblk[s])
        table[s, :k] = perm[off:off + k].to(torch.int32)
        off += k
    return lens.to(torch.int32), table, max(num_blocks, 1)


def quantize_e4m3_per_head(x: torch.Tensor, head_dim: int = 1):
    """Storage conversion of an N(0,1) cache to fp8-E4M3 with one fp32 scale
    per KV head: scale = amax/448 over that head's values, codes =
    torch's round-to-nearest cast of x/scale.  Input preparation only."""
    xf = x.float()
    dims = [i for i in range(xf.dim()) if i != head_dim]
    amax = xf.abs().amax(dim=dims)
    scale = (amax / 448.0).to(torch.float32)
    shape = [1] * xf.dim()
    shape[head_dim] = -1
    codes = (xf / scale.view(shape)).to(torch.float8_e4m3fn)
    return codes, scale


def make_decode(spec: DecodeSpec, seed: int = 0, device="cpu", lens=None,
                keep_unquantised: bool = False, extra_blocks: int = 0):
    """q [S,Hq,d]; K/V cache [num_blocks,Hkv,block_size,d]; block_table
    [S,max_blocks] int32; seq_lens [S] int32; per-head scales for E4M3."""
    lens_t, table, num_blocks = make_seq_structure(spec.num_seqs, spec.len_lo, spec.len_hi,
                                                   spec.block_size, seed, extra_blocks, lens)
    g = _gen(device, seed)
    qdt = DTYPES[spec.q_dtype]
    q = _randn((spec.num_seqs, spec.Hq, spec.d), qdt, g, device)
    store = torch.bfloat16 if spec.kv_dtype == "e4m3" else DTYPES[spec.kv_dtype]
    Kc = _randn((num_blocks, spec.Hkv, spec.block_size, spec.d), store, g, device)
    Vc = _randn((num_blocks, spec.Hkv, spec.block_size, spec.d), store, g, device)
    out = {"q": q, "block_table": table.to(device), "seq_lens": lens_t.to(device),
           "num_blocks": num_blocks, "k_scale": None, "v_scale": None}
    if spec.kv_dtype == "e4m3":
        kq, ks = quantize_e4m3_per_head(Kc, 1)
        vq, vs = quantize_e4m3_per_head(Vc, 1)
        out.update(Kc=kq, Vc=vq, k_scale=ks, v_scale=vs)
        if keep_unquantised:
            out.update(Kc_src=Kc, Vc_src=Vc)
    else:
        out.update(Kc=Kc, Vc=Vc)
    return out


def make_append(T: int, Hkv: int, d: int, dtype: str, seed: int = 0, device="cpu"):
    """New K/V rows [T,Hkv,d] for a cache append."""
    g = _gen(device, seed + 31)
    dt = DTYPES[dtype]
    return _randn((T, Hkv, d), dt, g, device), _randn((T, Hkv, d), dt, g, device)


def quantize_prefill_e4m3(t: dict) -> dict:
    """Storage conversion of prefill inputs to fp8-E4M3 with one fp32 scale
    per head of each tensor (amax/448, the same rule as the cache): returns
    Q, K, V codes and q_scale [B*Hq], k_scale, v_scale [B*Hkv].  Input
    preparation only."""
    out = {}
    for name in ("Q", "K", "V"):
        x = t[name]
        B, H = x.shape[:2]
        codes, scale = quantize_e4m3_per_head(x.reshape(B * H, *x.shape[2:]), 0)
        out[name] = codes.reshape(x.shape)
        out[name.lower() + "_scale"] = scale
    return out


def make_paged_prefill(spec: PagedPrefillSpec, seed: int = 0, device="cpu", lens=None):
    """Q [B,Hq,n_q,d]; K/V cache [num_blocks,Hkv,block_size,d] holding every
    sequence's tokens (the new ones last); block_table, seq_lens as for
    decode."""
    lens_t, table, num_blocks = make_seq_structure(spec.B, spec.len_lo, spec.len_hi,
                                                   spec.block_size, seed, 0, lens)
    g = _gen(device, seed)
    dt = DTYPES[spec.dtype]
    Q = _randn((spec.B, spec.Hq, spec.n_q, spec.d), dt, g, device)
    Kc = _randn((num_blocks, spec.Hkv, spec.block_size, spec.d), dt, g, device)
    Vc = _randn((num_blocks, spec.Hkv, spec.block_size, spec.d), dt, g, device)
    return {"Q": Q, "Kc": Kc, "Vc": Vc, "block_table": table.to(device),
            "seq_lens": lens_t.to(device), "num_blocks": num_blocks}


def make_backward(spec: PrefillSpec, seed: int = 0, device="cpu"):
    """Forward inputs (as make_prefill) plus an upstream gradient dO
    [B,Hq,n_q,d] iid N(0,1), drawn after V from the same generator."""
    g = _gen(device, seed)
    dt = DTYPES[spec.dtype]
    Q = _randn((spec.B, spec.Hq, spec.n_q, spec.d), dt, g, device)
    K = _randn((spec.B, spec.Hkv, spec.n_kv, spec.d), dt, g, device)
    V = _randn((spec.B, spec.Hkv, spec.n_kv, spec.d), dt, g, device)
    dO = _randn((spec.B, spec.Hq, spec.n_q, spec.d), dt, g, device)
    return {"Q": Q, "K": K, "V": V, "dO": dO}
