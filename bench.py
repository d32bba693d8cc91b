#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path on B300.

One step = one pass of the whole path over one batch of synthetic input:
  1. prefill: causal GQA attention, B=1, 64 query / 8 KV heads, d=128,
     n = 32768, bf16 (the long-context workload the prefill target is quoted
     on);
  2. KV append: one new token per sequence written into the paged cache;
  3. decode: one query token for each of 64 sequences (32 query / 8 KV heads,
     d=128, lengths U[1024, 32768]) over the bf16 cache in 16-token blocks.

Metric (as quoted): prefill attention TFLOP/s and decode KV GB/s, as % of
the roofline.  `value` is the step's roofline time -- sum over its kernels of
max(F/compute peak, B/HBM bandwidth), with algorithmic F and B -- divided by
the measured step time, in percent; with N replica GPUs it is the sum over
ranks of their roofline time over the slowest rank's time (weak scaling).
The line also carries each part's absolute TFLOP/s or GB/s and fraction.

Inputs are generated on the device before timing and are larger than L2 (the
prefill reads 640 MB, the decode 4.4 GB), so no L2 flush is needed between
steps.  Timing: CUDA events on the launching stream, W warm-up steps, then K
timed steps bracketed by barrier + synchronize; max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_io_aware_106_b300 import workloads as W  # noqa: E402

PREFILL = W.PREFILL_WORKLOADS["long-32k"]
DECODE = W.DECODE_WORKLOADS["paged-decode"]
METRIC = "prefill attn TFLOP/s & decode KV GB/s on 1 B300, as % of roofline"
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
ESZ = {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1, "e4m3b": 1}


# --------------------------------------------------------------- roofline

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]), "source": "measured"}
    return dict(FALLBACK, source="fallback")


def prefill_pairs(spec) -> int:
    """Unmasked (query, key) pairs summed over (batch, query head)."""
    if not spec.causal:
        per_head = spec.n_q * spec.n_kv
    else:
        off = spec.n_kv - spec.n_q
        per_head = sum(min(spec.n_kv, i + off + 1) for i in range(spec.n_q))
    return per_head * spec.B * spec.Hq


def prefill_flops(spec) -> float:
    """F = 4 d pairs: two GEMMs (QK^T and PV) at 2 flops per multiply-add."""
    return 4.0 * spec.d * prefill_pairs(spec)


def prefill_bytes(spec) -> float:
    """Q, K, V read once and O, lse written once (K/V once per KV head)."""
    e = ESZ[spec.dtype]
    q = spec.B * spec.Hq * spec.n_q * spec.d * e
    kv = 2 * spec.B * spec.Hkv * spec.n_kv * spec.d * e
    o = spec.B * spec.Hq * spec.n_q * spec.d * ESZ[spec.out_dtype]
    return float(q + kv + o + 4 * spec.B * spec.Hq * spec.n_q)


def decode_bytes(spec, lens) -> float:
    """K and V of every visible token once per KV head, plus q, O, lse and
    the block-table entries read."""
    tot = int(sum(int(x) for x in lens))
    blocks = int(sum((int(x) + spec.block_size - 1) // spec.block_size for x in lens))
    kv = 2 * tot * spec.Hkv * spec.d * ESZ[spec.kv_dtype]
    q = spec.num_seqs * spec.Hq * spec.d * ESZ[spec.q_dtype]
    o = spec.num_seqs * spec.Hq * spec.d * ESZ[spec.out_dtype]
    return float(kv + q + o + 4 * spec.num_seqs * spec.Hq + 4 * blocks + 4 * spec.num_seqs)


def decode_flops(spec, lens) -> float:
    return 4.0 * spec.Hq * spec.d * float(sum(int(x) for x in lens))


def append_bytes(spec) -> float:
    T = spec.num_seqs
    return float(2 * T * spec.Hkv * spec.d * (ESZ[spec.q_dtype] + ESZ[spec.kv_dtype]) + 12 * T)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled during timing."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(self.dev)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.strip()]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def _src_sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def measured_traffic(kernel_file: str, workload: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    table profiles/traffic.txt, if the kernel source is unchanged since the
    counters were taken; else None.  Each line of the table:
    `<workload> <kernel source file> <source sha256[:16]> <bytes per launch>`."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    src = os.path.join(ROOT, "exact_io_aware_106_b300", "csrc", kernel_file)
    sha = _src_sha(src)
    for ln in open(p):
        f = ln.split()
        if len(f) == 4 and not ln.startswith("#") and f[0] == workload and f[1] == kernel_file \
                and f[2] == sha:
            return float(f[3])
    return None


def run_ours(args, rank, world):
    from exact_io_aware_106_b300 import attn

    global PREFILL, DECODE
    if args.prefill_n:
        PREFILL = W.PrefillSpec(PREFILL.B, PREFILL.Hq, PREFILL.Hkv, args.prefill_n, args.prefill_n,
                                PREFILL.d, PREFILL.causal, PREFILL.dtype, PREFILL.out_dtype,
                                PREFILL.name + f"-n{args.prefill_n}")
    if args.decode_seqs:
        DECODE = W.DecodeSpec(args.decode_seqs, DECODE.Hq, DECODE.Hkv, DECODE.d, DECODE.len_lo,
                              DECODE.len_hi, DECODE.block_size, DECODE.q_dtype, DECODE.kv_dtype,
                              DECODE.out_dtype, DECODE.name + f"-S{args.decode_seqs}")
    do_pre = args.only in ("step", "prefill")
    do_dec = args.only in ("step", "decode")
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pk = peaks()
    seed = 1000 * rank

    # ---- inputs resident in HBM before timing
    Q = K = V = O = lse = None
    if do_pre:
        pin = W.make_prefill(PREFILL, seed=seed, device=dev)
        Q, K, V = pin["Q"], pin["K"], pin["V"]
        O = torch.empty_like(Q)
        lse = torch.empty(Q.shape[:3], dtype=torch.float32, device=dev)
    S = DECODE.num_seqs
    if do_dec:
        dd = W.make_decode(DECODE, seed=seed, device=dev)
        lens = dd["seq_lens"].cpu()
        k_new, v_new = W.make_append(S, DECODE.Hkv, DECODE.d, DECODE.q_dtype, seed=seed,
                                     device=dev)
        seq_ids = torch.arange(S, dtype=torch.int32, device=dev)
        positions = (dd["seq_lens"] - 1).to(torch.int32)  # the newest token's slot
        Od = torch.empty((S, DECODE.Hq, DECODE.d), dtype=W.DTYPES[DECODE.out_dtype],
                         device=dev)
        lsed = torch.empty((S, DECODE.Hq), dtype=torch.float32, device=dev)
        ws = torch.empty(attn.decode_workspace_bytes(S, DECODE.Hq, DECODE.d, DECODE.len_hi),
                         dtype=torch.uint8, device=dev)
    else:
        lens = torch.zeros(S, dtype=torch.int32)
    stream = torch.cuda.current_stream(dev)

    launches = [0]

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        if do_pre:
            attn.prefill(Q, K, V, True, O=O, lse=lse, stream=stream)
            launches[0] += attn.last_launch_count()
        if ev:
            ev[1].record(stream)
        if do_dec:
            attn.kv_append(k_new, v_new, dd["Kc"], dd["Vc"], dd["block_table"], seq_ids,
                           positions, stream=stream)
            launches[0] += attn.last_launch_count()
        if ev:
            ev[2].record(stream)
        if do_dec:
            attn.decode(dd["q"], dd["Kc"], dd["Vc"], dd["block_table"], dd["seq_lens"],
                        max_seq_len=DECODE.len_hi, O=Od, lse=lsed, workspace=ws, stream=stream)
            launches[0] += attn.last_launch_count()
        if ev:
            ev[3].record(stream)

    # first call of each part, host wall time with synchronisation on both
    # sides: lazy module load, tensor-map encoding and the run itself
    first = {}
    torch.cuda.synchronize(dev)
    if do_pre:
        t0 = time.perf_counter()
        attn.prefill(Q, K, V, True, O=O, lse=lse, stream=stream)
        torch.cuda.synchronize(dev)
        first["prefill_ms"] = round((time.perf_counter() - t0) * 1e3, 3)
    if do_dec:
        t0 = time.perf_counter()
        attn.decode(dd["q"], dd["Kc"], dd["Vc"], dd["block_table"], dd["seq_lens"],
                    max_seq_len=DECODE.len_hi, O=Od, lse=lsed, workspace=ws, stream=stream)
        torch.cuda.synchronize(dev)
        first["decode_ms"] = round((time.perf_counter() - t0) * 1e3, 3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if attn.last_error(stream) != attn.OK:
        raise RuntimeError("device error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    launches[0] = 0
    with ClockSampler(dev.index) as clk:
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(evs[i])
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    n_launch = launches[0]
    if attn.last_error(stream) != attn.OK:
        raise RuntimeError("device error during the timed steps")
    per_pre = [e[0].elapsed_time(e[1]) for e in evs]
    per_dec = [e[2].elapsed_time(e[3]) for e in evs]
    t_pre = sum(per_pre) / 1e3
    t_app = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    t_dec = sum(per_dec) / 1e3
    t_step = sum(e[0].elapsed_time(e[3]) for e in evs) / 1e3

    F = prefill_flops(PREFILL)
    Bp = prefill_bytes(PREFILL)
    Bd = decode_bytes(DECODE, lens)
    Ba = append_bytes(DECODE)
    # the dense bf16 peak as a burst: the timed region is well under a second,
    # far shorter than the seconds-long loop the sustained figure comes from
    P = pk["bf16_tflops"] * 1e12
    BW = pk["hbm_gbs"] * 1e9
    roof_pre = max(F / P, Bp / BW) if do_pre else 0.0
    roof_dec = max(decode_flops(DECODE, lens) / P, Bd / BW) if do_dec else 0.0
    roof_app = Ba / BW if do_dec else 0.0
    roof_step = roof_pre + roof_app + roof_dec
    nst = args.steps
    res = {
        "t_step": t_step / nst, "t_pre": t_pre / nst, "t_dec": t_dec / nst,
        "t_app": t_app / nst,
        "roof_step": roof_step, "roof_pre": roof_pre, "roof_dec": roof_dec, "F": F, "Bd": Bd,
        "launches": n_launch, "clocks": clk.summary(), "wall": wall, "peaks": pk,
        "first_call": first,
        "pre_med_best": (statistics.median(per_pre), min(per_pre)),
        "dec_med_best": (statistics.median(per_dec), min(per_dec)),
    }

    res["traffic"] = measured_traffic("prefill_sm103.cu", PREFILL.name)
    res["traffic_dec"] = measured_traffic("decode.cu", DECODE.name)
    if args.no_e2e or args.only != "step":
        res["t_e2e"], res["h2d"], res["d2h"] = None, 0, 0
        return res

    # ---- end to end through the public API with host buffers
    hQ = Q.cpu().pin_memory()
    hK = K.cpu().pin_memory()
    hV = V.cpu().pin_memory()
    hq = dd["q"].cpu().pin_memory()
    hkn, hvn = k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
    hbt = dd["block_table"].cpu().pin_memory()
    hsl = dd["seq_lens"].cpu().pin_memory()
    hpos = positions.cpu().pin_memory()
    hO = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
    hlse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    hOd = torch.empty(Od.shape, dtype=Od.dtype, pin_memory=True)
    dbt, dsl, dpos = torch.empty_like(dd["block_table"]), torch.empty_like(dd["seq_lens"]), \
        torch.empty_like(positions)
    dq = torch.empty_like(dd["q"])

    # The decode half is independent of the prefill: it runs on a stream of
    # its own, inside the time the prefill spends waiting on its first copy.
    dstream = torch.cuda.Stream(dev)
    fork, join = torch.cuda.Event(), torch.cuda.Event()

    def e2e_step():
        fork.record(stream)
        dstream.wait_event(fork)
        with torch.cuda.stream(dstream):
            dq.copy_(hq, non_blocking=True)
            k_new.copy_(hkn, non_blocking=True)
            v_new.copy_(hvn, non_blocking=True)
            dbt.copy_(hbt, non_blocking=True)
            dsl.copy_(hsl, non_blocking=True)
            dpos.copy_(hpos, non_blocking=True)
            attn.kv_append(k_new, v_new, dd["Kc"], dd["Vc"], dbt, seq_ids, dpos, stream=dstream)
            attn.decode(dq, dd["Kc"], dd["Vc"], dbt, dsl, max_seq_len=DECODE.len_hi, O=Od,
                        lse=lsed, workspace=ws, stream=dstream)
            hOd.copy_(Od, non_blocking=True)
        join.record(dstream)
        # prefill: host Q/K/V in, host O/lse out, copies overlapped with the
        # kernels chunk by chunk of heads inside the library
        attn.prefill_from_host(hQ, hK, hV, True, hO=hO, hlse=hlse, Q=Q, K=K, V=V, O=O, lse=lse,
                               chunks=args.e2e_chunks, stream=stream)
        stream.wait_event(join)

    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    res["t_e2e"] = a.elapsed_time(b) / 1e3 / e2e_steps
    res["h2d"] = sum(x.numel() * x.element_size() for x in (hQ, hK, hV, hq, hkn, hvn, hbt, hsl,
                                                            hpos))
    res["d2h"] = sum(x.numel() * x.element_size() for x in (hO, hlse, hOd))
    hpc = attn.prefill_from_host_heads_per_chunk(
        PREFILL.B, PREFILL.Hq, PREFILL.Hkv, PREFILL.n_q, PREFILL.d, args.e2e_chunks,
        torch.cuda.get_device_properties(dev).multi_processor_count)
    res["e2e_chunks"] = -(-(PREFILL.B * PREFILL.Hq) // hpc)
    return res


# ------------------------------------------------- single named workloads

_FIRST_CALL = {}


def _time_kernel(fn, stream, warmup, steps, flush):
    """Median and best device time of fn() over `steps` runs, L2 flushed
    (a 256 MiB write) before every run, outside the timed events.  The
    first call's host wall time (synchronised on both sides: lazy module
    load, tensor-map encoding and the run) is left in _FIRST_CALL["ms"]."""
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fn()
    torch.cuda.synchronize()
    _FIRST_CALL["ms"] = round((time.perf_counter() - t0) * 1e3, 3)
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) / 1e3)
    return statistics.median(ts), min(ts)


def workload_lines(name: str, steps: int, warmup: int):
    """Time one named workload (or every cell of the G x d x dtype sweep) by
    itself and yield one JSON-ready dict per measurement."""
    from exact_io_aware_106_b300 import attn

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk = peaks()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    jobs = []
    if name in W.PREFILL_WORKLOADS:
        jobs.append(("prefill", W.PREFILL_WORKLOADS[name]))
    elif name in W.PAGED_PREFILL_WORKLOADS:
        jobs.append(("paged-prefill", W.PAGED_PREFILL_WORKLOADS[name]))
    elif name.startswith("bwd-") and name[4:] in W.PREFILL_WORKLOADS:
        jobs.append(("backward", W.PREFILL_WORKLOADS[name[4:]]))
    elif name in W.DECODE_TOKENS_WORKLOADS:
        base = W.DECODE_WORKLOADS["paged-decode"]
        jobs.append(("decode-tokens", (W.DECODE_TOKENS_WORKLOADS[name][0], base, name)))
    elif name in W.DECODE_WORKLOADS:
        jobs.append(("decode", W.DECODE_WORKLOADS[name]))
    elif name.startswith(("sweep-decode-G", "sweep-prefill-G")):
        # one cell of the G x d sweep, e.g. sweep-decode-G16-d64-e4m3
        kind, g_, d_, kv = name.split("-")[1:]
        G, d = int(g_[1:]), int(d_[1:])
        jobs.append((kind, (W.sweep_decode if kind == "decode" else W.sweep_prefill)(G, d, kv)))
    elif name == "sweep":
        for kv in ("bf16", "e4m3"):
            for G in (1, 4, 8, 16):
                for d in (64, 128, 256):
                    jobs.append(("decode", W.sweep_decode(G, d, kv)))
                    jobs.append(("prefill", W.sweep_prefill(G, d, kv)))
    else:
        raise SystemExit(f"unknown workload {name}")
    for kind, spec in jobs:
        line = {"workload": getattr(spec, "name", ""), "kind": kind}
        try:
            if kind == "prefill":
                t = W.make_prefill(spec, seed=0, device=dev)
                kw = {}
                call = attn.prefill
                if spec.dtype == "e4m3":
                    kw = W.quantize_prefill_e4m3(t)
                elif spec.dtype == "e4m3b":
                    # block-wise Q / K scales (128 rows), V per head: quantised by
                    # the library's own kernel, outside the timed region
                    kw = W.quantize_prefill_e4m3(t)
                    for n in ("Q", "K"):
                        x = t[n]
                        c, s_ = attn.rotate_quantize_e4m3(
                            x.reshape(-1, x.shape[2], x.shape[3]).contiguous(), None,
                            rows_per_block=attn.E4M3_SCALE_BLOCK)
                        kw[n], kw[n.lower() + "_scale"] = c.view(x.shape), s_
                    call = attn.prefill_e4m3_blocks
                Q, K, V = kw.pop("Q", t["Q"]), kw.pop("K", t["K"]), kw.pop("V", t["V"])
                O = torch.empty(t["Q"].shape, dtype=W.DTYPES[spec.out_dtype], device=dev)
                lse = torch.empty(t["Q"].shape[:3], dtype=torch.float32, device=dev)

                def fn():
                    call(Q, K, V, spec.causal, O=O, lse=lse, stream=stream, **kw)
                med, best = _time_kernel(fn, stream, warmup, steps, flush)
                F = prefill_flops(spec)
                f8 = spec.dtype.startswith("e4m3")
                peak = pk["bf16_tflops"] * (2.0 if f8 else 1.0)
                Bp = prefill_bytes(spec)
                roof = max(F / (peak * 1e12), Bp / (pk["hbm_gbs"] * 1e9))
                line.update(ms=round(med * 1e3, 4), best_ms=round(best * 1e3, 4),
                            first_call_ms=_FIRST_CALL.get("ms"),
                            tflops=round(F / med / 1e12, 2),
                            pct_roofline=round(100 * roof / med, 2),
                            peak_tflops=peak,
                            peak_kind="measured burst bf16" + (
                                " x 2 (nominal fp8/bf16 ratio)" if f8 else ""))
            elif kind == "backward":
                line["workload"] = "bwd-" + spec.name
                t = W.make_backward(spec, seed=0, device=dev)
                O, lse = attn.prefill(t["Q"], t["K"], t["V"], spec.causal,
                                      out_dtype=W.DTYPES[spec.dtype])
                dQ, dK, dV = (torch.empty_like(t[k]) for k in ("Q", "K", "V"))
                ws = torch.empty(int(attn.lib().attn_backward_workspace_bytes(
                    spec.B, spec.Hq, spec.n_q)), dtype=torch.uint8, device=dev)

                def fn():
                    attn.backward(t["Q"], t["K"], t["V"], O, t["dO"], lse, spec.causal,
                                  dQ=dQ, dK=dK, dV=dV, workspace=ws, stream=stream)
                med, best = _time_kernel(fn, stream, warmup, steps, flush)
                # five products per visible pair (S, dP, dV, dK, dQ): 2.5 x the forward's
                F = 2.5 * prefill_flops(spec)
                roof = F / (pk["bf16_tflops"] * 1e12)
                line.update(ms=round(med * 1e3, 4), best_ms=round(best * 1e3, 4),
                            first_call_ms=_FIRST_CALL.get("ms"),
                            tflops=round(F / med / 1e12, 2),
                            pct_roofline=round(100 * roof / med, 2),
                            peak_tflops=pk["bf16_tflops"], peak_kind="measured burst bf16",
                            note="algorithmic flops = 5 products per pair; the kernels issue 7 "
                                 "(S and dP are recomputed by the dQ kernel)")
            elif kind == "decode-tokens":
                T, base, wname = spec
                line["workload"] = wname
                dd = W.make_decode(base, seed=0, device=dev)
                lens = dd["seq_lens"].cpu()
                g = torch.Generator(device=dev).manual_seed(5)
                q = torch.randn((base.num_seqs, base.Hq, T, base.d), generator=g, device=dev,
                                dtype=torch.float32).to(W.DTYPES[base.q_dtype])
                Od = torch.empty(q.shape, dtype=W.DTYPES[base.out_dtype], device=dev)
                lsed = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
                ws = torch.empty(attn.decode_workspace_bytes(base.num_seqs * T, base.Hq, base.d,
                                                             base.len_hi),
                                 dtype=torch.uint8, device=dev)

                def fn():
                    attn.decode_tokens(q, dd["Kc"], dd["Vc"], dd["block_table"],
                                       dd["seq_lens"], max_seq_len=base.len_hi, O=Od, lse=lsed,
                                       workspace=ws, stream=stream)
                med, best = _time_kernel(fn, stream, warmup, steps, flush)
                Bd = decode_bytes(base, lens) + (T - 1) * 2 * base.num_seqs * base.Hq * base.d * 2
                roof = max(T * decode_flops(base, lens) / (pk["bf16_tflops"] * 1e12),
                           Bd / (pk["hbm_gbs"] * 1e9))
                line.update(ms=round(med * 1e3, 4), best_ms=round(best * 1e3, 4),
                            first_call_ms=_FIRST_CALL.get("ms"),
                            gbs=round(Bd / med / 1e9, 1), bytes=Bd, new_tokens=T,
                            pct_roofline=round(100 * roof / med, 2),
                            peak_gbs=pk["hbm_gbs"], peak_kind="measured HBM copy")
            elif kind == "paged-prefill":
                t = W.make_paged_prefill(spec, seed=0, device=dev)
                lens = t["seq_lens"].cpu()
                O = torch.empty(t["Q"].shape, dtype=W.DTYPES[spec.out_dtype], device=dev)
                lse = torch.empty(t["Q"].shape[:3], dtype=torch.float32, device=dev)

                def fn():
                    attn.prefill_paged(t["Q"], t["Kc"], t["Vc"], t["block_table"],
                                       t["seq_lens"], max_seq_len=spec.len_hi,
                                       causal=spec.causal, O=O, lse=lse, stream=stream)
                med, best = _time_kernel(fn, stream, warmup, steps, flush)
                # pairs: new token i of sequence b sees len_b - n_q + i + 1 keys
                n = spec.n_q
                pairs = sum(n * (int(L) - n) + n * (n + 1) // 2 for L in lens) * spec.Hq
                F = 4.0 * spec.d * pairs
                e = ESZ[spec.dtype]
                Bp = (2 * spec.B * spec.Hq * n * spec.d * e
                      + 2 * spec.Hkv * spec.d * e * float(sum(int(L) for L in lens)))
                roof = max(F / (pk["bf16_tflops"] * 1e12), Bp / (pk["hbm_gbs"] * 1e9))
                line.update(ms=round(med * 1e3, 4), best_ms=round(best * 1e3, 4),
                            first_call_ms=_FIRST_CALL.get("ms"),
                            tflops=round(F / med / 1e12, 2),
                            pct_roofline=round(100 * roof / med, 2),
                            peak_tflops=pk["bf16_tflops"], peak_kind="measured burst bf16")
            else:
                dd = W.make_decode(spec, seed=0, device=dev)
                lens = dd["seq_lens"].cpu()
                S = spec.num_seqs
                Od = torch.empty((S, spec.Hq, spec.d), dtype=W.DTYPES[spec.out_dtype], device=dev)
                lsed = torch.empty((S, spec.Hq), dtype=torch.float32, device=dev)
                ws = torch.empty(attn.decode_workspace_bytes(S, spec.Hq, spec.d, spec.len_hi),
                                 dtype=torch.uint8, device=dev)

                def fn():
                    attn.decode(dd["q"], dd["Kc"], dd["Vc"], dd["block_table"], dd["seq_lens"],
                                max_seq_len=spec.len_hi, k_scale=dd["k_scale"],
                                v_scale=dd["v_scale"], O=Od, lse=lsed, workspace=ws,
                                stream=stream)
                med, best = _time_kernel(fn, stream, warmup, steps, flush)
                Bd = decode_bytes(spec, lens)
                roof = max(decode_flops(spec, lens) / (pk["bf16_tflops"] * 1e12),
                           Bd / (pk["hbm_gbs"] * 1e9))
                line.update(ms=round(med * 1e3, 4), best_ms=round(best * 1e3, 4),
                            first_call_ms=_FIRST_CALL.get("ms"),
                            gbs=round(Bd / med / 1e9, 1), bytes=Bd,
                            pct_roofline=round(100 * roof / med, 2),
                            peak_gbs=pk["hbm_gbs"], peak_kind="measured HBM copy")
            if attn.last_error(stream) != attn.OK:
                line["device_error"] = True
        except Exception as e:  # an unsupported cell is reported, not hidden
            line["unsupported"] = str(e).splitlines()[0][:160]
        yield line


# ------------------------------------------------------------- CPU oracle

def oracle_sample(threads: int, rows: int, seqs: int, seed: int = 0):
    """Time the fp64 oracle on a bounded sample of the same workload: `rows`
    query rows at the end of head 0 of the prefill (each sees all n keys) and
    `seqs` decode sequences with all their query heads."""
    import oracle

    spec = PREFILL
    g = torch.Generator().manual_seed(seed)
    Qh = torch.randn((1, 1, rows, spec.d), generator=g).to(torch.bfloat16)
    Kh = torch.randn((1, 1, spec.n_kv, spec.d), generator=g).to(torch.bfloat16)
    Vh = torch.randn((1, 1, spec.n_kv, spec.d), generator=g).to(torch.bfloat16)
    # rows n-rows..n-1 of an n-row causal problem: row r sees r+1 keys
    n = spec.n_q
    Qfull_rows = [(0, 0, n - rows + i) for i in range(rows)]
    Qpad = torch.zeros((1, 1, n, spec.d), dtype=torch.bfloat16)
    Qpad[0, 0, n - rows:] = Qh[0, 0]
    t0 = time.perf_counter()
    oracle.sdpa_rows(Qpad, Kh, Vh, Qfull_rows, True, nthreads=threads)
    t_pre = time.perf_counter() - t0
    pairs = sum(r[2] + 1 for r in Qfull_rows)
    F = 4.0 * spec.d * pairs

    dspec = W.DecodeSpec(seqs, DECODE.Hq, DECODE.Hkv, DECODE.d, DECODE.len_lo, DECODE.len_hi,
                         DECODE.block_size, DECODE.q_dtype, DECODE.kv_dtype, DECODE.out_dtype)
    dd = W.make_decode(dspec, seed=seed)
    t0 = time.perf_counter()
    oracle.decode_paged(dd["q"], dd["Kc"], dd["Vc"], dd["block_table"], dd["seq_lens"],
                        nthreads=threads)
    t_dec = time.perf_counter() - t0
    Bd = decode_bytes(dspec, dd["seq_lens"])
    return {"t_pre": t_pre, "F": F, "t_dec": t_dec, "Bd": Bd,
            "sample": f"prefill: last {rows} query rows of one head of the n=32768 causal "
                      f"problem ({pairs} pairs); decode: {seqs} sequences x 32 query heads "
                      f"({int(dd['seq_lens'].sum())} tokens)"}


def oracle_values(smp, pk):
    P = pk["bf16_tflops"] * 1e12
    BW = pk["hbm_gbs"] * 1e9
    roof = smp["F"] / P + smp["Bd"] / BW
    return {"pct": 100.0 * roof / (smp["t_pre"] + smp["t_dec"]),
            "tflops": smp["F"] / smp["t_pre"] / 1e12, "gbs": smp["Bd"] / smp["t_dec"] / 1e9}


def run_reference(args):
    """The oracle, as it stands, on the host cores: each step a bounded sample
    of the workload."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    pk = peaks()
    for _ in range(args.warmup):
        oracle_sample(threads, rows=8, seqs=1, seed=1)
    tp = td = F = Bd = 0.0
    smp = None
    for i in range(args.steps):
        smp = oracle_sample(threads, rows=16, seqs=1, seed=2 + i)
        tp += smp["t_pre"]
        td += smp["t_dec"]
        F += smp["F"]
        Bd += smp["Bd"]
    v = oracle_values({"t_pre": tp, "t_dec": td, "F": F, "Bd": Bd}, pk)
    t = (tp + td) / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v["pct"], 8),
        "unit": "% of roofline", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "long-32k prefill + paged-decode (oracle sample per step)",
                   "prefill": "B1 Hq64 Hkv8 d128 n32768 causal bf16",
                   "decode": "64 seqs Hq32 Hkv8 d128 len U[1024,32768] bf16 16-token blocks"},
        "prefill": {"tflops": v["tflops"]}, "decode": {"gbs": v["gbs"]},
        "cpu_baseline": {"value": round(v["pct"], 8), "unit": "% of roofline",
                         "cores": threads, "kind": "oracle", "sample": smp["sample"]},
        "e2e": {"value": round(v["pct"], 8), "unit": "% of roofline",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- main

def max_over_ranks(values, device):
    """Elementwise maximum of `values` over the ranks of the default process
    group (the job's time is its slowest rank's); NCCL on the GPU, gloo on
    the CPU in the tests."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="head chunks of the host-buffer prefill (0: the library's choice)")
    ap.add_argument("--only", choices=["step", "prefill", "decode"], default="step",
                    help="run only part of the step (profiling)")
    ap.add_argument("--prefill-n", type=int, default=0,
                    help="override the prefill length (smaller profiling case)")
    ap.add_argument("--decode-seqs", type=int, default=0,
                    help="override the number of decode sequences (profiling case)")
    ap.add_argument("--workload", default="",
                    help="time one named workload alone (single-head, gqa-4k, long-23k, "
                         "long-32k, paged-decode, paged-prefill, spec-decode-4, "
                         "bwd-<prefill workload>, one sweep cell such as "
                         "sweep-decode-G16-d64-e4m3) or every cell of 'sweep'; one line each")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")

    if args.workload:
        for line in workload_lines(args.workload, args.steps, args.warmup):
            line.update(metric=METRIC, unit="% of roofline", n_gpus=1, impl="ours",
                        data="synthetic", l2="flushed before every timed run")
            print(json.dumps(line), flush=True)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)

    t_step = res["t_step"]
    t_e2e = res["t_e2e"] if res["t_e2e"] is not None else float("nan")
    roof_total = res["roof_step"]
    if world > 1:
        t_step, t_e2e = max_over_ranks([t_step, t_e2e], "cuda")
        roof_total = res["roof_step"] * world
    pk = res["peaks"]
    if rank == 0:
        value = 100.0 * roof_total / t_step
        pre_tflops = res["F"] / res["t_pre"] / 1e12 if args.only != "decode" else None
        dec_gbs = res["Bd"] / res["t_dec"] / 1e9 if args.only != "prefill" else None
        r2 = lambda x, n: None if x is None or x != x else round(x, n)  # noqa: E731
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "% of roofline",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_step * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": {"step": "long-32k prefill + kv-append + paged-decode",
                                    "prefill": f"{PREFILL.name} prefill only",
                                    "decode": f"{DECODE.name} kv-append + decode only"}[args.only],
                       "prefill": f"B{PREFILL.B} Hq{PREFILL.Hq} Hkv{PREFILL.Hkv} d{PREFILL.d} "
                                  f"n{PREFILL.n_q} causal bf16 -> bf16 + lse",
                       "decode": f"{DECODE.num_seqs} seqs Hq{DECODE.Hq} Hkv{DECODE.Hkv} "
                                 f"d{DECODE.d} len U[{DECODE.len_lo},{DECODE.len_hi}] bf16 "
                                 "cache, 16-token blocks, random block table",
                       "append": "1 token per sequence into its last slot",
                       "l2": "inputs larger than L2 (no flush)",
                       "parallelism": f"replicas x{world}"},
            "gpu_launches": res["launches"],
            "clocks": res["clocks"],
        }
        if pre_tflops is not None:
            line["prefill"] = {
                "tflops": round(pre_tflops, 2), "ms": round(res["t_pre"] * 1e3, 4),
                "pct_roofline": round(100 * res["roof_pre"] / res["t_pre"], 2),
                "pct_of_burst_peak": round(100 * pre_tflops / pk["bf16_tflops"], 2),
                "median_ms": round(res["pre_med_best"][0], 4),
                "best_ms": round(res["pre_med_best"][1], 4),
                "first_call_ms": res["first_call"].get("prefill_ms")}
            line["roofline"] = {
                "bound": "tensor", "kernel": "prefill_kernel<128,bf16,bf16>",
                "achieved": round(pre_tflops, 2), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(pre_tflops / pk["bf16_tflops"], 4),
                "frac_of_sustained": round(pre_tflops / pk["bf16_tflops_sustained"], 4),
                "peak_kind": f"{pk['source']} burst bf16 (sub-second timed region)",
                "traffic": res["traffic"]}
        if dec_gbs is not None:
            line["decode"] = {
                "gbs": round(dec_gbs, 1), "ms": round(res["t_dec"] * 1e3, 4),
                "pct_roofline": round(100 * res["roof_dec"] / res["t_dec"], 2),
                "frac_of_8tbs_spec": round(dec_gbs / 8000.0, 4), "bytes": res["Bd"],
                "median_ms": round(res["dec_med_best"][0], 4),
                "best_ms": round(res["dec_med_best"][1], 4),
                "first_call_ms": res["first_call"].get("decode_ms")}
            line["append"] = {"ms": round(res["t_app"] * 1e3, 4)}
            dec_roof = {
                "bound": "hbm", "kernel": "decode_mma_kernel<128,bf16> + decode_combine_kernel",
                "achieved": round(dec_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(dec_gbs / pk["hbm_gbs"], 4),
                "peak_kind": f"{pk['source']} HBM copy", "traffic": res["traffic_dec"]}
            if pre_tflops is None:
                line["roofline"] = dec_roof
            else:
                line["decode_roofline"] = dec_roof
        line["e2e"] = {"value": r2(100.0 * roof_total / t_e2e, 3), "unit": "% of roofline",
                       "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                       "ms_per_step": r2(t_e2e * 1e3, 3),
                       "prefill_chunks": res.get("e2e_chunks"),
                       "calls": "attn_prefill_from_host (pinned host Q/K/V in, O/lse out, copies "
                                "overlapped with the kernels) + attn_kv_append + attn_decode "
                                "(host q, new K/V, table, lengths in; O out)"}
        if not args.no_cpu_baseline:
            threads = os.cpu_count() or 1
            smp = oracle_sample(threads, rows=1024, seqs=24)
            v = oracle_values(smp, pk)
            line["cpu_baseline"] = {"value": round(v["pct"], 8), "unit": "% of roofline",
                                    "cores": threads, "kind": "oracle", "sample": smp["sample"],
                                    "tflops": v["tflops"], "gbs": v["gbs"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
