"""The boundary from plain C: tests/c/abi_smoke.c includes include/attn.h,
is compiled as C99 with warnings as errors, links libattn.so and runs its
host-side checks (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "exact_io_aware_106_b300")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_links_and_runs(tmp_path):
    from exact_io_aware_106_b300 import build
    lib = build.build()
    exe = tmp_path / "abi_smoke"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c", "abi_smoke.c"),
                           "-L", os.path.dirname(lib), "-lattn",
                           "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout


CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.mark.gpu
@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_runs_kernels_through_the_abi(tmp_path):
    """tests/c/abi_gpu.c, compiled as C11 against include/attn.h and the CUDA
    runtime, allocates device buffers with cudaMalloc and runs a prefill, a
    KV append and a paged decode; its outputs are gated against the oracle
    here."""
    import numpy as np
    import torch

    import oracle
    from exact_io_aware_106_b300 import build, workloads as W
    from tests.parity import assert_lse, assert_out

    lib = build.build()
    exe = tmp_path / "abi_gpu"
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                           os.path.join(ROOT, "tests", "c", "abi_gpu.c"),
                           "-L", os.path.dirname(lib), "-lattn",
                           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                           "-Wl,-rpath," + os.path.dirname(lib),
                           "-Wl,-rpath," + os.path.join(CUDA, "lib64"), "-o", str(exe)])

    def put(name, t):
        (tmp_path / name).write_bytes(np.ascontiguousarray(oracle._as_np(t)).tobytes())

    def get(name, dtype, shape):
        return np.frombuffer((tmp_path / name).read_bytes(), dtype=dtype).reshape(shape)

    # prefill inputs (sizes as in abi_gpu.c)
    p = W.make_prefill(W.PrefillSpec(1, 4, 2, 300, 300, 128, True, "bf16", "f32"), seed=21)
    for n in "QKV":
        put(f"{n}.bf16", p[n])
    # decode: 3 sequences, one new token each at its last position
    lens = [41, 2, 301]
    dspec = W.DecodeSpec(3, 8, 2, 128, 1, 512, 16, "bf16", "bf16", "f32")
    d = W.make_decode(dspec, seed=22, lens=lens)
    assert d["block_table"].shape[1] == 32
    kn, vn = W.make_append(3, 2, 128, "bf16", seed=22)
    sid = torch.arange(3, dtype=torch.int32)
    pos = torch.tensor([x - 1 for x in lens], dtype=torch.int32)
    put("num_blocks.i32", torch.tensor([d["num_blocks"]], dtype=torch.int32))
    for n, t in (("Kc.bf16", d["Kc"]), ("Vc.bf16", d["Vc"]), ("q.bf16", d["q"]),
                 ("block_table.i32", d["block_table"]), ("seq_lens.i32", d["seq_lens"]),
                 ("k_new.bf16", kn), ("v_new.bf16", vn), ("seq_ids.i32", sid),
                 ("positions.i32", pos)):
        put(n, t)
    out = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr
    assert "c abi gpu ok" in out.stdout

    O_ref, lse_ref = oracle.sdpa(p["Q"], p["K"], p["V"], True)
    assert_out(torch.from_numpy(get("O.f32", np.float32, (1, 4, 300, 128)).copy()), O_ref)
    assert_lse(torch.from_numpy(get("lse.f32", np.float32, (1, 4, 300)).copy()), lse_ref)
    Ko, Vo = oracle.kv_append(kn, vn, d["Kc"], d["Vc"], d["block_table"], sid, pos)
    assert np.array_equal(get("Kc_out.bf16", np.uint16, Ko.shape), Ko.view(np.uint16))
    assert np.array_equal(get("Vc_out.bf16", np.uint16, Vo.shape), Vo.view(np.uint16))
    Ko_t = torch.from_numpy(Ko.view(np.int16).copy()).view(torch.bfloat16)
    Vo_t = torch.from_numpy(Vo.view(np.int16).copy()).view(torch.bfloat16)
    Od_ref, lsed_ref = oracle.decode_paged(d["q"], Ko_t, Vo_t, d["block_table"], d["seq_lens"])
    assert_out(torch.from_numpy(get("Od.f32", np.float32, (3, 8, 128)).copy()), Od_ref)
    assert_lse(torch.from_numpy(get("lsed.f32", np.float32, (3, 8)).copy()), lsed_ref)
