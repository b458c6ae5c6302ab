"""The C ABI from a plain C program: `tests/c_caller/decode_step.c` links libpkv.so and the CUDA
runtime only (no Python, no PyTorch), lets the block manager place a batch's prompts and this
step's tokens, and runs the fused decode step with a workspace it allocated itself and the same
attention through the allocation-free entry.  This test writes the program's seeded inputs,
compiles and runs it, and checks what it wrote against the oracle: tables, lengths and slots
equal to the oracle's block manager, pools bit-exact after the step, attention within 2e-3, and
the two entry points' outputs bit for bit equal."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import attention as oracle_attention
from oracle import block_manager as obm
from oracle import cache_ops as oracle_cache_ops
from paged_kv_cache_73_gb300 import _build
from tests.helpers import ATOL

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _compile(tmp_path):
    lib = _build.build()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "decode_step")
    src = os.path.join(ROOT, "tests", "c_caller", "decode_step.c")
    lib_dir = os.path.dirname(lib)
    r = subprocess.run([nvcc, "-O2", "-I", os.path.join(ROOT, "include"), src, "-L", lib_dir, "-lpkv", "-lm",
                        "-Xlinker", f"-rpath,{lib_dir}", "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


@pytest.mark.parametrize("B,prompts", [(16, [40, 300, 1, 17, 1024]), (8, [7, 8, 9, 130])])
def test_plain_c_caller(tmp_path, cuda_device, B, prompts):
    exe = _compile(tmp_path)
    S, H, D, N, seed = len(prompts), 4, 128, 400, 77
    rng = np.random.default_rng(seed)
    order = rng.permutation(N).astype(np.int32)
    ora = obm.BlockManager(N, B, order)
    k = np.full((N, H, B, D), np.nan, dtype=np.float16)
    v = np.full((N, H, B, D), np.nan, dtype=np.float16)
    for s, n in enumerate(prompts):
        slots = ora.add_seq(s, n)
        oracle_cache_ops.reshape_and_cache(rng.standard_normal((n, H, D)).astype(np.float16),
                                           rng.standard_normal((n, H, D)).astype(np.float16), k, v, slots)
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    key = rng.standard_normal((S, H, D)).astype(np.float16)
    value = rng.standard_normal((S, H, D)).astype(np.float16)
    d = tmp_path
    for name, arr in (("prompts.i32", np.array(prompts, dtype=np.int32)), ("order.i32", order), ("k.f16", k),
                      ("v.f16", v), ("q.f16", q), ("key.f16", key), ("value.f16", value)):
        arr.tofile(d / name)
    r = subprocess.run([exe, str(d), str(S), str(H), str(D), str(B), str(N)], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    # the oracle's step: one token per sequence, written, then attention
    want = [ora.append_slot(s) for s in range(S)]
    max_blocks = -(-(max(prompts) + 1) // B)
    slots = np.fromfile(d / "slots.i64", dtype=np.int64)
    assert slots.tolist() == [w[0] for w in want] and all(w[1] < 0 for w in want)
    tables = np.fromfile(d / "tables.i32", dtype=np.int32).reshape(S, max_blocks)
    lens = np.fromfile(d / "lens.i32", dtype=np.int32)
    for s in range(S):
        ids, ctx = ora.block_table(s)
        assert tables[s, :len(ids)].tolist() == ids and (tables[s, len(ids):] == -1).all() and lens[s] == ctx
    oracle_cache_ops.reshape_and_cache(key, value, k, v, slots)
    assert np.array_equal(np.fromfile(d / "k_after.f16", dtype=np.uint16), k.view(np.uint16).ravel())
    assert np.array_equal(np.fromfile(d / "v_after.f16", dtype=np.uint16), v.view(np.uint16).ravel())
    ref = oracle_attention.paged_decode_attention(q, k, v, tables, lens, D ** -0.5)
    out = np.fromfile(d / "out.f16", dtype=np.float16).reshape(S, H, D)
    out_static = np.fromfile(d / "out_static.f16", dtype=np.float16).reshape(S, H, D)
    assert np.isfinite(out.astype(np.float64)).all()
    assert float(np.max(np.abs(out.astype(np.float64) - ref))) <= ATOL
    assert np.array_equal(out.view(np.uint16), out_static.view(np.uint16))
