"""A decode loop driven from the host the way the bench's end-to-end figure drives it, checked
against the oracle.

Every step the C++ block manager assigns the new tokens' slots and writes the padded tables and
lengths straight into page-locked host buffers (the next step's into the second of two buffer
sets); the fused decode call, captured once per buffer set as a CUDA graph through the C ABI,
reads them across the host link, stores the new K/V rows and attends; the host waits for the
output in page-locked memory.  Contexts grow by one token a step.  After every step the output
is compared with the oracle's attention over the oracle's own block manager and pools, and at the
end the pools must be bit-identical.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as oracle_attention
from oracle import block_manager as obm
from oracle import cache_ops as oracle_cache_ops
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl
from tests.helpers import ATOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [16, 8])
def test_host_driven_decode_loop(cuda_device, B):
    S, H, D, N, steps, seed = 6, 4, 128, 400, 24, 1234
    rng = np.random.default_rng(seed)
    prompts = [int(x) for x in rng.integers(5, 300, size=S)]
    order = wl.free_list_order(N, seed)
    nat = pkv.BlockManager(N, B, order)
    ora = obm.BlockManager(N, B, order)
    shape = (N, H, B, D)
    k = torch.full(shape, float("nan"), dtype=torch.float16, device=cuda_device)
    v = torch.full(shape, float("nan"), dtype=torch.float16, device=cuda_device)
    k_ref = np.full(shape, np.nan, dtype=np.float16)
    v_ref = np.full(shape, np.nan, dtype=np.float16)
    # prompts written through reshape_and_cache on both sides
    for s, n in enumerate(prompts):
        slots = nat.add_seq(s, n)
        assert list(slots) == ora.add_seq(s, n)
        key, value = wl.new_tokens(n, H, D, seed + s, cuda_device)
        pkv.reshape_and_cache(key, value, k, v, torch.from_numpy(slots).to(cuda_device))
        kh, vh = wl.new_tokens(n, H, D, seed + s, "cpu")
        oracle_cache_ops.reshape_and_cache(kh.numpy(), vh.numpy(), k_ref, v_ref, slots)
    torch.cuda.synchronize()

    lib = pkv.load()
    max_blocks = -(-(max(prompts) + steps + 1) // B)
    ids = np.arange(S, dtype=np.int64)
    q_h = wl.dense_tensor((S, H, D), seed, wl.STREAM_Q, "cpu").pin_memory()
    out_h = torch.empty((S, H, D), dtype=torch.float16).pin_memory()
    ws = pkv.workspace_for(S, H, D, max_blocks, B, cuda_device)

    class Buf:
        def __init__(self):
            self.slots = torch.zeros(S, dtype=torch.int64).pin_memory()
            self.pairs = torch.zeros((S, 2), dtype=torch.int64).pin_memory()
            self.tables = torch.full((S, max_blocks), -1, dtype=torch.int32).pin_memory()
            self.lens = torch.zeros(S, dtype=torch.int32).pin_memory()
            self.key = torch.zeros((S, H, D), dtype=torch.float16).pin_memory()
            self.value = torch.zeros((S, H, D), dtype=torch.float16).pin_memory()

    bufs = [Buf(), Buf()]

    def call(b, stream_handle):
        assert lib.pkv_paged_attention_decode_append(
            q_h.data_ptr(), b.key.data_ptr(), b.value.data_ptr(), b.slots.data_ptr(), k.data_ptr(), v.data_ptr(),
            b.tables.data_ptr(), b.lens.data_ptr(), S, H, D, N, max_blocks, float(D ** -0.5), B,
            out_h.data_ptr(), None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(),
            stream_handle) == pkv.PKV_OK, lib.pkv_last_error()

    graphs = []
    for b in bufs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(b, torch.cuda.current_stream().cuda_stream)
        graphs.append(g)
    torch.cuda.synchronize()

    ncow = ctypes.c_int(0)
    stream = torch.cuda.current_stream()
    for step in range(steps):
        b = bufs[step % 2]
        # the host's part of the step, written in place into page-locked memory
        assert lib.pkv_bm_append_slots(nat._h, ids.ctypes.data, S, b.slots.data_ptr(), b.pairs.data_ptr(),
                                       ctypes.byref(ncow)) == pkv.PKV_OK
        assert lib.pkv_bm_block_tables(nat._h, ids.ctypes.data, S, b.tables.data_ptr(), max_blocks,
                                       b.lens.data_ptr()) == pkv.PKV_OK
        kn, vn = wl.new_tokens(S, H, D, 9000 + step, "cpu")         # this step's new rows
        b.key.copy_(kn)
        b.value.copy_(vn)
        # the oracle's step
        want = [ora.append_slot(s) for s in range(S)]
        assert b.slots.numpy().tolist() == [w_[0] for w_ in want]
        copies = [(src, dst) for _, src, dst in want if src >= 0]
        assert ncow.value == len(copies) == 0                        # no sharing in this batch
        oracle_cache_ops.reshape_and_cache(kn.numpy(), vn.numpy(), k_ref, v_ref, [w_[0] for w_ in want])
        graphs[step % 2].replay()
        stream.synchronize()
        tables = b.tables.numpy().copy()
        lens = b.lens.numpy().copy()
        ref = oracle_attention.paged_decode_attention(q_h.numpy(), k_ref, v_ref, tables, lens, D ** -0.5)
        got = out_h.numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert float(np.max(np.abs(got - ref))) <= ATOL, step
    assert pkv.device_error() == 0
    assert np.array_equal(k.cpu().numpy().view(np.uint16), k_ref.view(np.uint16))
    assert np.array_equal(v.cpu().numpy().view(np.uint16), v_ref.view(np.uint16))
    assert int(lens.min()) == min(prompts) + steps
