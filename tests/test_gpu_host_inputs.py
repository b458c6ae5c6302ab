"""The decode step with its per-step inputs and its output in page-locked host memory.

The kernels read q, the block tables, the context lengths and the new K/V rows
across the host link and write the attention output there, with no staging copy.
The result must equal, bit for bit, the same call on device copies of the same
inputs, and match the fp64 oracle."""
import numpy as np
import pytest
import torch

from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl
from tests.helpers import ATOL, max_err, oracle_on

pytestmark = pytest.mark.gpu


def _pinned(t):
    return t.detach().cpu().contiguous().pin_memory()


@pytest.mark.parametrize("D,B", [(128, 16), (64, 8)])
def test_decode_reads_host_inputs(cuda_device, D, B):
    lens = [1, B, 300, 1000, 2049, 77]
    w = wl.custom(900 + D, lens, num_heads=3, head_dim=D, block_size=B)
    k, v = w.pools(cuda_device)
    q = w.q(cuda_device)
    tables = torch.from_numpy(w.block_tables).to(cuda_device)
    ctx = torch.from_numpy(w.context_lens).to(cuda_device)
    ref_dev = pkv.paged_attention_decode(q, k, v, tables, ctx, w.scale, w.block_size)
    assert pkv.device_error() == 0
    q_h, tables_h, ctx_h = _pinned(q), _pinned(tables), _pinned(ctx)
    out_h = torch.empty(tuple(q.shape), dtype=torch.float16).pin_memory()
    got = pkv.paged_attention_decode(q_h, k, v, tables_h, ctx_h, w.scale, w.block_size, out=out_h)
    assert pkv.device_error() == 0
    torch.cuda.synchronize()
    assert got.data_ptr() == out_h.data_ptr()
    assert torch.equal(out_h, ref_dev.cpu())
    assert max_err(out_h, oracle_on(w, range(w.num_seqs))) <= ATOL


def test_decode_allocates_host_output_for_host_q(cuda_device):
    w = wl.custom(905, [40, 3], num_heads=2, head_dim=128, block_size=16)
    k, v = w.pools(cuda_device)
    q_h = _pinned(w.q("cpu"))
    out = pkv.paged_attention_decode(q_h, k, v, _pinned(torch.from_numpy(w.block_tables)),
                                     _pinned(torch.from_numpy(w.context_lens)), w.scale, w.block_size)
    torch.cuda.synchronize()
    assert not out.is_cuda and out.is_pinned()
    assert max_err(out, oracle_on(w, range(w.num_seqs))) <= ATOL


def test_reshape_and_cache_reads_host_rows(cuda_device):
    w = wl.custom(906, [20, 47, 5], num_heads=4, head_dim=128, block_size=16)
    key, value = wl.new_tokens(8, 4, 128, 906, cuda_device)
    rng = np.random.default_rng(906)
    slots = rng.choice(w.num_blocks * w.block_size, size=8, replace=False).astype(np.int64)
    slots[3] = -1                                               # a padding token: skipped
    k1, v1 = w.pools(cuda_device)
    k2, v2 = k1.clone(), v1.clone()
    pkv.reshape_and_cache(key, value, k1, v1, torch.from_numpy(slots).to(cuda_device))
    pkv.reshape_and_cache(_pinned(key), _pinned(value), k2, v2, _pinned(torch.from_numpy(slots)))
    assert pkv.device_error() == 0
    torch.cuda.synchronize()
    # bit patterns: unfilled slots hold NaN, which compares unequal to itself
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))


def test_shared_prefix_decode_reads_host_tables(cuda_device):
    # 9 requests sharing a 64-token prefix (one group of 9 >= the shared minimum) plus a loner
    lens = [200, 70, 129, 65, 300, 96, 97, 160, 64, 40]
    base = wl.custom(907, lens, num_heads=2, head_dim=128, block_size=16)
    tables = base.block_tables.copy()
    for s in range(1, 9):
        tables[s, :4] = tables[0, :4]
    w = wl.from_tables("host_grouped", 907, 2, 128, 16, base.num_blocks, tables, base.context_lens)
    k, v = w.pools(cuda_device)
    q = w.q(cuda_device)
    gs, pl = torch.tensor([0, 9, 10], dtype=torch.int32), torch.tensor([64, 0], dtype=torch.int32)
    ref = pkv.paged_attention_decode_shared_prefix(q, k, v, torch.from_numpy(tables).to(cuda_device),
                                                   torch.from_numpy(w.context_lens).to(cuda_device),
                                                   gs.to(cuda_device), pl.to(cuda_device), w.scale, 16, 9)
    out_h = torch.empty(tuple(q.shape), dtype=torch.float16).pin_memory()
    pkv.paged_attention_decode_shared_prefix(q, k, v, _pinned(torch.from_numpy(tables)),
                                             _pinned(torch.from_numpy(w.context_lens)), _pinned(gs), _pinned(pl),
                                             w.scale, 16, 9, out=out_h)
    assert pkv.device_error() == 0
    torch.cuda.synchronize()
    assert torch.equal(out_h, ref.cpu())


def test_pageable_host_memory_is_refused(cuda_device):
    w = wl.custom(908, [10], num_heads=2, head_dim=64, block_size=8)
    k, v = w.pools(cuda_device)
    with pytest.raises(pkv.PkvError):
        pkv.paged_attention_decode(w.q("cpu"), k, v, torch.from_numpy(w.block_tables).to(cuda_device),
                                   torch.from_numpy(w.context_lens).to(cuda_device), w.scale, 8)


def test_copy_blocks_reads_host_mapping(cuda_device):
    w = wl.custom(909, [64, 48, 30], num_heads=2, head_dim=64, block_size=16)
    k1, v1 = w.pools(cuda_device)
    k2, v2 = k1.clone(), v1.clone()
    pairs = torch.tensor([[0, w.num_blocks - 1], [2, w.num_blocks - 2], [1, 3]], dtype=torch.int64)
    pkv.copy_blocks([k1], [v1], pairs.to(cuda_device))
    pkv.copy_blocks([k2], [v2], _pinned(pairs))
    assert pkv.device_error() == 0
    torch.cuda.synchronize()
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
