"""The allocation-free attention entry point against the ordinary one.

pkv_paged_attention_decode_static_workspace serves callers that cannot
allocate device memory (a C host program or plugin with no device allocator,
an engine whose block pools already hold all device memory, a path that must
not pay for cudaMalloc's device-wide synchronisation): it keeps the scratch in
a fixed array inside the library.  Through the C ABI, its output must equal
pkv_paged_attention_decode's with a caller workspace (the same kernels and
plan, so bit for bit) and match the oracle within the attention tolerance:
on two calls in a row, and on a call that follows another batch's call, whose
partial results are still in the array.  A batch too large for the array is
refused before anything runs.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oracle_attention
from paged_kv_cache_73_gb300 import _build
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = 2e-3

BATCHES = {
    "opt13b_full": wl.opt13b,
    "ragged_small": lambda: wl.custom(31, [1, 7, 300, 1000, 2049, 16], 4, 64, 8),
    # long contexts: more partitions per sequence than one cluster merges, so the partial results
    # go through the scratch
    "long_contexts": lambda: wl.custom(33, [12000, 9000, 300, 16000], 8, 128, 16),
    # one 2048-token sequence: its partitions merge inside clusters, so no scratch is needed
    "one_sequence": lambda: wl.capacity(seed=34, num_seqs=1),
}


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def _inputs(w, dev):
    k, v = w.pools(dev)
    return (w.q(dev), k, v, torch.from_numpy(w.block_tables).to(dev), torch.from_numpy(w.context_lens).to(dev))


def _oracle_err(w, out, seqs):
    kc, vc, tabs, lens = w.compact_pools(seqs)
    ref = oracle_attention.paged_decode_attention(w.q("cpu").numpy()[seqs], kc.numpy(), vc.numpy(), tabs, lens,
                                                  w.scale)
    got = out[seqs].double().cpu().numpy()
    assert np.isfinite(got).all()
    return float(np.max(np.abs(got - ref)))


def _static(w, inputs):
    q, k, v, tables, lens = inputs
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode_static_workspace(q, k, v, tables, lens, w.scale, w.block_size, out=out)
    assert pkv.device_error() == 0
    return out


@pytest.mark.parametrize("name", sorted(BATCHES))
def test_static_workspace_matches_caller_workspace(lib, cuda_device, name):
    w = BATCHES[name]()
    inputs = _inputs(w, cuda_device)
    q, k, v, tables, lens = inputs
    ref = pkv.paged_attention_decode(q, k, v, tables, lens, w.scale, w.block_size)
    assert pkv.device_error() == 0
    for _ in range(2):                               # the array keeps the previous call's contents
        out = _static(w, inputs)
        assert torch.equal(out, ref)
    seqs = [int(np.argmax(w.context_lens)), int(np.argmin(w.context_lens))]
    assert _oracle_err(w, out, sorted(set(seqs))) <= ATOL


def test_static_workspace_after_another_batch(lib, cuda_device):
    # a call on a large batch leaves its partial results in the array; a call on a different batch
    # (other sequences, heads and lengths) must write every partial result it reads
    big, small = BATCHES["long_contexts"](), BATCHES["ragged_small"]()
    _static(big, _inputs(big, cuda_device))
    inputs = _inputs(small, cuda_device)
    q, k, v, tables, lens = inputs
    out = _static(small, inputs)
    assert torch.equal(out, pkv.paged_attention_decode(q, k, v, tables, lens, small.scale, small.block_size))
    assert _oracle_err(small, out, list(range(small.num_seqs))) <= ATOL


def test_static_workspace_refuses_oversized_batch(lib, cuda_device):
    S, H, D, B, max_blocks = 256, 40, 128, 16, 1024           # 16384-token capacity: > 16 MiB of partials
    part_tokens, kernels = pkv.paged_attention_plan(S, H, D, max_blocks, B)
    assert kernels == 2                                       # too many partitions to merge on chip
    need = S * H * (-(-max_blocks * B // part_tokens)) * (D + 2) * 4
    assert need > pkv.paged_attention_static_workspace_bytes() == 16 << 20
    q = torch.zeros((S, H, D), dtype=torch.float16, device=cuda_device)
    kv = torch.zeros((4, H, B, D), dtype=torch.float16, device=cuda_device)
    tables = torch.zeros((S, max_blocks), dtype=torch.int32, device=cuda_device)
    lens = torch.ones(S, dtype=torch.int32, device=cuda_device)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_decode_static_workspace(q, kv, kv, tables, lens, 0.1, B)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE and "16777216" in str(e.value)
