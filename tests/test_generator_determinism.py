"""The seeded generator gives the same bits however it is sliced (the oracle
regenerates single blocks on the CPU that the GPU side made in bulk)."""
import numpy as np
import torch

from paged_kv_cache_73_gb300 import workloads as wl


def test_block_values_match_dense_tensor():
    H, B, D = 3, 8, 64
    dense = wl.dense_tensor((10, H, B, D), 42, wl.STREAM_K, "cpu", chunk=1000)
    blocks = wl.block_values(np.array([7, 2, 9]), H, B, D, 42, wl.STREAM_K)
    assert torch.equal(blocks.view(torch.int16), dense[[7, 2, 9]].view(torch.int16))


def test_streams_and_seeds_differ():
    i = torch.arange(1000)
    a = wl.values_at(1, 1, i)
    assert not torch.equal(a, wl.values_at(1, 2, i))
    assert not torch.equal(a, wl.values_at(2, 1, i))
    assert torch.equal(a, wl.values_at(1, 1, i))


def test_high_index_bits_matter():
    i = torch.arange(100, dtype=torch.int64)
    assert not torch.equal(wl.values_at(1, 1, i), wl.values_at(1, 1, i + (1 << 32)))


def test_distribution():
    x = wl.values_at(5, 1, torch.arange(1 << 20)).float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.02 and x.abs().max().item() < 3.6


def test_nan_marks_unfilled_slots():
    w = wl.custom(3, [5, 16], num_heads=2, head_dim=64, block_size=8, num_blocks=6)
    k, v = w.pools()
    t = w.block_tables
    assert torch.isnan(k[t[0, 0], :, 5:]).all() and not torch.isnan(k[t[0, 0], :, :5]).any()
    assert not torch.isnan(k[t[1, 1]]).any()
    unused = [b for b in range(6) if b not in w.block_fill]
    assert torch.isnan(k[unused]).all()


import pytest


@pytest.mark.gpu
def test_gpu_and_cpu_generators_agree(cuda_device):
    i = torch.arange(0, 1 << 22, 7, dtype=torch.int64)
    for stream in (wl.STREAM_Q, wl.STREAM_K, wl.STREAM_V):
        a = wl.values_at(1002, stream, i)
        b = wl.values_at(1002, stream, i.to(cuda_device)).cpu()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    hi = torch.arange(50, dtype=torch.int64) + (5 << 32)
    assert torch.equal(wl.values_at(3, 1, hi).view(torch.int16), wl.values_at(3, 1, hi.to(cuda_device)).cpu().view(torch.int16))
