"""Paged decode attention on the GPU against the fp64 oracle (max abs error <= 2e-3).

Small batches are compared element by element in full; the full-size
batches (the OPT-13B-shaped decode batch, parallel sampling, shared prefix,
the capacity sweep) run whole on the GPU, in the same launch configuration
the bench times, and the oracle checks sampled sequences, including the
longest and shortest, regenerated on the CPU.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oracle_attention
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl
from tests.helpers import ATOL, device_inputs, gpu_attention, max_err, oracle_on, sample_seqs

pytestmark = pytest.mark.gpu


def _full_check(w, dev):
    out = gpu_attention(w, dev)
    ref = oracle_on(w, range(w.num_seqs))
    err = max_err(out, ref)
    assert err <= ATOL, f"{w.name}: max abs error {err}"
    return out


def test_tiny_batch(cuda_device):
    _full_check(wl.tiny(), cuda_device)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [4, 8, 16, 32])
def test_ragged_lengths_every_shape(cuda_device, D, B):
    # lengths around chunk, block and partition edges: 1, B-1, B, B+1, 127..129, 255..257, 511..513, 1000
    lens = [1, B - 1, B, B + 1, 16, 17, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1000, 2049]
    w = wl.custom(100 + D + B, lens, num_heads=3, head_dim=D, block_size=B, name=f"ragged_D{D}_B{B}")
    _full_check(w, cuda_device)


def test_long_context_many_partitions(cuda_device):
    w = wl.custom(7, [4096, 3000, 1], num_heads=2, head_dim=128, block_size=16, name="long")
    _full_check(w, cuda_device)


def test_single_token_context_is_its_value(cuda_device):
    w = wl.custom(11, [1] * 5, num_heads=4, head_dim=128, block_size=16)
    q, k, v, tables, lens = device_inputs(w, cuda_device)
    out = gpu_attention(w, cuda_device, (q, k, v, tables, lens))
    first = v[tables[:, 0].long(), :, 0, :]
    assert torch.equal(out, first)


def test_zero_length_context_gives_zero_row(cuda_device):
    w = wl.custom(12, [0, 33, 0, 5], num_heads=2, head_dim=64, block_size=16)
    out = gpu_attention(w, cuda_device)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    ref = oracle_on(w, [1, 3])
    assert max_err(out[[1, 3]], ref) <= ATOL


def test_empty_batch_is_a_no_op(cuda_device):
    q = torch.empty((0, 2, 64), dtype=torch.float16, device=cuda_device)
    k = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=cuda_device)
    out = pkv.paged_attention_decode(q, k, k, torch.zeros((0, 1), dtype=torch.int32, device=cuda_device),
                                     torch.zeros(0, dtype=torch.int32, device=cuda_device), 0.125, 16)
    assert out.shape == (0, 2, 64)


def test_deterministic_and_invariant_under_relabelling(cuda_device):
    w = wl.opt13b(seed=5, num_seqs=8, lo=100, hi=900)
    q, k, v, tables, lens = device_inputs(w, cuda_device)
    a = gpu_attention(w, cuda_device, (q, k, v, tables, lens))
    b = gpu_attention(w, cuda_device, (q, k, v, tables, lens))
    assert torch.equal(a, b)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(3)).to(cuda_device)
    k2 = torch.empty_like(k)
    v2 = torch.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    t2 = torch.where(tables >= 0, perm[tables.clamp(min=0).long()].int(), tables)
    c = gpu_attention(w, cuda_device, (q, k2, v2, t2, lens))
    assert torch.equal(a, c)


def test_garbage_in_unused_table_columns_is_ignored(cuda_device):
    w = wl.custom(13, [20, 70, 3], num_heads=2, head_dim=128, block_size=16, num_blocks=16)
    q, k, v, tables, lens = device_inputs(w, cuda_device)
    base = gpu_attention(w, cuda_device, (q, k, v, tables, lens))
    junk = tables.clone()
    junk[junk < 0] = 123456789                       # far outside the pool, never used
    assert torch.equal(gpu_attention(w, cuda_device, (q, k, v, junk, lens)), base)


def test_out_of_range_block_id_is_recorded_not_read(cuda_device):
    w = wl.custom(14, [40, 40], num_heads=2, head_dim=64, block_size=16, num_blocks=8)
    q, k, v, tables, lens = device_inputs(w, cuda_device)
    bad = tables.clone()
    bad[1, 1] = w.num_blocks + 5
    out = pkv.paged_attention_decode(q, k, v, bad, lens, w.scale, 16)
    assert pkv.device_error() == 1
    assert pkv.device_error() == 0                    # the read cleared it
    ref = oracle_on(w, [0])
    assert max_err(out[:1], ref) <= ATOL and torch.all(out[1] == 0)


def test_context_beyond_table_capacity_is_recorded(cuda_device):
    w = wl.custom(15, [30, 20], num_heads=2, head_dim=64, block_size=16)
    q, k, v, tables, lens = device_inputs(w, cuda_device)
    lens2 = lens.clone()
    lens2[0] = tables.shape[1] * 16 + 1
    out = pkv.paged_attention_decode(q, k, v, tables, lens2, w.scale, 16)
    assert pkv.device_error() == 2
    assert torch.all(out[0] == 0)


def test_workspace_too_small_is_refused(cuda_device):
    # 2000 tokens on a 2-head grid: 16 partitions of 128 tokens, more than one cluster merges, so
    # the partial results need the workspace
    w = wl.custom(16, [2000], num_heads=2, head_dim=64, block_size=16)
    assert pkv.paged_attention_plan(1, 2, 64, w.max_blocks_per_seq, 16)[1] == 2
    q, k, v, tables, lens = device_inputs(w, cuda_device)
    tiny_ws = torch.empty(16, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_decode(q, k, v, tables, lens, w.scale, 16, workspace=tiny_ws)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE


def test_on_chip_merge_needs_no_workspace(cuda_device):
    # 600 tokens on a 2-head grid: 5 partitions merged inside one cluster per head; no workspace
    w = wl.custom(17, [600, 150], num_heads=2, head_dim=64, block_size=16)
    assert pkv.paged_attention_plan(2, 2, 64, w.max_blocks_per_seq, 16)[1] == 1
    q, k, v, tables, lens = device_inputs(w, cuda_device)
    out = torch.empty_like(q)
    assert pkv.load().pkv_paged_attention_decode(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), tables.data_ptr(), lens.data_ptr(), 2, 2, 64, k.shape[0],
        w.max_blocks_per_seq, w.scale, 16, out.data_ptr(), None, 0, None) == pkv.PKV_OK
    assert pkv.device_error() == 0
    assert max_err(out, oracle_on(w, [0, 1])) <= ATOL


def test_opt13b_batch_full_size(cuda_device):
    w = wl.opt13b()
    out = gpu_attention(w, cuda_device)
    seqs = sample_seqs(w, 6)
    assert max_err(out[seqs], oracle_on(w, seqs)) <= ATOL


@pytest.mark.parametrize("prompt_len", [512, 511])
def test_parallel_sampling_full_size(cuda_device, prompt_len):
    w = wl.parallel_sampling(prompt_len=prompt_len)
    out = gpu_attention(w, cuda_device)
    # the n samples of prompt 0 (shared blocks) plus the longest/shortest
    seqs = sorted(set([0, 1, 2, 3] + sample_seqs(w, 2)))
    assert max_err(out[seqs], oracle_on(w, seqs)) <= ATOL


def test_shared_prefix_full_size(cuda_device):
    w = wl.shared_prefix()
    assert w.shared_blocks == 64
    out = gpu_attention(w, cuda_device)
    seqs = sample_seqs(w, 5)
    assert max_err(out[seqs], oracle_on(w, seqs)) <= ATOL


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("S", [1, 16, 64, 256])
def test_capacity_sweep(cuda_device, S, B):
    w = wl.capacity(num_seqs=S, block_size=B)
    out = gpu_attention(w, cuda_device)
    seqs = sample_seqs(w, 4)
    assert max_err(out[seqs], oracle_on(w, seqs)) <= ATOL


def test_capacity_pool_filling_most_of_hbm(cuda_device):
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info(cuda_device)
    B, H, D = 16, 40, 128
    block_bytes = H * B * D * 2
    n = int(0.80 * free / (2 * block_bytes))
    w = wl.capacity(num_seqs=64, block_size=B, num_blocks=n)
    inputs = device_inputs(w, cuda_device, num_blocks=n)
    try:
        out = gpu_attention(w, cuda_device, inputs)
        seqs = sample_seqs(w, 4)
        assert max_err(out[seqs], oracle_on(w, seqs)) <= ATOL
        assert int(w.block_tables.max()) > n // 2          # ids really spread over the pool
    finally:
        del inputs
        torch.cuda.empty_cache()


@pytest.mark.parametrize("shards", [2, 4])
def test_head_sharded_pools_match_unsharded(cuda_device, shards):
    # tensor parallelism as the pages describe it: every shard keeps the same block table and
    # holds only its heads of every block; concatenating the shards' outputs gives the
    # unsharded result (bit for bit while the launch plan is the same)
    w = wl.opt13b(seed=9, num_seqs=64)
    q, k, v, tables, lens = device_inputs(w, cuda_device)
    full = gpu_attention(w, cuda_device, (q, k, v, tables, lens))
    H = w.num_heads
    step = H // shards
    plan = pkv.paged_attention_plan(64, H, 128, w.max_blocks_per_seq, 16)
    parts = []
    for r in range(shards):
        hs = slice(r * step, (r + 1) * step)
        qs, ks, vs = q[:, hs].contiguous(), k[:, hs].contiguous(), v[:, hs].contiguous()
        parts.append(pkv.paged_attention_decode(qs, ks, vs, tables, lens, w.scale, 16))
        assert pkv.paged_attention_plan(64, step, 128, w.max_blocks_per_seq, 16) == plan
    assert pkv.device_error() == 0
    assert torch.equal(torch.cat(parts, dim=1), full)
