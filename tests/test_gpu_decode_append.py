"""The fused decode step (pkv_paged_attention_decode_append) against the two calls it fuses.

reshape_and_cache(key, value, slots) followed by paged_attention_decode must give, bit for bit,
the same attention output and the same pools as the single fused launch, and both must match the
fp64 oracle.  Covered: every head size and block size, one and several partitions per sequence,
a padding slot (-1), a slot the table does not map the last position to, a slot outside the pool,
inputs in page-locked host memory, and the full-size OPT-13B-shaped batch in the launch
configuration the bench times."""
import numpy as np
import pytest
import torch

from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl
from tests.helpers import ATOL, max_err, sample_seqs

pytestmark = pytest.mark.gpu


def _last_slots(w):
    """The slot of each sequence's last position (its new token) through the block table."""
    B = w.block_size
    slots = np.full(w.num_seqs, -1, dtype=np.int64)
    for s, c in enumerate(w.context_lens):
        if c > 0:
            slots[s] = int(w.block_tables[s, (c - 1) // B]) * B + (c - 1) % B
    return slots


def _both(w, slots, dev, host=False):
    k0, v0 = w.pools(dev)
    q = w.q(dev)
    key, value = wl.new_tokens(w.num_seqs, w.num_heads, w.head_dim, 4242 + w.head_dim, dev)
    tables = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    slots_d = torch.from_numpy(slots).to(dev)
    # the two calls
    k1, v1 = k0.clone(), v0.clone()
    pkv.reshape_and_cache(key, value, k1, v1, slots_d)
    ref = pkv.paged_attention_decode(q, k1, v1, tables, lens, w.scale, w.block_size)
    code_ref = pkv.device_error()
    # the fused launch
    k2, v2 = k0.clone(), v0.clone()
    if host:
        pin = lambda t: t.detach().cpu().contiguous().pin_memory()
        out = torch.empty(tuple(q.shape), dtype=torch.float16).pin_memory()
        got = pkv.paged_attention_decode_append(pin(q), pin(key), pin(value), pin(slots_d), k2, v2, pin(tables),
                                                pin(lens), w.scale, w.block_size, out=out)
    else:
        got = pkv.paged_attention_decode_append(q, key, value, slots_d, k2, v2, tables, lens, w.scale,
                                                w.block_size)
    code = pkv.device_error()
    torch.cuda.synchronize()
    return ref, got, code_ref, code, (k1, v1), (k2, v2), key, value


def _same_pools(a, b):
    # bit patterns: unfilled slots hold NaN, which compares unequal to itself
    return all(torch.equal(x.view(torch.int16), y.view(torch.int16)) for x, y in zip(a, b))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [4, 8, 16, 32])
def test_append_equals_reshape_then_decode(cuda_device, D, B):
    lens = [1, B, B + 1, 130, 700, 2049, 57]
    w = wl.custom(3100 + D + B, lens, num_heads=3, head_dim=D, block_size=B)
    slots = _last_slots(w)
    ref, got, code_ref, code, pools_ref, pools_got, key, value = _both(w, slots, cuda_device)
    assert code_ref == 0 and code == 0
    assert torch.equal(got.cpu(), ref.cpu())
    assert _same_pools(pools_ref, pools_got)


def test_append_long_contexts_many_partitions(cuda_device):
    # two sequences x two heads: 128-token partitions, the new token in the last of many
    w = wl.custom(3201, [4096, 3001], num_heads=2, head_dim=128, block_size=16)
    ref, got, code_ref, code, pools_ref, pools_got, _, _ = _both(w, _last_slots(w), cuda_device)
    assert code_ref == 0 and code == 0
    assert torch.equal(got.cpu(), ref.cpu())
    assert _same_pools(pools_ref, pools_got)


def test_append_matches_the_oracle(cuda_device):
    w = wl.custom(3202, [300, 17, 1024], num_heads=4, head_dim=128, block_size=16)
    slots = _last_slots(w)
    ref, got, _, code, _, (k2, v2), key, value = _both(w, slots, cuda_device)
    assert code == 0
    # the oracle on the pools as the appended token left them: the new rows at their slots
    kh, vh = w.pools("cpu")
    B = w.block_size
    for s, slot in enumerate(slots):
        kh[slot // B, :, slot % B, :] = key[s].cpu()
        vh[slot // B, :, slot % B, :] = value[s].cpu()
    from oracle import attention as oracle_attention
    expect = oracle_attention.paged_decode_attention(w.q("cpu").numpy(), kh.numpy(), vh.numpy(), w.block_tables,
                                                     w.context_lens, w.scale)
    assert max_err(got, expect) <= ATOL


def test_append_padding_and_unmapped_slots(cuda_device):
    # sequence 1: no new row (-1); sequence 2: a slot the table does not map its last position to
    # (the row is stored there, and the last position reads what the pool holds)
    w = wl.custom(3203, [200, 90, 150, 40], num_heads=2, head_dim=64, block_size=8, num_blocks=70)
    slots = _last_slots(w)
    slots[1] = -1
    used = {int(b) for b in w.block_tables.ravel() if b >= 0}
    free = next(b for b in range(w.num_blocks) if b not in used)
    slots[2] = free * w.block_size + 3
    ref, got, code_ref, code, pools_ref, pools_got, _, _ = _both(w, slots, cuda_device)
    assert code_ref == 0 and code == 0
    assert torch.equal(got.cpu(), ref.cpu())
    assert _same_pools(pools_ref, pools_got)


def test_append_slot_outside_pool_recorded(cuda_device):
    w = wl.custom(3204, [60, 33], num_heads=2, head_dim=128, block_size=16)
    slots = _last_slots(w)
    slots[0] = w.num_blocks * w.block_size + 7
    ref, got, code_ref, code, pools_ref, pools_got, _, _ = _both(w, slots, cuda_device)
    assert code_ref == 3 and code == 3                         # PKV_DEV_BAD_SLOT from both
    assert torch.equal(got.cpu(), ref.cpu())
    assert _same_pools(pools_ref, pools_got)


def test_append_reads_host_inputs(cuda_device):
    w = wl.custom(3205, [500, 1, 2100, 64], num_heads=3, head_dim=128, block_size=16)
    ref, got, code_ref, code, pools_ref, pools_got, _, _ = _both(w, _last_slots(w), cuda_device, host=True)
    assert code_ref == 0 and code == 0
    assert not got.is_cuda
    assert torch.equal(got, ref.cpu())
    assert _same_pools(pools_ref, pools_got)


@pytest.mark.parametrize("batch", ["opt13b", "capacity_1x2048"])
def test_append_full_size(cuda_device, batch):
    # the OPT-13B-shaped step (1024-token partitions, as the bench times it) and one 2048-token
    # sequence (512-token partitions, the new token in the fourth): the fused launch equals the two
    # calls bit for bit, output and both pools; sampled sequences match the oracle on blocks
    # regenerated on the CPU with the new rows at their slots
    w = wl.opt13b() if batch == "opt13b" else wl.capacity(num_seqs=1, block_size=16)
    slots = _last_slots(w)
    ref, got, code_ref, code, pools_ref, pools_got, key, value = _both(w, slots, cuda_device)
    assert code_ref == 0 and code == 0
    assert torch.equal(got, ref)
    assert _same_pools(pools_ref, pools_got)
    del pools_ref, pools_got
    seqs = sample_seqs(w, 6)
    kc, vc, tabs, lens = w.compact_pools(seqs)
    B = w.block_size
    for i, s in enumerate(seqs):
        last = int(lens[i]) - 1
        blk, row = int(tabs[i, last // B]), last % B
        kc[blk, :, row, :] = key[s].cpu()
        vc[blk, :, row, :] = value[s].cpu()
    from oracle import attention as oracle_attention
    expect = oracle_attention.paged_decode_attention(w.q("cpu").numpy()[seqs], kc.numpy(), vc.numpy(), tabs, lens,
                                                     w.scale)
    assert max_err(got[seqs], expect) <= ATOL
