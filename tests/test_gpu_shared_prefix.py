"""Shared-prefix decode attention on the GPU against the fp64 oracle.

paged_attention_decode_shared_prefix must give paged_attention_decode's result
(max abs error <= 2e-3 against the oracle) while reading each group's shared
prefix once: the prefix part runs on the tensor cores for the whole group and is
merged with each sequence's own part."""
import numpy as np
import pytest
import torch

from oracle import attention as oracle_attention
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl
from tests.helpers import ATOL

pytestmark = pytest.mark.gpu


def _run(w, group_start, prefix_lens, dev, tables=None):
    k, v = w.pools(dev)
    q = w.q(dev)
    tab = torch.from_numpy(w.block_tables if tables is None else tables).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    gs = torch.tensor(group_start, dtype=torch.int32, device=dev)
    pl = torch.tensor(prefix_lens, dtype=torch.int32, device=dev)
    max_group = int(np.max(np.diff(group_start)))
    out = pkv.paged_attention_decode_shared_prefix(q, k, v, tab, lens, gs, pl, w.scale, w.block_size, max_group)
    code = pkv.device_error()
    plain = pkv.paged_attention_decode(q, k, v, tab, lens, w.scale, w.block_size)
    return out, plain, q, code


def _check(w, out, q, seqs):
    kc, vc, tabs, lens = w.compact_pools(seqs)
    ref = oracle_attention.paged_decode_attention(q.cpu().numpy()[seqs].astype(np.float64), kc.numpy(), vc.numpy(),
                                                  tabs, lens, w.scale)
    got = out.cpu().numpy()[seqs].astype(np.float64)
    assert np.isfinite(got).all()
    err = float(np.max(np.abs(got - ref)))
    assert err <= ATOL, err
    return err


def test_shared_prefix_small(cuda_device):
    # 12 requests sharing a 1024-token prefix (64 blocks): one group, every sequence checked
    w = wl.shared_prefix(seed=1004, requests=12, suffix_lo=32, suffix_hi=300)
    out, plain, q, code = _run(w, [0, 12], [1024], cuda_device)
    assert code == 0, pkv.DEV_CODES.get(code, code)
    _check(w, out, q, list(range(12)))
    assert (out.double() - plain.double()).abs().max().item() <= 2 * ATOL


def test_shared_prefix_full_size(cuda_device):
    # the shared-prefix batch as the bench runs it (256 requests, 40 x 128, block 16), whole on the
    # GPU; the oracle on the longest, the shortest and two more sequences
    w = wl.shared_prefix()
    S = w.num_seqs
    out, plain, q, code = _run(w, [0, S], [1024], cuda_device)
    assert code == 0, pkv.DEV_CODES.get(code, code)
    lens = w.context_lens
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, S // 2})
    _check(w, out, q, seqs)
    assert (out.double() - plain.double()).abs().max().item() <= 2 * ATOL


@pytest.mark.parametrize("prompt_len,shared", [(512, 512), (511, 496)])
def test_parallel_sampling_groups(cuda_device, prompt_len, shared):
    # 32 prompts x 4 samples (prompt-major): groups of 4 share the prompt's whole blocks (with a
    # 511-token prompt the partly filled last block was copied on write, so 31 blocks are shared);
    # groups this small are read per sequence, so the call is plain decode
    w = wl.parallel_sampling(prompt_len=prompt_len)
    groups = list(range(0, w.num_seqs + 1, 4))
    out, plain, q, code = _run(w, groups, [shared] * (len(groups) - 1), cuda_device)
    assert code == 0, pkv.DEV_CODES.get(code, code)
    _check(w, out, q, [0, 1, 5, 63, 126, 127])
    assert (out.double() - plain.double()).abs().max().item() <= 2 * ATOL


def _grouped(D, B, seed):
    # groups [0, 9) prefix 64, [9, 10) no prefix, [10, 18) prefix 96 (member 11's context is exactly
    # its prefix), [18, 20) prefix 32 (fewer than 8 members: read per sequence): members map their
    # first blocks onto the group's first sequence's
    lens = [300, 70, 129, 65, 200, 96, 97, 160, 64, 17, 200, 96, 97, 160, 400, 129, 250, 111, 33, 40]
    groups, prefixes = [0, 9, 10, 18, 20], [64, 0, 96, 32]
    base = wl.custom(seed, lens, num_heads=3, head_dim=D, block_size=B)
    tables = base.block_tables.copy()
    for g in range(len(prefixes)):
        nb = prefixes[g] // B
        for s_ in range(groups[g] + 1, groups[g + 1]):
            tables[s_, :nb] = tables[groups[g], :nb]
    w = wl.from_tables(f"grouped_D{D}_B{B}", seed, 3, D, B, base.num_blocks, tables, base.context_lens)
    return w, groups, prefixes


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [4, 8, 16, 32])
def test_groups_every_shape(cuda_device, D, B):
    w, groups, prefixes = _grouped(D, B, 500 + D + B)
    out, plain, q, code = _run(w, groups, prefixes, cuda_device)
    assert code == 0, pkv.DEV_CODES.get(code, code)
    _check(w, out, q, list(range(w.num_seqs)))


def test_prefix_mismatch_recorded(cuda_device):
    # member 2 of group [0, 9) maps its first block elsewhere: the kernel reads the prefix through
    # member 0's row and records the mismatch
    w, groups, prefixes = _grouped(128, 16, 611)
    tables = w.block_tables.copy()
    tables[2, 0] = tables[19, 1]
    out, plain, q, code = _run(w, groups, prefixes, cuda_device, tables=tables)
    assert code == 7


def test_groups_not_covering_the_batch_recorded(cuda_device):
    w, groups, prefixes = _grouped(64, 8, 612)
    out, plain, q, code = _run(w, groups[:-1], prefixes[:-1], cuda_device)   # 18, 19 in no group
    assert code == 7
    _check(w, out, q, list(range(18)))
