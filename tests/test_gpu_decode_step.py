"""Whole decode steps, product path against oracle path, from the same seeded inputs.

Product: C++ block manager -> copy_blocks -> reshape_and_cache -> paged decode
attention, all on the GPU through the C ABI.  Oracle: the oracle's block
manager, cache ops and attention on the CPU.  Pools must stay bit-identical
after every step; attention outputs agree within 2e-3.
"""
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


class TwoSides:
    def __init__(self, dev, num_blocks, H, D, B, seed):
        self.dev, self.N, self.H, self.D, self.B, self.seed = dev, num_blocks, H, D, B, seed
        order = wl.free_list_order(num_blocks, seed)
        self.nat = pkv.BlockManager(num_blocks, B, order)
        self.ora = obm.BlockManager(num_blocks, B, order)
        shape = (num_blocks, H, B, D)
        self.k = torch.full(shape, float("nan"), dtype=torch.float16, device=dev)
        self.v = torch.full(shape, float("nan"), dtype=torch.float16, device=dev)
        self.k_ref = np.full(shape, np.nan, dtype=np.float16)
        self.v_ref = np.full(shape, np.nan, dtype=np.float16)
        self.tok_seed = seed * 1000

    def write(self, slots_nat, slots_ora):
        assert list(map(int, slots_nat)) == list(map(int, slots_ora))
        T = len(slots_ora)
        self.tok_seed += 1
        key, value = wl.new_tokens(T, self.H, self.D, self.tok_seed, self.dev)
        pkv.reshape_and_cache(key, value, self.k, self.v, torch.as_tensor(np.asarray(slots_nat), device=self.dev))
        key_h, value_h = wl.new_tokens(T, self.H, self.D, self.tok_seed, "cpu")    # same bits, made on the host
        oracle_cache_ops.reshape_and_cache(key_h.numpy(), value_h.numpy(), self.k_ref, self.v_ref, slots_ora)

    def copy(self, pairs_nat, pairs_ora):
        assert [list(map(int, p)) for p in pairs_nat] == [list(p) for p in pairs_ora]
        if len(pairs_ora):
            pkv.copy_blocks([self.k], [self.v], torch.as_tensor(np.asarray(pairs_nat), device=self.dev))
            oracle_cache_ops.copy_blocks([self.k_ref], [self.v_ref], pairs_ora)

    def append(self, seqs):
        slots, pairs = self.nat.append_slots(seqs)
        ora_slots, ora_pairs = [], []
        for s in seqs:
            slot, src, dst = self.ora.append_slot(s)
            ora_slots.append(slot)
            if src >= 0:
                ora_pairs.append((src, dst))
        self.copy(pairs, ora_pairs)           # the copy runs before the write that needed it
        self.write(slots, ora_slots)

    def pools_equal(self):
        return (np.array_equal(self.k.cpu().numpy().view(np.uint16), self.k_ref.view(np.uint16))
                and np.array_equal(self.v.cpu().numpy().view(np.uint16), self.v_ref.view(np.uint16)))

    def attend(self, seqs):
        max_blocks = max(len(self.ora.block_table(s)[0]) for s in seqs)
        tables, lens = self.nat.block_tables(seqs, max_blocks)
        q = wl.dense_tensor((len(seqs), self.H, self.D), self.seed, wl.STREAM_Q, self.dev)
        out = pkv.paged_attention_decode(q, self.k, self.v, torch.from_numpy(tables).to(self.dev),
                                         torch.from_numpy(lens).to(self.dev), self.D ** -0.5, self.B)
        assert pkv.device_error() == 0
        ref_tables = np.full((len(seqs), max_blocks), -1)
        ref_lens = np.zeros(len(seqs), dtype=np.int64)
        for i, s in enumerate(seqs):
            t, c = self.ora.block_table(s)
            ref_tables[i, :len(t)] = t
            ref_lens[i] = c
        assert np.array_equal(tables, ref_tables) and np.array_equal(lens, ref_lens)
        q_h = wl.dense_tensor((len(seqs), self.H, self.D), self.seed, wl.STREAM_Q, "cpu")
        ref = oracle_attention.paged_decode_attention(q_h.numpy(), self.k_ref, self.v_ref, ref_tables,
                                                      ref_lens, self.D ** -0.5)
        return float(np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)))


@pytest.mark.parametrize("prompt_len", [511, 512, 37])
def test_parallel_sampling_decode(cuda_device, prompt_len):
    H, D, B, n, prompts = 8, 128, 16, 4, 6
    rng = np.random.default_rng(prompt_len)
    x = TwoSides(cuda_device, 1200, H, D, B, seed=1003)
    seqs, tails = [], []
    for p in range(prompts):
        base = p * n
        x.write(x.nat.add_seq(base, prompt_len), x.ora.add_seq(base, prompt_len))
        for i in range(1, n):
            x.nat.fork(base, base + i)
            x.ora.fork(base, base + i)
        seqs += list(range(base, base + n))
        tails += [int(t) for t in rng.integers(1, 41, size=n)]
    for step in range(max(tails)):
        live = [s for s, t in zip(seqs, tails) if t > step]
        x.append(live)
        if step == 0:
            want = prompts * (n - 1) if prompt_len % B else 0
            assert x.ora.cow_copies == want and x.nat.stats()[2] == want
            assert x.pools_equal()
            assert x.attend(seqs) <= ATOL
    assert x.pools_equal()
    assert x.attend(seqs) <= ATOL
    free, waste, copies = x.nat.stats()
    assert free == x.ora.num_free() and waste == x.ora.tail_waste_tokens()


def test_shared_prefix_decode(cuda_device):
    H, D, B = 8, 64, 16
    x = TwoSides(cuda_device, 900, H, D, B, seed=1004)
    prefix_len = 1024 + 5                                   # 64 full blocks + a 5-token block
    x.write(x.nat.register_prefix(0, prefix_len), x.ora.register_prefix(0, prefix_len))
    rng = np.random.default_rng(4)
    seqs = list(range(12))
    suffix = [int(s) for s in rng.integers(1, 40, size=len(seqs))]
    for s in seqs:
        x.nat.add_seq_with_prefix(s, 0)
        x.ora.add_seq_with_prefix(s, 0)
    for step in range(max(suffix)):
        live = [s for s in seqs if suffix[s] > step]
        x.append(live)
    assert x.ora.cow_copies == len(seqs)                    # every request copies the partial prefix block
    assert x.pools_equal()
    assert x.attend(seqs) <= ATOL


@pytest.mark.parametrize("prefix_len", [1024, 1029])
def test_prefix_requests_prompt_phase(cuda_device, prefix_len):
    # [guide] 04: requests map their first blocks onto a cached prefix and run the prompt phase
    # over their own tokens only.  Each request and all its own tokens are placed in one manager
    # call (the copy of a partly filled last prefix block, then the tokens' slots); the tokens'
    # K/V is written, then prefill attention gives each own token attention over the prefix and,
    # causally, the tokens before it; then one decode step.  Pools bit-exact, attention <= 2e-3.
    H, D, B = 4, 128, 16
    x = TwoSides(cuda_device, 1000, H, D, B, seed=1004)
    x.write(x.nat.register_prefix(0, prefix_len), x.ora.register_prefix(0, prefix_len))
    rng = np.random.default_rng(prefix_len)
    seqs = list(range(10))
    suffix = [int(n) for n in rng.integers(1, 300, size=len(seqs))]
    all_nat, all_ora = [], []
    for s, n in zip(seqs, suffix):
        slots, pairs = x.nat.add_seq_with_prefix(s, 0, n)
        ora_slots, ora_pairs = x.ora.add_seq_with_prefix(s, 0, n)
        assert len(ora_pairs) == (1 if prefix_len % B else 0)
        x.copy(pairs, ora_pairs)                      # the copy runs before the request's writes
        all_nat += list(slots)
        all_ora += ora_slots
    x.write(all_nat, all_ora)                         # every request's own tokens in one call
    assert x.pools_equal()
    # prefill: the own tokens of every request over prefix + causal own tokens
    max_blocks = max(len(x.ora.block_table(s)[0]) for s in seqs)
    tables, lens = x.nat.block_tables(seqs, max_blocks)
    qs = np.concatenate([[0], np.cumsum(suffix)]).astype(np.int32)
    q = wl.dense_tensor((int(qs[-1]), H, D), 55, wl.STREAM_Q, cuda_device)
    out = pkv.paged_attention_prefill(q, x.k, x.v, torch.from_numpy(tables).to(cuda_device),
                                      torch.from_numpy(lens).to(cuda_device), torch.from_numpy(qs).to(cuda_device),
                                      D ** -0.5, B, max(suffix))
    assert pkv.device_error() == 0
    ref = oracle_attention.paged_prefill_attention(q.cpu().numpy().astype(np.float64), x.k_ref, x.v_ref, tables,
                                                   lens, qs, D ** -0.5)
    assert float(np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref))) <= ATOL
    x.append(seqs)                                    # then a decode step on top
    assert x.pools_equal()
    assert x.attend(seqs) <= ATOL


@pytest.mark.parametrize("width,B", [(4, 16), (6, 8)])
def test_beam_search_decode(cuda_device, width, B):
    # a beam step forks the survivors, retires the old beam and appends one token per candidate;
    # the one-block copies run through copy_blocks before the writes
    H, D, requests = 4, 128, 3
    rng = np.random.default_rng(width)
    x = TwoSides(cuda_device, 600, H, D, B, seed=2000 + width)
    beams, nid = [], 0
    for r in range(requests):
        n = int(rng.integers(20, 90))
        x.write(x.nat.add_seq(nid, n), x.ora.add_seq(nid, n))
        beams.append([nid])
        nid += 1
    copies = 0
    for step in range(40):
        for r in range(requests):
            parents = [int(p) for p in rng.choice(beams[r], size=width)]
            children = list(range(nid, nid + width))
            nid += width
            slots, pairs = x.nat.beam_step(parents, children, beams[r])
            want = x.ora.beam_step(parents, children, beams[r])
            x.copy(pairs, [(s, d) for _, s, d in want if s >= 0])
            x.write(slots, [w[0] for w in want])
            copies += len(pairs)
            beams[r] = children
    assert copies > 0
    assert x.pools_equal()
    assert x.attend([c for b in beams for c in b]) <= ATOL
