"""The C++ block manager (libpkv.so) against the oracle's, on the pages' examples
and on long random operation sequences: identical slots, copies, tables,
reference counts and statistics after every step."""
import json
import os

import numpy as np
import pytest

from oracle import block_manager as obm
from paged_kv_cache_73_gb300 import _build
from paged_kv_cache_73_gb300 import binding as pkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "block_manager_examples.json")


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.load()


def _free_order(n, head):
    return list(head) + [b for b in range(n) if b not in head]


def test_pages_single_request_example():
    g = json.load(open(GOLDEN))["single_request"]
    B = g["block_size"]
    bm = pkv.BlockManager(16, B, _free_order(16, g["free_order_head"]))
    slots = bm.add_seq(0, len(g["prompt"]))
    table, ctx = bm.block_table(0)
    assert table == g["after_prefill"]["table"] and ctx == 7
    assert list(slots) == [7 * B + r for r in range(4)] + [1 * B + r for r in range(3)]
    for step, n_tokens in zip(g["decode"], (8, 9)):
        slot, src, dst = bm.append_slot(0)
        assert (src, dst) == (-1, -1)
        table, ctx = bm.block_table(0)
        assert len(table) == step["num_logical_blocks"] and ctx == n_tokens
    assert table[2] == 3 and slot == 3 * B
    free, waste, copies = bm.stats()
    assert (free, waste, copies) == (13, 3, 0)


def test_pages_parallel_sampling_example():
    g = json.load(open(GOLDEN))["parallel_sampling"]
    B = g["block_size"]
    bm = pkv.BlockManager(16, B, _free_order(16, g["free_order_head"]))
    bm.add_seq(1, g["prompt_len"])
    bm.fork(1, 2)
    for b, r in g["after_prefill"]["ref"].items():
        assert bm.ref_count(int(b)) == r
    slot, src, dst = bm.append_slot(1)
    assert [src, dst] == g["A1_writes_first"]["copy"] and slot == 3 * B + 3
    for b, r in g["A1_writes_first"]["ref"].items():
        assert bm.ref_count(int(b)) == r
    slot, src, dst = bm.append_slot(2)
    assert (src, dst) == (-1, -1) and slot == 1 * B + 3
    assert bm.block_table(2)[0] == g["A2_writes_next"]["A2"]


def _compare(nat, ora, live, num_blocks):
    for s in live:
        assert nat.block_table(s) == ora.block_table(s)
    for b in range(num_blocks):
        assert nat.ref_count(b) == ora.ref_count(b)
    free, waste, copies = nat.stats()
    assert (free, waste, copies) == (ora.num_free(), ora.tail_waste_tokens(), ora.cow_copies)
    assert nat.ref_histogram(6).tolist() == ora.ref_histogram(6)
    assert nat.counters() == ora.counters()


@pytest.mark.parametrize("B,N,seed", [(4, 64, 0), (16, 300, 1), (8, 40, 2), (1, 50, 3)])
def test_random_operations_match_oracle(B, N, seed):
    rng = np.random.default_rng(seed)
    order = rng.permutation(N)
    nat = pkv.BlockManager(N, B, order)
    ora = obm.BlockManager(N, B, order)
    live, prefixes = [], []
    nid = 0
    for step in range(1500):
        op = int(rng.integers(0, 15))
        try:
            if op < 2 or not live:
                n = int(rng.integers(1, 5 * B))
                try:
                    want = ora.add_seq(nid, n)
                except MemoryError:
                    with pytest.raises(pkv.PkvOutOfBlocks):
                        nat.add_seq(nid, n)
                    continue
                assert list(nat.add_seq(nid, n)) == want
                live.append(nid)
                nid += 1
            elif op < 4:
                p = int(rng.choice(live))
                ora.fork(p, nid)
                nat.fork(p, nid)
                live.append(nid)
                nid += 1
            elif op < 5 and len(live) > 1:
                s = int(rng.choice(live))
                ora.free(s)
                nat.free(s)
                live.remove(s)
            elif op < 6:
                pid = 1000 + step
                try:
                    want = ora.register_prefix(pid, int(rng.integers(1, 3 * B)))
                except MemoryError:
                    continue
                got = nat.register_prefix(pid, len(want))
                assert list(got) == want
                prefixes.append(pid)
            elif op < 7 and prefixes:
                # a request on a prefix, with its suffix placed in the same call (all or nothing)
                pid = int(rng.choice(prefixes))
                suffix = int(rng.integers(0, 3 * B))
                try:
                    want_slots, want_pairs = ora.add_seq_with_prefix(nid, pid, suffix)
                except MemoryError:
                    with pytest.raises(pkv.PkvOutOfBlocks):
                        nat.add_seq_with_prefix(nid, pid, suffix)
                    continue
                got_slots, got_pairs = nat.add_seq_with_prefix(nid, pid, suffix)
                assert list(got_slots) == want_slots and got_pairs.tolist() == [list(p) for p in want_pairs]
                live.append(nid)
                nid += 1
            elif op < 8 and prefixes:
                pid = prefixes.pop(int(rng.integers(0, len(prefixes))))
                ora.drop_prefix(pid)
                nat.drop_prefix(pid)
            elif op < 10:
                # a batch of distinct sequences, all-or-nothing
                k = int(rng.integers(1, min(6, len(live)) + 1))
                batch = [int(x) for x in rng.choice(live, size=k, replace=False)]
                snapshot_free = ora.num_free()
                try:
                    slots, pairs = nat.append_slots(batch)
                except pkv.PkvOutOfBlocks:
                    # the oracle, appending one by one, must also run out somewhere in the batch;
                    # replay on a copy to confirm, leaving the real oracle untouched
                    import copy
                    probe = copy.deepcopy(ora)
                    with pytest.raises(MemoryError):
                        for s in batch:
                            probe.append_slot(s)
                    assert ora.num_free() == snapshot_free
                    continue
                want_pairs = []
                for s, got in zip(batch, slots):
                    slot, src, dst = ora.append_slot(s)
                    assert slot == got
                    if src >= 0:
                        want_pairs.append([src, dst])
                assert pairs.tolist() == want_pairs
            elif op < 11:
                # several tokens of one sequence at once (all or nothing)
                s = int(rng.choice(live))
                n = int(rng.integers(0, 3 * B + 2))
                try:
                    want_slots, want_pairs = ora.extend(s, n)
                except MemoryError:
                    with pytest.raises(pkv.PkvOutOfBlocks):
                        nat.extend(s, n)
                    continue
                got_slots, got_pairs = nat.extend(s, n)
                assert list(got_slots) == want_slots and got_pairs.tolist() == [list(p) for p in want_pairs]
            else:
                s = int(rng.choice(live))
                try:
                    want = ora.append_slot(s)
                except MemoryError:
                    with pytest.raises(pkv.PkvOutOfBlocks):
                        nat.append_slot(s)
                    continue
                assert nat.append_slot(s) == want
        finally:
            pass
        if step % 50 == 0:
            _compare(nat, ora, live, N)
    _compare(nat, ora, live, N)


def test_errors_leave_state_unchanged():
    bm = pkv.BlockManager(4, 4)
    bm.add_seq(0, 13)
    with pytest.raises(pkv.PkvOutOfBlocks):
        bm.add_seq(1, 1)
    bm.fork(0, 1)
    with pytest.raises(pkv.PkvOutOfBlocks):
        bm.append_slot(1)
    assert bm.block_table(1) == bm.block_table(0)
    with pytest.raises(pkv.PkvError):
        bm.fork(0, 1)                         # child exists
    with pytest.raises(pkv.PkvError):
        bm.append_slot(99)                    # unknown sequence
    with pytest.raises(pkv.PkvError):
        bm.append_slots([0, 0])               # listed twice
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(4, 4, [0, 1, 1, 2])  # not a permutation
    assert bm.stats()[0] == 0


def test_extend_and_prefix_suffix_all_or_nothing():
    bm = pkv.BlockManager(6, 4, list(range(6)))
    bm.register_prefix(1, 6)                  # blocks 0 (4 tokens), 1 (2 tokens)
    with pytest.raises(pkv.PkvOutOfBlocks):
        bm.add_seq_with_prefix(2, 1, 15)      # copy of block 1 + 3 new blocks > 4 free
    assert bm.stats()[0] == 4 and bm.ref_count(0) == 1 and bm.ref_count(1) == 1
    with pytest.raises(pkv.PkvError):
        bm.block_table(2)                     # the failed request left no sequence behind
    slots, pairs = bm.add_seq_with_prefix(2, 1, 10)   # copy 1 -> 2, then blocks 3 and 4
    assert pairs.tolist() == [[1, 2]]
    assert slots.tolist() == [2 * 4 + 2, 2 * 4 + 3] + [3 * 4 + r for r in range(4)] + [4 * 4 + r for r in range(4)]
    assert bm.block_table(2) == ([0, 2, 3, 4], 16)
    with pytest.raises(pkv.PkvOutOfBlocks):
        bm.extend(2, 5)                       # 2 new blocks, 1 free
    assert bm.block_table(2) == ([0, 2, 3, 4], 16) and bm.stats()[0] == 1
    slots, pairs = bm.extend(2, 4)
    assert slots.tolist() == [5 * 4 + r for r in range(4)] and pairs.shape == (0, 2)
    assert bm.extend(2, 0)[0].shape == (0,)


def test_batch_tables_padded():
    bm = pkv.BlockManager(32, 4, list(range(32)))
    bm.add_seq(5, 9)
    bm.add_seq(6, 1)
    tables, lens = bm.block_tables([6, 5], 4)
    assert tables.tolist() == [[3, -1, -1, -1], [0, 1, 2, -1]] and lens.tolist() == [1, 9]
    with pytest.raises(pkv.PkvError):
        bm.block_tables([5], 2)


# ---- beam search --------------------------------------------------------------------------------

def _beam_tree(bm):
    c0, c1, c2, c3 = 10, 11, 12, 13
    bm.add_seq(c0, 1)
    bm.fork(c0, c3)
    for c in (c0, c3, c0, c3):
        bm.append_slot(c)
    bm.fork(c0, c1)
    bm.fork(c0, c2)
    for c in (c0, c1, c2, c3):
        bm.append_slot(c)
    return {"cand0": c0, "cand1": c1, "cand2": c2, "cand3": c3}


def test_pages_beam_search_example():
    g = json.load(open(GOLDEN))["beam_search"]
    bm = pkv.BlockManager(32, g["block_size"])
    ids = _beam_tree(bm)
    for name, lineage in g["lineages_before"].items():
        assert bm.block_table(ids[name])[0] == lineage
    new = [20, 21, 22, 23]
    slots, pairs = bm.beam_step([ids[p] for p in g["step"]["parents"]], new, [ids[r] for r in g["step"]["retire"]])
    assert len(pairs) == 0
    for i, lineage in enumerate(g["lineages_after"].values()):
        assert bm.block_table(new[i])[0] == lineage
    assert list(slots) == [9, 10, 11, 12]
    for b, r in g["ref_after"].items():
        assert bm.ref_count(int(b)) == r
    assert bm.stats()[0] == 32 - 9


@pytest.mark.parametrize("B,width,seed", [(16, 4, 0), (16, 6, 1), (4, 4, 2), (1, 3, 3)])
def test_random_beam_search_matches_oracle(B, width, seed):
    rng = np.random.default_rng(seed)
    N = 400
    order = rng.permutation(N)
    nat = pkv.BlockManager(N, B, order)
    ora = obm.BlockManager(N, B, order)
    nat.add_seq(0, 37)
    ora.add_seq(0, 37)
    beam = [0]
    nid = 1
    for step in range(60):
        parents = [int(rng.choice(beam)) for _ in range(width)]
        children = list(range(nid, nid + width))
        nid += width
        try:
            want = ora.beam_step(parents, children, beam)
        except MemoryError:
            with pytest.raises(pkv.PkvOutOfBlocks):
                nat.beam_step(parents, children, beam)
            break
        slots, pairs = nat.beam_step(parents, children, beam)
        assert list(slots) == [w[0] for w in want]
        assert pairs.tolist() == [[w[1], w[2]] for w in want if w[1] >= 0]
        beam = children
        _compare(nat, ora, beam, N)


def test_beam_step_errors_leave_state_unchanged():
    bm = pkv.BlockManager(4, 4)
    bm.add_seq(0, 6)
    with pytest.raises(pkv.PkvOutOfBlocks):
        bm.beam_step([0, 0, 0, 0], [1, 2, 3, 4], [0])
    with pytest.raises(pkv.PkvError):
        bm.beam_step([0], [0], [])                # child exists
    with pytest.raises(pkv.PkvError):
        bm.beam_step([9], [1], [])                # unknown parent
    with pytest.raises(pkv.PkvError):
        bm.beam_step([0], [1], [0, 0])            # retired twice
    assert bm.block_table(0) == ([0, 1], 6) and bm.stats()[0] == 2
    slots, pairs = bm.beam_step([0, 0, 0], [1, 2, 3], [0])
    assert len(pairs) == 2 and bm.stats()[0] == 0


@pytest.mark.parametrize("B,N,M,seed", [(4, 48, 32, 0), (16, 40, 24, 1), (1, 60, 60, 2)])
def test_random_group_swaps_match_oracle(B, N, M, seed):
    # request groups (a prompt and its forks) grow on a device manager, are swapped out whole to a
    # host manager and back: the same moves, tables, reference counts and free lists on both sides
    rng = np.random.default_rng(200 + seed)
    od, oh = rng.permutation(N), rng.permutation(M)
    nat_d, nat_h = pkv.BlockManager(N, B, od), pkv.BlockManager(M, B, oh)
    ora_d, ora_h = obm.BlockManager(N, B, od), obm.BlockManager(M, B, oh)
    on_dev, on_host = [], []
    nid = 0
    swaps = 0
    for step in range(600):
        op = int(rng.integers(0, 6))
        if op == 0 or not (on_dev or on_host):
            n, plen = int(rng.integers(1, 4)), int(rng.integers(1, 4 * B + 1))
            try:
                ora_d.add_seq(nid, plen)
            except MemoryError:
                with pytest.raises(pkv.PkvOutOfBlocks):
                    nat_d.add_seq(nid, plen)
                continue
            nat_d.add_seq(nid, plen)
            for i in range(1, n):
                ora_d.fork(nid, nid + i)
                nat_d.fork(nid, nid + i)
            on_dev.append(list(range(nid, nid + n)))
            nid += n
        elif op in (1, 2) and on_dev:
            g = on_dev[int(rng.integers(0, len(on_dev)))]
            s = int(rng.choice(g))
            try:
                want = ora_d.append_slot(s)
            except MemoryError:
                with pytest.raises(pkv.PkvOutOfBlocks):
                    nat_d.append_slot(s)
                continue
            assert nat_d.append_slot(s) == want
        elif op == 3 and on_dev:
            i = int(rng.integers(0, len(on_dev)))
            try:
                want = obm.swap(ora_d, ora_h, on_dev[i])
            except MemoryError:
                with pytest.raises(pkv.PkvOutOfBlocks):
                    nat_d.swap(nat_h, on_dev[i])
                continue
            assert nat_d.swap(nat_h, on_dev[i]).tolist() == [list(p) for p in want]
            on_host.append(on_dev.pop(i))
            swaps += 1
        elif op == 4 and on_host:
            i = int(rng.integers(0, len(on_host)))
            try:
                want = obm.swap(ora_h, ora_d, on_host[i])
            except MemoryError:
                with pytest.raises(pkv.PkvOutOfBlocks):
                    nat_h.swap(nat_d, on_host[i])
                continue
            assert nat_h.swap(nat_d, on_host[i]).tolist() == [list(p) for p in want]
            on_dev.append(on_host.pop(i))
            swaps += 1
        elif op == 5 and len(on_dev) > 1:
            for s in on_dev.pop(int(rng.integers(0, len(on_dev)))):
                ora_d.free(s)
                nat_d.free(s)
        if step % 25 == 0:
            _compare(nat_d, ora_d, [s for g in on_dev for s in g], N)
            _compare(nat_h, ora_h, [s for g in on_host for s in g], M)
    _compare(nat_d, ora_d, [s for g in on_dev for s in g], N)
    _compare(nat_h, ora_h, [s for g in on_host for s in g], M)
    assert swaps >= 20


def test_group_swap_errors_leave_state_unchanged():
    dev, host = pkv.BlockManager(16, 4), pkv.BlockManager(2, 4)
    dev.add_seq(0, 6)
    dev.fork(0, 1)
    dev.add_seq(2, 9)
    state = ([dev.block_table(s) for s in (0, 1, 2)], dev.stats(), host.stats())
    with pytest.raises(pkv.PkvError):
        dev.swap(host, [0])                             # its sibling holds the same blocks
    with pytest.raises(pkv.PkvOutOfBlocks):
        dev.swap(host, [2])                             # 3 blocks, the host has 2
    with pytest.raises(pkv.PkvError):
        dev.swap(host, [0, 1, 0])
    with pytest.raises(pkv.PkvError):
        dev.swap(dev, [2])
    other = pkv.BlockManager(16, 8)
    with pytest.raises(pkv.PkvError):
        dev.swap(other, [2])                            # block sizes differ
    assert state == ([dev.block_table(s) for s in (0, 1, 2)], dev.stats(), host.stats())
    assert dev.swap(host, [0, 1]).shape == (2, 2)       # the whole group fits
