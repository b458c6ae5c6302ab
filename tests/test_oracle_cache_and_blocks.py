"""Pins for the cache-op, size and block-manager oracles.

The block-manager pins are the pages' own worked examples (stored under
tests/golden/ with their citations) plus the invariants the pages state:
at most one partly filled block per sequence, reference counts, n-1 copies
when n sequences share a partly filled block, and the physical-block count
under sharing.
"""
import json
import os

import numpy as np
import pytest

from oracle import block_manager as obm
from oracle import cache_ops as oc
from oracle import sizes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "block_manager_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _free_order(n, head):
    rest = [b for b in range(n) if b not in head]
    return list(head) + rest


# ---- sizes --------------------------------------------------------------------------------

def test_kv_bytes_per_token_matches_page():
    g = _golden()["kv_size"]
    heads, head_dim = 40, 128
    assert heads * head_dim == g["hidden"]
    per_token = sizes.kv_bytes_per_token(g["num_layers"], heads, head_dim, g["dtype_bytes"])
    assert per_token == 2 * 5120 * 40 * 2 == 819200
    assert 780_000 <= per_token <= 820_000                          # "about 800 KB"
    req = per_token * g["max_tokens"]
    assert 1.55e9 <= req <= 1.75e9                                   # "about 1.6 GB"


def test_block_bytes():
    assert sizes.kv_bytes_per_block(40, 128, 16) * 2 == 16 * sizes.kv_bytes_per_token(1, 40, 128)


# ---- cache ops ----------------------------------------------------------------------------

def test_reshape_and_cache_places_rows_and_skips_padding():
    rng = np.random.default_rng(1)
    N, H, B, D, T = 6, 3, 4, 8, 7
    k = rng.standard_normal((N, H, B, D)).astype(np.float16)
    v = rng.standard_normal((N, H, B, D)).astype(np.float16)
    k0, v0 = k.copy(), v.copy()
    key = rng.standard_normal((T, H, D)).astype(np.float16)
    val = rng.standard_normal((T, H, D)).astype(np.float16)
    slots = [5, -1, 0, 23, 13, -7, 8]
    oc.reshape_and_cache(key, val, k, v, slots)
    # read back through the flat-slot view: pool[n, h, r, :] is slot n*B + r of head h
    flat_k = k.transpose(1, 0, 2, 3).reshape(H, N * B, D)
    flat_v = v.transpose(1, 0, 2, 3).reshape(H, N * B, D)
    written = set()
    for t, s in enumerate(slots):
        if s >= 0:
            np.testing.assert_array_equal(flat_k[:, s], key[t])
            np.testing.assert_array_equal(flat_v[:, s], val[t])
            written.add(s)
    untouched = [s for s in range(N * B) if s not in written]
    f0k = k0.transpose(1, 0, 2, 3).reshape(H, N * B, D)
    np.testing.assert_array_equal(flat_k[:, untouched], f0k[:, untouched])


def test_copy_blocks_copies_every_layer_and_nothing_else():
    rng = np.random.default_rng(2)
    L, N, H, B, D = 3, 8, 2, 4, 8
    ks = [rng.standard_normal((N, H, B, D)).astype(np.float16) for _ in range(L)]
    vs = [rng.standard_normal((N, H, B, D)).astype(np.float16) for _ in range(L)]
    before_k = [x.copy() for x in ks]
    before_v = [x.copy() for x in vs]
    pairs = [(1, 5), (2, 7), (0, 3)]
    oc.copy_blocks(ks, vs, pairs)
    for layer in range(L):
        for src, dst in pairs:
            np.testing.assert_array_equal(ks[layer][dst], before_k[layer][src])
            np.testing.assert_array_equal(vs[layer][dst], before_v[layer][src])
        for b in (0, 1, 2, 4, 6):
            np.testing.assert_array_equal(ks[layer][b], before_k[layer][b])
            np.testing.assert_array_equal(vs[layer][b], before_v[layer][b])


# ---- block manager: the pages' worked examples --------------------------------------------

def test_single_request_walkthrough():
    g = _golden()["single_request"]
    B = g["block_size"]
    bm = obm.BlockManager(16, B, _free_order(16, g["free_order_head"]))
    slots = bm.add_seq(0, len(g["prompt"]))
    table, ctx = bm.block_table(0)
    assert len(table) == g["after_prefill"]["num_logical_blocks"]
    assert bm.filled(0) == g["after_prefill"]["filled"]
    assert table == g["after_prefill"]["table"]
    assert table[0] == 7                                              # logical 0 -> physical 7
    assert slots == [7 * B + r for r in range(4)] + [1 * B + r for r in range(3)]
    for step in g["decode"]:
        slot, src, dst = bm.append_slot(0)
        assert (src, dst) == (-1, -1)
        assert bm.filled(0) == step["filled"]
        assert len(bm.block_table(0)[0]) == step["num_logical_blocks"]
    # "fathers" went to the reserved slot of block 1, "brought" to row 0 of the new block
    table, ctx = bm.block_table(0)
    assert ctx == 9 and table[2] == 3 and slot == 3 * B


def test_parallel_sampling_copy_on_write():
    g = _golden()["parallel_sampling"]
    B = g["block_size"]
    bm = obm.BlockManager(16, B, _free_order(16, g["free_order_head"]))
    bm.add_seq(1, g["prompt_len"])                                    # A1
    bm.fork(1, 2)                                                     # A2 shares A1's blocks
    assert bm.block_table(1)[0] == g["after_prefill"]["A1"]
    assert bm.block_table(2)[0] == g["after_prefill"]["A2"]
    for b, r in g["after_prefill"]["ref"].items():
        assert bm.ref_count(int(b)) == r
    slot, src, dst = bm.append_slot(1)                                # A1 writes "fathers"
    step = g["A1_writes_first"]
    assert [src, dst] == step["copy"]
    assert bm.block_table(1)[0] == step["A1"] and bm.block_table(2)[0] == step["A2"]
    for b, r in step["ref"].items():
        assert bm.ref_count(int(b)) == r
    assert slot == 3 * B + 3
    slot, src, dst = bm.append_slot(2)                                # A2 writes "mothers" in place
    assert (src, dst) == (-1, -1) and g["A2_writes_next"]["copy"] is None
    assert bm.block_table(2)[0] == g["A2_writes_next"]["A2"] and slot == 1 * B + 3


# ---- block manager: invariants the pages state ---------------------------------------------

def _random_ops(bm, rng, steps, max_prompt=40):
    live = []
    next_id = 0
    copies = []
    for _ in range(steps):
        op = rng.integers(0, 10)
        try:
            if op < 2 or not live:
                bm.add_seq(next_id, int(rng.integers(1, max_prompt)))
                live.append(next_id)
                next_id += 1
            elif op < 3:
                bm.fork(int(rng.choice(live)), next_id)
                live.append(next_id)
                next_id += 1
            elif op < 4 and len(live) > 1:
                s = int(rng.choice(live))
                bm.free(s)
                live.remove(s)
            else:
                s = int(rng.choice(live))
                slot, src, dst = bm.append_slot(s)
                if src >= 0:
                    copies.append((src, dst))
        except MemoryError:
            pass
    return live, copies


@pytest.mark.parametrize("B", [1, 4, 16])
def test_at_most_one_partial_block_and_counts_consistent(B):
    rng = np.random.default_rng(B)
    bm = obm.BlockManager(200, B, rng.permutation(200))
    live, _ = _random_ops(bm, rng, 600)
    refs = np.zeros(200, dtype=int)
    for s in live:
        table, ctx = bm.block_table(s)
        filled = bm.filled(s)
        assert all(f == B for f in filled[:-1]) and 1 <= filled[-1] <= B   # one partial block at most
        assert 0 <= B * len(table) - ctx < B                                 # 0 <= tail waste < B
        for b in table:
            refs[b] += 1
    for b in range(200):
        assert bm.ref_count(b) == refs[b]
    assert bm.num_free() == int((refs == 0).sum())


def test_n_sharers_of_a_partial_block_make_n_minus_1_copies():
    B, n = 16, 4
    bm = obm.BlockManager(64, B)
    bm.add_seq(0, 511)                                 # 31 full blocks + one 15-token block
    for i in range(1, n):
        bm.fork(0, i)
    last = bm.block_table(0)[0][-1]
    copies = [bm.append_slot(i)[1:] for i in range(n)]
    made = [c for c in copies if c[0] >= 0]
    assert len(made) == n - 1 and all(c[0] == last for c in made)
    assert bm.ref_count(last) == 1 and copies[-1] == (-1, -1)


def test_full_shared_last_block_needs_no_copy():
    bm = obm.BlockManager(64, 16)
    bm.add_seq(0, 512)
    for i in range(1, 4):
        bm.fork(0, i)
    assert all(bm.append_slot(i)[1] == -1 for i in range(4))
    assert bm.cow_copies == 0


def test_physical_block_count_under_sharing():
    # N_physical = sum_r ceil(L_r / B) - (references saved by sharing)
    B, prompts, n = 16, 5, 4
    rng = np.random.default_rng(4)
    bm = obm.BlockManager(4096, B, rng.permutation(4096))
    lens = {}
    sid = 0
    for p in range(prompts):
        base = sid
        bm.add_seq(base, 512)
        for i in range(1, n):
            bm.fork(base, base + i)
        for i in range(n):
            for _ in range(int(rng.integers(1, 257))):
                bm.append_slot(base + i)
        sid += n
    total_logical = 0
    saved = 0
    for s in range(sid):
        table, ctx = bm.block_table(s)
        assert len(table) == -(-ctx // B)
        total_logical += len(table)
    for b in range(4096):
        if bm.ref_count(b) > 1:
            saved += bm.ref_count(b) - 1
    assert 4096 - bm.num_free() == total_logical - saved
    assert saved == prompts * (n - 1) * 32


def test_shared_prefix_last_block_is_copy_on_write():
    B = 16
    bm = obm.BlockManager(256, B)
    pre_slots = bm.register_prefix(9, 40)                  # 2 full blocks + 8 tokens
    assert len(pre_slots) == 40
    table_p = [s // B for s in pre_slots[::B]]
    bm.add_seq_with_prefix(1, 9)
    bm.add_seq_with_prefix(2, 9)
    assert bm.ref_count(table_p[2]) == 3
    slot, src, dst = bm.append_slot(1)
    assert src == table_p[2] and dst >= 0 and slot == dst * B + 8
    slot, src, dst = bm.append_slot(2)
    assert src == table_p[2]                                # the provider still holds the original
    assert bm.ref_count(table_p[2]) == 1
    bm.free(1)
    bm.free(2)
    bm.drop_prefix(9)
    assert bm.num_free() == 256


def test_extend_places_the_walkthrough_decode_tokens_at_once():
    # the single-request walk-through: after the 7-token prompt (blocks 7 and 1, fills 4 and 3),
    # "fathers" fills logical block 1 and "brought" opens a third block; placing both tokens in
    # one call gives the same slots and fills
    g = _golden()["single_request"]
    B = g["block_size"]
    bm = obm.BlockManager(8, B, _free_order(8, g["free_order_head"]))
    bm.add_seq(0, len(g["prompt"]))
    slots, copies = bm.extend(0, len(g["decode"]))
    third = g["free_order_head"][2]
    assert slots == [g["after_prefill"]["table"][1] * B + 3, third * B + 0] and copies == []
    assert bm.filled(0) == g["decode"][-1]["filled"]
    assert len(bm.block_table(0)[0]) == g["decode"][-1]["num_logical_blocks"]


@pytest.mark.parametrize("prefix_len,suffix", [(1024, 300), (1029, 300), (1029, 3), (40, 0), (7, 9)])
def test_prefix_request_places_its_suffix(prefix_len, suffix):
    # [guide] 04, steps 2 and 4: the request maps its first logical blocks onto the cached prefix
    # and its prompt phase covers only its own tokens; a partly filled last prefix block is
    # copied once, before the first own token is written into it
    B, N = 16, 256
    bm = obm.BlockManager(N, B)
    pre = bm.register_prefix(0, prefix_len)
    free0 = bm.num_free()
    slots, copies = bm.add_seq_with_prefix(1, 0, suffix)
    table, ctx = bm.block_table(1)
    assert ctx == prefix_len + suffix and len(slots) == suffix == len(set(slots))
    assert len(table) == -(-ctx // B)                       # blocks for exactly ctx tokens
    partial = prefix_len % B != 0
    assert len(copies) == (1 if partial and suffix > 0 else 0)
    if copies:
        assert copies[0] == (pre[-1] // B, table[prefix_len // B])
    shared = prefix_len // B + (1 if partial and suffix == 0 else 0)
    assert [b for b in table[:shared]] == [x // B for x in pre[::B]][:shared]
    assert free0 - bm.num_free() == len(table) - shared        # blocks taken = blocks not shared
    # each own token sits at its position: row (p mod B) of the table's block p / B
    for i, sl in enumerate(slots):
        p_ = prefix_len + i
        assert sl == table[p_ // B] * B + p_ % B
    assert bm.filled(1)[:-1] == [B] * (len(table) - 1)          # at most one partly filled block


def test_extend_is_all_or_nothing():
    bm = obm.BlockManager(4, 4, [0, 1, 2, 3])
    bm.add_seq(0, 3)
    bm.fork(0, 1)
    with pytest.raises(MemoryError):
        bm.extend(1, 14)                                    # copy + 3 new blocks > 3 free
    assert bm.filled(1) == [3] and bm.ref_count(0) == 2 and bm.num_free() == 3
    bm.register_prefix(7, 2)                                # block 1
    with pytest.raises(MemoryError):
        bm.add_seq_with_prefix(2, 7, 11)                    # copy + 3 new blocks > 2 free
    assert 2 not in bm.seqs and bm.ref_count(1) == 1 and bm.prefix_seqs == 0


def test_full_prefix_blocks_shared_without_copy():
    bm = obm.BlockManager(256, 16)
    bm.register_prefix(0, 1024)
    for s in range(8):
        bm.add_seq_with_prefix(s, 0)
        bm.append_slot(s)
    assert bm.cow_copies == 0 and bm.num_free() == 256 - 64 - 8


def test_out_of_blocks_changes_nothing():
    bm = obm.BlockManager(4, 4)
    bm.add_seq(0, 13)                                       # 4 blocks
    with pytest.raises(MemoryError):
        bm.add_seq(1, 1)
    assert 1 not in bm.seqs
    bm.fork(0, 1)
    with pytest.raises(MemoryError):
        bm.append_slot(1)                                   # needs a copy of the shared 1-token block
    assert bm.block_table(1)[0] == bm.block_table(0)[0] and bm.filled(1)[-1] == 1


def test_free_returns_blocks_only_when_unreferenced():
    bm = obm.BlockManager(32, 4, list(range(32)))
    bm.add_seq(0, 8)                                        # blocks 0, 1
    bm.fork(0, 1)
    bm.append_slot(1)                                       # full -> new block 2 for seq 1
    bm.free(0)
    assert bm.num_free() == 29 and bm.ref_count(0) == 1
    bm.free(1)
    assert bm.num_free() == 32
    assert list(bm.free_list)[-3:] == [0, 1, 2]              # FIFO: freed blocks go to the back


# ---- beam search ----------------------------------------------------------------------------

def _beam_tree(bm):
    """The figure's tree: with B = 1, ids are taken in the order 0..8 of the figure."""
    c0, c1, c2, c3 = 10, 11, 12, 13
    bm.add_seq(c0, 1)               # block 0
    bm.fork(c0, c3)
    bm.append_slot(c0)              # block 1
    bm.append_slot(c3)              # block 2
    bm.append_slot(c0)              # block 3
    bm.append_slot(c3)              # block 4
    bm.fork(c0, c1)
    bm.fork(c0, c2)
    for c in (c0, c1, c2, c3):      # blocks 5, 6, 7, 8
        bm.append_slot(c)
    return {"cand0": c0, "cand1": c1, "cand2": c2, "cand3": c3}


def test_beam_search_walkthrough():
    g = _golden()["beam_search"]
    bm = obm.BlockManager(32, g["block_size"])
    ids = _beam_tree(bm)
    for name, lineage in g["lineages_before"].items():
        assert bm.block_table(ids[name])[0] == lineage
    new = [20, 21, 22, 23]
    out = bm.beam_step([ids[p] for p in g["step"]["parents"]], new, [ids[r] for r in g["step"]["retire"]])
    assert all(src == -1 for _, src, _ in out)                       # B = 1: every token opens a block
    for i, (name, lineage) in enumerate(g["lineages_after"].items()):
        assert bm.block_table(new[i])[0] == lineage
    assert list(bm.free_list)[-4:] == g["freed_in_order"]
    for b, r in g["ref_after"].items():
        assert bm.ref_count(int(b)) == r


def test_beam_step_copies_one_block_per_extra_sibling():
    B = 16
    bm = obm.BlockManager(64, B)
    bm.add_seq(0, 40)                                                 # last block holds 8 tokens
    bm.fork(0, 1)
    out = bm.beam_step([0, 0, 0, 1], [2, 3, 4, 5], [0, 1])
    copies = [(s, d) for _, s, d in out if s >= 0]
    # four candidates now share the partial block: three copy it, the last writes in place
    assert len(copies) == 3 and all(s == bm.block_table(5)[0][-1] for s, _ in copies)
    assert bm.ref_count(bm.block_table(5)[0][0]) == 4


def test_beam_step_all_or_nothing():
    bm = obm.BlockManager(4, 4)
    bm.add_seq(0, 6)                                                  # 2 blocks, last has 2 tokens
    before = (list(bm.free_list), dict(bm.seqs))
    with pytest.raises(MemoryError):
        bm.beam_step([0, 0, 0, 0], [1, 2, 3, 4], [0])                 # needs 3 copies, 2 free
    assert list(bm.free_list) == before[0] and set(bm.seqs) == {0}
    out = bm.beam_step([0, 0, 0], [1, 2, 3], [0])                    # needs 2 copies: fits
    assert sum(1 for _, s, _ in out if s >= 0) == 2 and bm.num_free() == 0


def test_swap_out_and_back_restores_blocks():
    rng = np.random.default_rng(8)
    L, N, M, H, B, D = 2, 10, 6, 2, 4, 8
    dev_k = [rng.standard_normal((N, H, B, D)).astype(np.float16) for _ in range(L)]
    dev_v = [rng.standard_normal((N, H, B, D)).astype(np.float16) for _ in range(L)]
    orig_k = [x.copy() for x in dev_k]
    host_k = [np.zeros((M, H, B, D), np.float16) for _ in range(L)]
    host_v = [np.zeros((M, H, B, D), np.float16) for _ in range(L)]
    out_map = [(3, 0), (7, 1), (9, 2)]
    oc.swap_blocks(dev_k, dev_v, host_k, host_v, out_map)
    for layer in range(L):
        for s, d in out_map:
            np.testing.assert_array_equal(host_k[layer][d], dev_k[layer][s])
            np.testing.assert_array_equal(host_v[layer][d], dev_v[layer][s])
        np.testing.assert_array_equal(host_k[layer][3:], 0)
    for layer in range(L):                      # the device blocks are reused meanwhile
        dev_k[layer][[3, 7, 9]] = 0
    back_map = [(0, 1), (1, 4), (2, 5)]         # swapped back in, into other free blocks
    oc.swap_blocks(host_k, host_v, dev_k, dev_v, back_map)
    for layer in range(L):
        for (s0, _), (_, d1) in zip(out_map, back_map):
            np.testing.assert_array_equal(dev_k[layer][d1], orig_k[layer][s0])


# -- swapping a preempted group between two managers ([lecture] 调度和抢占; [guide] 05) ----------
def _layout(bm, seqs):
    """Each sequence's fills, and which (sequence, logical block) positions share a physical block:
    everything of the state that does not depend on physical ids."""
    fills = {s: bm.filled(s) for s in seqs}
    where = {}
    for s in seqs:
        for j, phys in enumerate(bm.block_table(s)[0]):
            where.setdefault(phys, []).append((s, j))
    classes = sorted(sorted(v) for v in where.values())
    refs = sorted((sorted(v), bm.ref_count(p)) for p, v in where.items())
    return fills, classes, refs


def _request_group(bm, first_id, prompt_len, n):
    """A request's n samples: one prompt, n-1 forks, one appended token each (copy-on-write)."""
    bm.add_seq(first_id, prompt_len)
    for i in range(1, n):
        bm.fork(first_id, first_id + i)
    for i in range(n):
        bm.append_slot(first_id + i)
    return list(range(first_id, first_id + n))


def test_group_swap_round_trip_keeps_layout_and_sharing():
    dev = obm.BlockManager(40, 4, list(np.random.default_rng(3).permutation(40)))
    host = obm.BlockManager(30, 4, list(np.random.default_rng(4).permutation(30)))
    group = _request_group(dev, 0, 10, 4)                  # 3 blocks: 2 shared full, 1 shared partial + copies
    other = _request_group(dev, 10, 6, 2)                  # stays on the device
    before = _layout(dev, group)
    other_before = [dev.block_table(s) for s in other]
    distinct = {p for s in group for p in dev.block_table(s)[0]}
    free_dev, free_host = dev.num_free(), host.num_free()
    pairs = obm.swap(dev, host, group)
    # one move per distinct block, each side's blocks distinct, the sources exactly the group's blocks
    assert len(pairs) == len(distinct)
    assert {s for s, _ in pairs} == distinct and len({d for _, d in pairs}) == len(pairs)
    assert dev.num_free() == free_dev + len(pairs) and host.num_free() == free_host - len(pairs)
    assert all(s not in dev.seqs for s in group) and _layout(host, group) == before
    assert all(dev.ref_count(s) == 0 for s, _ in pairs)
    assert [dev.block_table(s) for s in other] == other_before
    # the freed device blocks are reused meanwhile; the group comes back into other blocks
    dev.add_seq(99, 4 * len(pairs))
    back = obm.swap(host, dev, group)
    assert len(back) == len(pairs) and _layout(dev, group) == before
    assert host.num_free() == free_host and not host.seqs
    # a moved block is the same block: the pairs compose to a map from old to new device ids
    old_to_new = {s0: d1 for (s0, h0) in pairs for (h1, d1) in back if h0 == h1}
    assert len(old_to_new) == len(pairs)


def test_group_swap_keeps_copy_on_write_pending():
    # two samples share a partly filled last block when swapped; after coming back, the first to
    # write still copies it and the second writes in place
    dev = obm.BlockManager(16, 4)
    host = obm.BlockManager(16, 4)
    dev.add_seq(0, 6)
    dev.fork(0, 1)
    obm.swap(dev, host, [0, 1])
    obm.swap(host, dev, [0, 1])
    last = dev.block_table(0)[0][-1]
    assert dev.ref_count(last) == 2
    _, src, dst = dev.append_slot(0)
    assert src == last and dst >= 0
    assert dev.append_slot(1)[1:] == (-1, -1)


def test_group_swap_refuses_a_block_held_outside_the_group():
    dev = obm.BlockManager(16, 4)
    host = obm.BlockManager(16, 4)
    dev.add_seq(0, 6)
    dev.fork(0, 1)
    pid_slots = dev.register_prefix(7, 8)
    dev.add_seq_with_prefix(2, 7)
    state = (list(dev.free_list), {s: dev.block_table(s) for s in dev.seqs}, list(dev.ref))
    with pytest.raises(ValueError):
        obm.swap(dev, host, [0])                           # its sibling holds the same blocks
    with pytest.raises(ValueError):
        obm.swap(dev, host, [2])                           # the registered prefix holds its blocks
    with pytest.raises(ValueError):
        obm.swap(dev, host, [0, 0, 1])
    with pytest.raises(KeyError):
        obm.swap(dev, host, [0, 1, 5])
    assert state == (list(dev.free_list), {s: dev.block_table(s) for s in dev.seqs}, list(dev.ref))
    assert host.num_free() == 16 and not host.seqs and len(pid_slots) == 8


def test_group_swap_out_of_blocks_changes_nothing():
    dev = obm.BlockManager(16, 4)
    host = obm.BlockManager(2, 4)
    dev.add_seq(0, 9)                                      # 3 blocks, the host has 2
    state = (list(dev.free_list), dev.block_table(0), list(dev.ref))
    with pytest.raises(MemoryError):
        obm.swap(dev, host, [0])
    assert state == (list(dev.free_list), dev.block_table(0), list(dev.ref))
    assert host.num_free() == 2 and not host.seqs


def test_observability_counts():
    # the reference-count histogram is a partition of the pool, and the counters count events
    bm = obm.BlockManager(32, 4)
    host = obm.BlockManager(16, 4)
    bm.register_prefix(1, 8)                               # 2 blocks held by the prefix
    for s in range(3):
        bm.add_seq_with_prefix(s, 1)                       # 3 sequences x 2 prefix blocks
    bm.add_seq(10, 6)
    bm.fork(10, 11)
    bm.append_slot(10)                                     # copies the shared partial block
    hist = bm.ref_histogram(8)
    assert sum(hist) == 32 and hist[0] == bm.num_free()
    assert hist[4] == 2                                    # the prefix blocks: prefix + 3 sequences
    assert hist[2] == 1 and hist[1] == 2                   # 10/11's full block; 11's partial and 10's copy
    c = bm.counters()
    assert (c["prefix_seqs"], c["prefix_blocks"], c["cow_copies"]) == (3, 6, 1)
    obm.swap(bm, host, [10, 11])
    assert bm.counters()["groups_out"] == 1 and bm.counters()["blocks_out"] == 3
    assert host.counters()["groups_in"] == 1 and host.counters()["blocks_in"] == 3
    assert bm.ref_histogram(3)[2] == 2                     # counts >= 2 fold into the last entry
