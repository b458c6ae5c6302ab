"""Host logic of the bench's shared-prefix grouping: groups of consecutive sequences whose leading
blocks are the same physical blocks, and each group's shared whole-block prefix length (CPU)."""
import numpy as np

import bench
from paged_kv_cache_73_gb300 import workloads as wl


def test_one_shared_prefix_group():
    w = wl.shared_prefix(seed=1004, requests=12, suffix_lo=32, suffix_hi=300)
    starts, prefixes = bench.shared_prefix_groups(w.block_tables, w.context_lens, w.block_size)
    assert starts.tolist() == [0, 12] and prefixes.tolist() == [1024]


def test_prompt_groups_of_parallel_sampling():
    for prompt, shared in ((512, 512), (511, 496)):
        w = wl.parallel_sampling(prompt_len=prompt)
        starts, prefixes = bench.shared_prefix_groups(w.block_tables, w.context_lens, w.block_size)
        assert starts.tolist() == list(range(0, w.num_seqs + 1, 4))
        assert set(prefixes.tolist()) == {shared}


def test_independent_sequences_share_nothing():
    w = wl.custom(3, [40, 17, 100], 2, 64, 16)
    starts, prefixes = bench.shared_prefix_groups(w.block_tables, w.context_lens, w.block_size)
    assert starts.tolist() == [0, 1, 2, 3] and prefixes.tolist() == [0, 0, 0]


def test_prefix_capped_at_the_shortest_members_full_blocks():
    # two sequences mapping the same four blocks, one only 40 tokens long: 2 full blocks shared
    B = 16
    tables = np.array([[5, 6, 7, 8], [5, 6, 7, -1]], dtype=np.int32)
    lens = np.array([64, 40], dtype=np.int32)
    starts, prefixes = bench.shared_prefix_groups(tables, lens, B)
    assert starts.tolist() == [0, 2] and prefixes.tolist() == [32]


def test_block_manager_summary_of_the_step_batches():
    # the bench's batches as the block manager built them: parallel sampling with 511-token prompts
    # makes 3 copies per prompt (96) and keeps each prompt's 31 full blocks shared by its 4 samples;
    # the shared prefix's 64 blocks are held by the prefix and all 256 requests
    x = bench.build_step_inputs(1003, "parallel_sampling_cow")["bm"]
    assert x["cow_copies"] == 96 and x["ref_histogram"][4] == 32 * 31
    y = bench.build_step_inputs(1004, "shared_prefix")["bm"]
    assert (y["prefix_seqs"], y["prefix_blocks"]) == (256, 256 * 64) and y["ref_histogram"][7] == 64
    z = bench.build_step_inputs(1002, "opt13b")["bm"]
    assert z["cow_copies"] == 0 and sum(z["ref_histogram"][2:]) == 0
    assert z["ref_histogram"][0] == z["free_blocks"]
