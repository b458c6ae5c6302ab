"""The two cache-maintenance operations around decode attention, as host loops.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[note] section "关键设计 5：Kernel 级优化" names three fused kernels; two of
them move bytes and nothing else:

* "fused reshape and block write": each new token's key/value rows are
  rearranged into the block layout and stored at their slot;
* "fused block copy": the many small copies that copy-on-write triggers are
  done as one batch.

Both are defined by where bytes go, so the oracle is a plain loop over the
index formulas; results are compared byte for byte.

Readings where the pages are silent:

* slot = physical_block * B + row, the slot numbering a block table implies;
* a negative slot marks a padding token that is not stored;
* a copy (src, dst) copies the whole block, every head and every row,
  including rows past the last filled token.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


def reshape_and_cache(key: np.ndarray, value: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                      slot_mapping: Sequence[int]) -> None:
    """Store key[t], value[t] ([H, D] each) at slot_mapping[t], in place.

    The pools are [N, H, B, D]; slot s is row s % B of block s // B.
    """
    B = k_cache.shape[2]
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        block, row = divmod(slot, B)
        for h in range(key.shape[1]):
            k_cache[block, h, row, :] = key[t, h, :]
            v_cache[block, h, row, :] = value[t, h, :]


def copy_blocks(k_caches: Sequence[np.ndarray], v_caches: Sequence[np.ndarray],
                block_mapping: Sequence[Sequence[int]]) -> None:
    """For every (src, dst) pair and every layer: block dst becomes a copy of block src."""
    for src, dst in block_mapping:
        for k_cache, v_cache in zip(k_caches, v_caches):
            k_cache[int(dst)] = k_cache[int(src)]
            v_cache[int(dst)] = v_cache[int(src)]


def swap_blocks(src_k: Sequence[np.ndarray], src_v: Sequence[np.ndarray], dst_k: Sequence[np.ndarray],
                dst_v: Sequence[np.ndarray], block_mapping: Sequence[Sequence[int]]) -> None:
    """Swapping ([lecture] 调度和抢占, Swapping; [guide] 05): for every (src, dst) pair and layer,
    block dst of the destination pools becomes a copy of block src of the source pools (the two
    sides are different pools, e.g. GPU memory and CPU memory)."""
    for src, dst in block_mapping:
        for sk, sv, dk, dv in zip(src_k, src_v, dst_k, dst_v):
            dk[int(dst)] = sk[int(src)]
            dv[int(dst)] = sv[int(src)]
