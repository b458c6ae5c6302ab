"""Single-query (decode) attention over a paged K/V pool, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it computes follows [note] section "关键设计 1：PagedAttention 的块式注意力":

* the first equation there defines, for query i,
  a_ij = exp(q_i.k_j / sqrt(d)) / sum_{t<=i} exp(q_i.k_t / sqrt(d)) and
  o_i = sum_{j<=i} a_ij v_j;
* the second equation splits the keys and values into blocks of B tokens,
  K_j = (k_{(j-1)B+1} .. k_{jB}), and states that o_i is the same sum read block
  by block (the softmax still normalises over all tokens <= i, not per block);
* the prose beneath it says the kernel reaches each logical block through the
  block table's physical id.

Because the paged form reaches exactly the textbook result, this oracle is
that definition written out: gather the sequence's keys and values through
its block table into contiguous arrays, then plain softmax attention.

Readings where the pages are silent:

* pool layout: K and V pools are [num_blocks, num_heads, block_size, head_dim];
  token t of a sequence lives in physical block table[t // B] at row t % B;
* the scale is a parameter (the pages use 1/sqrt(d));
* a sequence with context length 0 attends over nothing: its output is zero;
* the new token is part of its own context (the sum runs to t = i), so
  context_len counts it.
"""
from __future__ import annotations

import numpy as np


def gather_sequence(cache: np.ndarray, table_row: np.ndarray, context_len: int) -> np.ndarray:
    """Contiguous [context_len, H, D] float64 copy of one sequence's keys (or values).

    Token t is read from physical block ``table_row[t // B]`` at row ``t % B``
    ([note] 关键设计 2: the block table maps each logical block to its
    physical block; [lecture] PagedAttention 原理, single-request walk-through).
    """
    B = cache.shape[2]
    t = np.arange(int(context_len))
    phys = np.asarray(table_row, dtype=np.int64)[t // B]
    if context_len > 0:
        assert phys.min() >= 0 and phys.max() < cache.shape[0], "table points outside the pool"
    return cache[phys, :, t % B, :].astype(np.float64)          # [ctx, H, D]


def contiguous_attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """Textbook attention of one query per head over contiguous keys/values, float64.

    q [H, D]; keys, values [T, H, D]; returns [H, D].  ([note] 关键设计 1, first
    equation.)  The maximum logit is subtracted before exponentiating, which
    leaves every a_ij unchanged.
    """
    q = np.asarray(q, dtype=np.float64)
    H, D = q.shape
    if keys.shape[0] == 0:
        return np.zeros((H, D), dtype=np.float64)
    logits = scale * np.einsum("thd,hd->ht", keys, q)              # [H, T]
    logits -= logits.max(axis=1, keepdims=True)
    w = np.exp(logits)
    a = w / w.sum(axis=1, keepdims=True)                           # a_ij
    return np.einsum("ht,thd->hd", a, values)                      # o_i = sum_j a_ij v_j


def paged_decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                           block_tables: np.ndarray, context_lens: np.ndarray,
                           scale: float) -> np.ndarray:
    """o[s, h] for every sequence s and head h; float64 [S, H, D].

    q [S, H, D]; k_cache, v_cache [N, H, B, D]; block_tables [S, max_blocks]
    (entries past ceil(ctx/B) are never read); context_lens [S].
    """
    S, H, D = q.shape
    out = np.zeros((S, H, D), dtype=np.float64)
    for s in range(S):
        ctx = int(context_lens[s])
        keys = gather_sequence(k_cache, block_tables[s], ctx)
        values = gather_sequence(v_cache, block_tables[s], ctx)
        out[s] = contiguous_attention(q[s], keys, values, scale)
    return out


def paged_prefill_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                            block_tables: np.ndarray, context_lens: np.ndarray,
                            query_start: np.ndarray, scale: float) -> np.ndarray:
    """Attention of every new token of every sequence over its cached context, float64.

    The prompt phase over the task input only ([guide] 04, shared prefix: the
    request maps its first logical blocks onto the cached prefix blocks and the
    prompt phase runs only over its own tokens), with the attention of [note]
    关键设计 1 for each of those tokens: token i of the n_s new tokens of sequence
    s sits at position p = ctx_s - n_s + i and attends to positions t <= p
    (the sum to t = i of the first equation).

    q [T_total, H, D]: the new tokens of sequence s are rows
    query_start[s] .. query_start[s+1] - 1.  context_lens[s] counts the cached
    tokens and the new ones (whose keys and values are already in the pool).
    Returns [T_total, H, D].
    """
    T, H, D = q.shape
    out = np.zeros((T, H, D), dtype=np.float64)
    for s in range(len(context_lens)):
        ctx = int(context_lens[s])
        q0, q1 = int(query_start[s]), int(query_start[s + 1])
        n = q1 - q0
        if n == 0:
            continue
        keys = gather_sequence(k_cache, block_tables[s], ctx)
        values = gather_sequence(v_cache, block_tables[s], ctx)
        for i in range(n):
            p = ctx - n + i
            out[q0 + i] = contiguous_attention(q[q0 + i], keys[:p + 1], values[:p + 1], scale)
    return out
