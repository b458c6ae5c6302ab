"""Pins for the attention oracle, against facts fixed outside it.

Each test checks the oracle against something it does not compute itself:
a library attention routine (torch's scaled_dot_product_attention in float64
on contiguous K/V, which the page says the paged form reaches exactly), closed
forms, and invariants the definition implies.  The last tests plant mistakes
in the oracle, on the CPU, and check that a pin catches each one.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oa
from paged_kv_cache_73_gb300 import workloads as wl


def _pool_from_contiguous(keys, values, table, num_blocks, block_size, fill=np.nan):
    """Lay contiguous [T, H, D] keys/values into a pool through ``table`` by reshaping.

    The sequence is padded to whole blocks, viewed as [blocks, B, H, D],
    transposed to [blocks, H, B, D] and each block stored at its physical id.
    This route shares no indexing with the oracle's gather.
    """
    T, H, D = keys.shape
    nb = -(-T // block_size)
    kp = np.full((num_blocks, H, block_size, D), fill)
    vp = np.full((num_blocks, H, block_size, D), fill)
    for src, dst in ((keys, kp), (values, vp)):
        padded = np.full((nb * block_size, H, D), fill)
        padded[:T] = src
        blocks = padded.reshape(nb, block_size, H, D).transpose(0, 2, 1, 3)
        for j in range(nb):
            dst[table[j]] = blocks[j]
    return kp, vp


def _sdpa(q, keys, values, scale):
    """torch SDPA, float64, one query per head: q [H, D], keys/values [T, H, D] -> [H, D]."""
    qt = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float64))[None, :, None, :]
    kt = torch.from_numpy(np.ascontiguousarray(keys.transpose(1, 0, 2), dtype=np.float64))[None]
    vt = torch.from_numpy(np.ascontiguousarray(values.transpose(1, 0, 2), dtype=np.float64))[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, :, 0, :].numpy()


def _check_against_sdpa(attn_fn, seed, ctx_list, H, D, B, scale=None):
    """Max abs difference between ``attn_fn`` (oracle signature) and SDPA over a paged batch."""
    rng = np.random.default_rng(seed)
    S = len(ctx_list)
    nbs = [-(-c // B) for c in ctx_list]
    N = sum(nbs) + 5
    perm = rng.permutation(N)
    tables = np.full((S, max(nbs)), -1, dtype=np.int64)
    pos = 0
    kp = np.full((N, H, B, D), np.nan)
    vp = np.full((N, H, B, D), np.nan)
    q = rng.standard_normal((S, H, D))
    ref = np.zeros((S, H, D))
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    for s, c in enumerate(ctx_list):
        tables[s, :nbs[s]] = perm[pos:pos + nbs[s]]
        pos += nbs[s]
        keys = rng.standard_normal((c, H, D))
        values = rng.standard_normal((c, H, D))
        k1, v1 = _pool_from_contiguous(keys, values, tables[s], N, B)
        used = tables[s, :nbs[s]]
        kp[used] = k1[used]
        vp[used] = v1[used]
        ref[s] = _sdpa(q[s], keys, values, scale)
    got = attn_fn(q, kp, vp, tables, np.array(ctx_list), scale)
    return float(np.max(np.abs(got - ref)))


@pytest.mark.parametrize("ctx_list,H,D,B", [
    ([7, 5, 12], 2, 64, 4),          # the tiny batch's lengths
    ([1, 16, 17, 33, 100], 3, 128, 16),
    ([31, 64, 9], 2, 64, 32),
    ([8, 3], 1, 16, 8),
])
def test_matches_library_attention(ctx_list, H, D, B):
    assert _check_against_sdpa(oa.paged_decode_attention, 7, ctx_list, H, D, B) < 1e-12


def test_two_token_closed_form():
    # o = v0 + sigmoid(scale * q.(k1 - k0)) * (v1 - v0) for a context of two tokens
    rng = np.random.default_rng(3)
    D, B = 8, 4
    q = rng.standard_normal((1, 1, D))
    keys = rng.standard_normal((2, 1, D))
    values = rng.standard_normal((2, 1, D))
    kp, vp = _pool_from_contiguous(keys, values, [2], 4, B)
    scale = 0.37
    got = oa.paged_decode_attention(q, kp, vp, np.array([[2]]), np.array([2]), scale)[0, 0]
    z = scale * float(q[0, 0] @ (keys[1, 0] - keys[0, 0]))
    sig = 1.0 / (1.0 + math.exp(-z))
    want = values[0, 0] + sig * (values[1, 0] - values[0, 0])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_single_token_returns_its_value():
    t = wl.custom(11, [1, 1, 1], 2, 64, 16)
    k, v = t.pools()
    q = t.q().numpy()
    out = oa.paged_decode_attention(q, k.numpy(), v.numpy(), t.block_tables, t.context_lens, t.scale)
    for s in range(3):
        np.testing.assert_array_equal(out[s], v.numpy()[t.block_tables[s, 0], :, 0, :].astype(np.float64))


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(5)
    T, H, D, B = 37, 2, 16, 8
    keys = rng.standard_normal((T, H, D))
    values = rng.standard_normal((T, H, D))
    table = rng.permutation(10)[:5]
    kp, vp = _pool_from_contiguous(keys, values, table, 10, B)
    got = oa.paged_decode_attention(np.zeros((1, H, D)), kp, vp, table[None], np.array([T]), 0.25)[0]
    np.testing.assert_allclose(got, values.mean(axis=0), rtol=0, atol=1e-13)


def test_large_scale_selects_argmax_value():
    rng = np.random.default_rng(9)
    T, H, D, B = 20, 3, 8, 4
    keys = rng.standard_normal((T, H, D))
    values = rng.standard_normal((T, H, D))
    q = rng.standard_normal((1, H, D))
    table = np.arange(5)[::-1].copy()
    kp, vp = _pool_from_contiguous(keys, values, table, 5, B)
    got = oa.paged_decode_attention(q, kp, vp, table[None], np.array([T]), 1e6)[0]
    for h in range(H):
        j = int(np.argmax(keys[:, h] @ q[0, h]))
        np.testing.assert_allclose(got[h], values[j, h], atol=1e-9)


def test_context_zero_is_zero():
    out = oa.paged_decode_attention(np.ones((1, 2, 8)), np.full((2, 2, 4, 8), np.nan),
                                    np.full((2, 2, 4, 8), np.nan), np.array([[-1]]), np.array([0]), 1.0)
    assert np.all(out == 0)


def test_invariant_under_relabelling_physical_blocks():
    t = wl.tiny()
    k, v = t.pools()
    k, v, q = k.numpy(), v.numpy(), t.q().numpy()
    base = oa.paged_decode_attention(q, k, v, t.block_tables, t.context_lens, t.scale)
    rng = np.random.default_rng(123)
    for _ in range(3):
        perm = rng.permutation(t.num_blocks)          # new id of old block i is perm[i]
        k2 = np.empty_like(k)
        v2 = np.empty_like(v)
        k2[perm] = k
        v2[perm] = v
        tab2 = np.where(t.block_tables >= 0, perm[np.maximum(t.block_tables, 0)], -1)
        got = oa.paged_decode_attention(q, k2, v2, tab2, t.context_lens, t.scale)
        np.testing.assert_array_equal(got, base)


def test_nan_outside_the_context_never_reaches_the_result():
    # the tiny batch's pools are NaN in every unused block and past every last token
    t = wl.tiny()
    k, v = t.pools()
    assert torch.isnan(k).any()
    out = oa.paged_decode_attention(t.q().numpy(), k.numpy(), v.numpy(), t.block_tables, t.context_lens, t.scale)
    assert np.isfinite(out).all()


def test_compact_pool_sample_equals_full_pool():
    t = wl.opt13b(num_seqs=6, lo=20, hi=90, block_size=16)
    k, v = t.pools()
    q = t.q().numpy()
    full = oa.paged_decode_attention(q, k.numpy(), v.numpy(), t.block_tables, t.context_lens, t.scale)
    seqs = [4, 1]
    kc, vc, tabs, lens = t.compact_pools(seqs)
    part = oa.paged_decode_attention(q[seqs], kc.numpy(), vc.numpy(), tabs, lens, t.scale)
    np.testing.assert_array_equal(part, full[seqs])


# ---- planted mistakes: each must be caught by a pin above -------------------------------

_GATHER = oa.gather_sequence
_ATTEND = oa.contiguous_attention


def _mutant_swapped_index(cache, table_row, ctx):
    B = cache.shape[2]
    t = np.arange(int(ctx))
    phys = np.asarray(table_row)[np.minimum(t % B, len(table_row) - 1)]
    return cache[phys, :, np.minimum(t // B, B - 1), :].astype(np.float64)


def _mutant_drops_newest(cache, table_row, ctx):
    return _GATHER(cache, table_row, max(int(ctx) - 1, 0))


def _mutant_per_block_softmax(q, keys, values, scale, B=4):
    out = np.zeros(q.shape)
    for start in range(0, keys.shape[0], B):
        out += _ATTEND(q, keys[start:start + B], values[start:start + B], scale)
    return out


def _mutant_transposed_value(q, keys, values, scale):
    logits = scale * np.einsum("thd,hd->ht", keys, q)
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    a = w / w.sum(axis=1, keepdims=True)
    return np.einsum("ht,thd->hd", a, keys)          # uses keys where values belong


@pytest.mark.parametrize("name", ["swapped_index", "drops_newest", "per_block_softmax", "transposed_value"])
def test_planted_mistakes_are_caught(monkeypatch, name):
    if name == "swapped_index":
        monkeypatch.setattr(oa, "gather_sequence", _mutant_swapped_index)
    elif name == "drops_newest":
        monkeypatch.setattr(oa, "gather_sequence", _mutant_drops_newest)
    elif name == "per_block_softmax":
        monkeypatch.setattr(oa, "contiguous_attention", _mutant_per_block_softmax)
    else:
        monkeypatch.setattr(oa, "contiguous_attention", _mutant_transposed_value)
    with np.errstate(all="ignore"):
        err = _check_against_sdpa(oa.paged_decode_attention, 7, [7, 5, 12], 2, 64, 4)
    assert not (err < 1e-6), f"planted mistake {name} not caught (err={err})"
