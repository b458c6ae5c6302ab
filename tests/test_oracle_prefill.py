"""Pins for the prefill oracle: causal attention of a library routine on contiguous
K/V, the decode oracle when each sequence brings one new token, and the
invariance under physical-id relabelling."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oa


def _layout(rng, lens, H, D, B):
    """Pools and tables for contiguous per-sequence K/V (pools filled by a reshape route)."""
    nbs = [-(-c // B) for c in lens]
    N = sum(nbs) + 3
    perm = rng.permutation(N)
    tables = np.full((len(lens), max(nbs)), -1, dtype=np.int64)
    kp = np.full((N, H, B, D), np.nan)
    vp = np.full((N, H, B, D), np.nan)
    seqs = []
    pos = 0
    for s, c in enumerate(lens):
        tables[s, :nbs[s]] = perm[pos:pos + nbs[s]]
        pos += nbs[s]
        keys = rng.standard_normal((c, H, D))
        values = rng.standard_normal((c, H, D))
        for src, dst in ((keys, kp), (values, vp)):
            padded = np.full((nbs[s] * B, H, D), np.nan)
            padded[:c] = src
            blocks = padded.reshape(nbs[s], B, H, D).transpose(0, 2, 1, 3)
            for j in range(nbs[s]):
                dst[tables[s, j]] = blocks[j]
        seqs.append((keys, values))
    return kp, vp, tables, seqs


def _err_vs_library(lens, news, H, D, B):
    """Max |oracle - torch SDPA with an explicit causal mask| over a paged batch."""
    rng = np.random.default_rng(sum(lens))
    kp, vp, tables, seqs = _layout(rng, lens, H, D, B)
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int64)
    q = rng.standard_normal((int(qs[-1]), H, D))
    scale = 1 / math.sqrt(D)
    got = oa.paged_prefill_attention(q, kp, vp, tables, np.array(lens), qs, scale)
    err = 0.0
    for s, (c, n) in enumerate(zip(lens, news)):
        keys, values = seqs[s]
        qt = torch.from_numpy(q[qs[s]:qs[s + 1]].transpose(1, 0, 2).copy())[None]     # [1, H, n, D]
        kt = torch.from_numpy(keys.transpose(1, 0, 2).copy())[None]
        vt = torch.from_numpy(values.transpose(1, 0, 2).copy())[None]
        pos = torch.arange(c - n, c)[:, None]
        mask = torch.arange(c)[None, :] <= pos                                      # [n, c]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
        err = max(err, float(np.max(np.abs(got[qs[s]:qs[s + 1]] - ref[0].numpy().transpose(1, 0, 2)))))
    return err


CASES = [
    ([20, 9, 40], [5, 9, 1], 2, 64, 4),
    ([100, 33], [64, 17], 3, 128, 16),
    ([70], [70], 1, 32, 8),                     # whole prompt, nothing cached
]


@pytest.mark.parametrize("lens,news,H,D,B", CASES)
def test_matches_library_causal_attention(lens, news, H, D, B):
    assert _err_vs_library(lens, news, H, D, B) < 1e-12


def test_one_new_token_is_decode():
    rng = np.random.default_rng(4)
    lens = [13, 1, 40]
    kp, vp, tables, _ = _layout(rng, lens, 2, 16, 4)
    q = rng.standard_normal((3, 2, 16))
    a = oa.paged_prefill_attention(q, kp, vp, tables, np.array(lens), np.arange(4), 0.3)
    b = oa.paged_decode_attention(q, kp, vp, tables, np.array(lens), 0.3)
    np.testing.assert_array_equal(a, b)


def test_first_new_token_of_an_uncached_prompt_sees_only_itself():
    rng = np.random.default_rng(5)
    kp, vp, tables, seqs = _layout(rng, [9], 1, 8, 4)
    q = rng.standard_normal((9, 1, 8))
    got = oa.paged_prefill_attention(q, kp, vp, tables, np.array([9]), np.array([0, 9]), 1.0)
    np.testing.assert_array_equal(got[0], seqs[0][1][0])


_ATTEND = oa.contiguous_attention


@pytest.mark.parametrize("mutant", ["one_key_short", "one_key_long"])
def test_planted_causal_limit_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "one_key_short":            # drops the token's own key
        fake = lambda qq, k, v, sc: _ATTEND(qq, k[:-1], v[:-1], sc) if len(k) > 1 else _ATTEND(qq, k, v, sc)
        monkeypatch.setattr(oa, "contiguous_attention", fake)
    else:                                    # lets each token see one future key
        orig_gather = oa.gather_sequence
        monkeypatch.setattr(oa, "gather_sequence", lambda c, t, n: orig_gather(c, t, n))
        fake = lambda qq, k, v, sc: _ATTEND(qq, k, v, sc)
        orig_prefill = oa.paged_prefill_attention

        def shifted(q, kc, vc, bt, lens, qs, sc):
            out = np.zeros(q.shape)
            for s in range(len(lens)):
                ctx = int(lens[s]); q0, q1 = int(qs[s]), int(qs[s + 1]); n = q1 - q0
                keys = orig_gather(kc, bt[s], ctx); values = orig_gather(vc, bt[s], ctx)
                for i in range(n):
                    p = min(ctx - n + i + 1, ctx - 1)
                    out[q0 + i] = _ATTEND(q[q0 + i], keys[:p + 1], values[:p + 1], sc)
            return out
        monkeypatch.setattr(oa, "paged_prefill_attention", shifted)
    assert _err_vs_library(*CASES[1]) > 1e-3
