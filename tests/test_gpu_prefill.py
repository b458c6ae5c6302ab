"""Paged prefill attention on the GPU (tensor cores) against the fp64 oracle.

New tokens attend over the cached context plus, causally, themselves; K/V are
read through the block table.  Max abs error <= 2e-3, as for decode (the
softmax weights are rounded to fp16 before they multiply V)."""
import numpy as np
import pytest
import torch

from oracle import attention as oracle_attention
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl
from tests.helpers import ATOL

pytestmark = pytest.mark.gpu


def _run(w, news, dev, seed=77):
    news = list(news)
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    T = int(qs[-1])
    k, v = w.pools(dev)
    q = wl.dense_tensor((T, w.num_heads, w.head_dim), seed, wl.STREAM_Q, dev)
    out = pkv.paged_attention_prefill(q, k, v, torch.from_numpy(w.block_tables).to(dev),
                                      torch.from_numpy(w.context_lens).to(dev), torch.from_numpy(qs).to(dev),
                                      w.scale, w.block_size, max(news) if news else 0)
    code = pkv.device_error()
    return out, q, qs, code


def _oracle(w, q, qs, seqs):
    kc, vc, tabs, lens = w.compact_pools(seqs)
    rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in seqs]).astype(np.int64)
    sub_qs = np.concatenate([[0], np.cumsum([qs[s + 1] - qs[s] for s in seqs])])
    ref = oracle_attention.paged_prefill_attention(q.cpu().numpy()[rows].astype(np.float64), kc.numpy(), vc.numpy(),
                                                   tabs, lens, sub_qs, w.scale)
    return rows, ref


def _check(w, news, dev, seqs=None):
    out, q, qs, code = _run(w, news, dev)
    assert code == 0, pkv.DEV_CODES.get(code, code)
    seqs = list(range(w.num_seqs)) if seqs is None else seqs
    seqs = [s for s in seqs if news[s] > 0]
    rows, ref = _oracle(w, q, qs, seqs)
    got = out.cpu().numpy()[rows].astype(np.float64)
    assert np.isfinite(got).all()
    err = float(np.max(np.abs(got - ref)))
    assert err <= ATOL, err
    return err


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [4, 8, 16, 32])
def test_ragged_prefill_every_shape(cuda_device, D, B):
    # cached prefixes of every alignment, new-token counts around the 64-token tiles
    lens = [1, 17, 64, 65, 130, 300, 257, 200]
    news = [1, 17, 30, 65, 64, 129, 1, 200]
    w = wl.custom(300 + D + B, lens, num_heads=3, head_dim=D, block_size=B, name=f"prefill_D{D}_B{B}")
    _check(w, news, cuda_device)


def test_whole_prompts_nothing_cached(cuda_device):
    lens = [513, 64, 1000]
    w = wl.custom(41, lens, num_heads=4, head_dim=128, block_size=16)
    _check(w, lens, cuda_device)


def test_zero_new_tokens_skipped(cuda_device):
    lens = [40, 90, 7]
    news = [0, 33, 0]
    w = wl.custom(42, lens, num_heads=2, head_dim=128, block_size=16)
    out, q, qs, code = _run(w, news, cuda_device)
    assert code == 0
    rows, ref = _oracle(w, q, qs, [1])
    assert np.max(np.abs(out.cpu().numpy()[rows].astype(np.float64) - ref)) <= ATOL


def test_one_new_token_matches_decode_kernel(cuda_device):
    w = wl.opt13b(seed=12, num_seqs=16, lo=100, hi=1500)
    out, q, qs, code = _run(w, [1] * 16, cuda_device)
    assert code == 0
    k, v = w.pools(cuda_device)
    dec = pkv.paged_attention_decode(q, k, v, torch.from_numpy(w.block_tables).to(cuda_device),
                                     torch.from_numpy(w.context_lens).to(cuda_device), w.scale, 16)
    assert (out.double() - dec.double()).abs().max().item() <= 2 * ATOL


def test_shared_prefix_prefill(cuda_device):
    # requests whose first 64 blocks are one cached 1024-token prefix; each prefills its suffix
    w = wl.shared_prefix(seed=1004, requests=12, suffix_lo=32, suffix_hi=300)
    news = [int(c) - 1024 for c in w.context_lens]
    _check(w, news, cuda_device)


def test_shared_prefix_prefill_full_size(cuda_device):
    # 256 requests sharing the 1024-token prefix, suffixes U[32, 512]: whole batch on the GPU,
    # the oracle on three sequences (longest, shortest, one more)
    w = wl.shared_prefix()
    news = [int(c) - 1024 for c in w.context_lens]
    lens = w.context_lens
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 7})
    _check(w, news, cuda_device, seqs)


def test_bad_query_range_recorded(cuda_device):
    w = wl.custom(43, [10, 20], num_heads=2, head_dim=64, block_size=16)
    out, q, qs, code = _run(w, [5, 25], cuda_device)     # 25 new tokens > context 20
    assert code == 6
    rows, ref = _oracle(w, q, qs, [0])
    assert np.max(np.abs(out.cpu().numpy()[rows].astype(np.float64) - ref)) <= ATOL


@pytest.mark.parametrize("B", [4, 16])
def test_bad_block_id_recorded(cuda_device, B):
    # an out-of-range and a negative entry inside sequence 0's context: the code is recorded, the
    # bad sequence's rows are not written, and the other sequence is unaffected (B = 16 takes the
    # tensor-map path for whole blocks, B = 4 the copy path)
    w = wl.custom(44 + B, [200, 150], num_heads=2, head_dim=128, block_size=B)
    news = [40, 60]
    tables = w.block_tables.copy()
    tables[0, 1] = w.num_blocks + 5
    tables[0, 3] = -2
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    k, v = w.pools(cuda_device)
    q = wl.dense_tensor((int(qs[-1]), w.num_heads, w.head_dim), 78, wl.STREAM_Q, cuda_device)
    out = torch.full_like(q, 7.0)
    pkv.paged_attention_prefill(q, k, v, torch.from_numpy(tables).to(cuda_device),
                                torch.from_numpy(w.context_lens).to(cuda_device), torch.from_numpy(qs).to(cuda_device),
                                w.scale, w.block_size, max(news), out=out)
    assert pkv.device_error() == 1
    got = out.cpu().numpy().astype(np.float64)
    assert (got[: news[0]] == 7.0).all()
    rows, ref = _oracle(w, q, qs, [1])
    assert np.max(np.abs(got[rows] - ref)) <= ATOL


def test_long_prompts_full_size_sampled(cuda_device):
    # the bench's long-prompt launch: 8 prompts x 4096 tokens, nothing cached, 40 heads x 128,
    # block 16, whole batch on the GPU in one launch; the oracle recomputes sampled rows (tile and
    # block edges, the first and the last token) of three sequences and three heads row by row
    w = wl.custom(1009, [4096] * 8, 40, 128, 16, name="prefill_8x4096")
    news = [4096] * 8
    out, q, qs, code = _run(w, news, cuda_device)
    assert code == 0, pkv.DEV_CODES.get(code, code)
    got = out.cpu().numpy().astype(np.float64)
    qh = q.cpu().numpy().astype(np.float64)
    rows = [0, 1, 63, 64, 127, 128, 255, 256, 1000, 2047, 2048, 4031, 4095]
    for s in (0, 5, 7):
        kc, vc, tabs, lens = w.compact_pools([s])
        keys = oracle_attention.gather_sequence(kc.numpy(), tabs[0], int(lens[0]))
        values = oracle_attention.gather_sequence(vc.numpy(), tabs[0], int(lens[0]))
        for h in (0, 17, 39):
            for i in rows:
                ref = oracle_attention.contiguous_attention(qh[qs[s] + i, h][None], keys[: i + 1, h][:, None],
                                                           values[: i + 1, h][:, None], w.scale)
                err = float(np.max(np.abs(got[qs[s] + i, h] - ref.reshape(-1))))
                assert err <= ATOL, (s, h, i, err)
