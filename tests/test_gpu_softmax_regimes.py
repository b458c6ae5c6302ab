"""GPU parity in the softmax's hard regimes, against the fp64 oracle.

The other GPU tests draw q, K and V from the counter generator (spread 1, range +-3.5) at
scale 1/sqrt(D), where the logits span a few units.  Here:

* scale 1 and 4 on those inputs: logits spanning tens to hundreds of units, so the online
  softmax's running maximum moves often and the partitions' maxima differ widely at the merge;
* logits that rise (or fall) steadily along each context ([note] 关键设计 1: one softmax over all
  t <= i, whatever the logit range): every partition's maximum exceeds the last one's by tens of
  units, and in prefill the running maximum rises tile after tile, so the rule that moves it only
  when a tile raises it by more than 2^8 both fires and is skipped;
* fp16 inputs drawn much wider than +-3.5 (the output compared after dividing by the values'
  spread, since fp16 rounds it relative to its size), and inputs in the fp16 subnormal range.

Every case runs through the C ABI on batches spanning several partitions and a ragged tail.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import attention as oracle_attention
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl
from tests.helpers import ATOL

pytestmark = pytest.mark.gpu

# Two batches with contexts around partition and block edges.  Both leave the grid small, so the
# decode kernel splits each context into short partitions: 4 x 4 heads up to 3001 tokens gives 12
# partitions of 256 tokens (merged by the second kernel through the workspace); 4 x 8 heads up to
# 2048 tokens gives 8 (merged inside one thread-block cluster per sequence and head).
LAYOUTS = {"merge_kernel": ([3001, 1, 257, 2048], 4, 2), "cluster_merge": ([2048, 1, 257, 1999], 8, 1)}


def _batch(name, seed, D, B):
    lens, H, kernels = LAYOUTS[name]
    w = wl.custom(seed, lens, num_heads=H, head_dim=D, block_size=B)
    part, got = pkv.paged_attention_plan(w.num_seqs, H, D, w.max_blocks_per_seq, B)
    assert got == kernels and -(-max(lens) // part) >= 8       # several partitions per sequence
    return w


def _decode(w, q, k, v, scale, dev, fused=False):
    tables = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if fused:
        # the fused step re-stores each sequence's last row (its own slot) before attending
        B = w.block_size
        last = w.context_lens - 1
        slots = np.array([w.block_tables[s, last[s] // B] * B + last[s] % B for s in range(w.num_seqs)], np.int64)
        key = torch.stack([k[int(slots[s]) // B, :, int(slots[s]) % B, :] for s in range(w.num_seqs)])
        val = torch.stack([v[int(slots[s]) // B, :, int(slots[s]) % B, :] for s in range(w.num_seqs)])
        out = pkv.paged_attention_decode_append(qd, key.to(dev), val.to(dev), torch.from_numpy(slots).to(dev), kd,
                                                vd, tables, lens, scale, w.block_size)
    else:
        out = pkv.paged_attention_decode(qd, kd, vd, tables, lens, scale, w.block_size)
    code = pkv.device_error()
    assert code == 0, pkv.DEV_CODES.get(code, code)
    return out.cpu().numpy().astype(np.float64)


def _oracle(w, q, k, v, scale):
    return oracle_attention.paged_decode_attention(q.numpy().astype(np.float64), k.numpy(), v.numpy(),
                                                   w.block_tables, w.context_lens, scale)


def _err(got, ref, spread=1.0):
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.max(np.abs(got - ref))) / spread


@pytest.mark.parametrize("layout", sorted(LAYOUTS))
@pytest.mark.parametrize("D,B", [(128, 16), (64, 8), (128, 32)])
@pytest.mark.parametrize("scale", [1.0, 4.0])
def test_decode_large_scale(cuda_device, layout, D, B, scale):
    w = _batch(layout, 900 + D + B, D, B)
    q, k, v = wl.gaussian_inputs(w, 17 + B)
    assert _err(_decode(w, q, k, v, scale, cuda_device), _oracle(w, q, k, v, scale)) <= ATOL


@pytest.mark.parametrize("layout", sorted(LAYOUTS))
@pytest.mark.parametrize("first,last", [(-40.0, 40.0), (40.0, -40.0), (0.0, 300.0)],
                         ids=["rising", "falling", "steep_rise"])
@pytest.mark.parametrize("fused", [False, True], ids=["decode", "fused_append"])
def test_decode_logit_ramp_across_partitions(cuda_device, layout, first, last, fused):
    # q.k_t moves steadily along the context, so consecutive partitions' maxima differ by tens of
    # units (hundreds for the steep rise); the merge must rescale every partition by its own max
    w = _batch(layout, 77, 128, 16)
    q, k, v = wl.ramp_inputs(w, 5, first, last)
    got = _decode(w, q, k, v, 1.0, cuda_device, fused=fused)
    assert _err(got, _oracle(w, q, k, v, 1.0)) <= ATOL


@pytest.mark.parametrize("layout", sorted(LAYOUTS))
def test_decode_wide_values(cuda_device, layout):
    # q and k drawn with spread 4 (logits of hundreds of units at scale 1/sqrt(D)) and v with
    # spread 30; the error is compared after dividing by v's spread
    w = _batch(layout, 31, 128, 16)
    q, k, v = wl.gaussian_inputs(w, 8, q_std=4.0, k_std=4.0, v_std=30.0)
    assert float(v[~torch.isnan(v)].abs().max()) > 100.0
    assert _err(_decode(w, q, k, v, w.scale, cuda_device), _oracle(w, q, k, v, w.scale), spread=30.0) <= ATOL


@pytest.mark.parametrize("layout", sorted(LAYOUTS))
def test_decode_subnormal_values(cuda_device, layout):
    # keys and values in the fp16 subnormal range (below 2^-14): fp32 accumulation keeps them,
    # and the output rounds to fp16 subnormals, whose spacing is 2^-24; the bound is half that
    # spacing plus 2e-3 of the value spread
    w = _batch(layout, 32, 64, 16)
    q, k, v = wl.gaussian_inputs(w, 9, q_std=1.0, k_std=2.0 ** -16, v_std=2.0 ** -18)
    vv = v[~torch.isnan(v)]
    assert float(vv.abs().max()) < 2.0 ** -14 and float((vv != 0).float().mean()) > 0.9
    got, ref = _decode(w, q, k, v, w.scale, cuda_device), _oracle(w, q, k, v, w.scale)
    assert np.isfinite(got).all() and np.abs(got).max() > 0
    assert float(np.max(np.abs(got - ref))) <= 2.0 ** -25 + ATOL * 2.0 ** -18


def _prefill(w, news, q, k, v, scale, dev):
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    out = pkv.paged_attention_prefill(q.to(dev), k.to(dev), v.to(dev), torch.from_numpy(w.block_tables).to(dev),
                                      torch.from_numpy(w.context_lens).to(dev), torch.from_numpy(qs).to(dev), scale,
                                      w.block_size, max(news))
    code = pkv.device_error()
    assert code == 0, pkv.DEV_CODES.get(code, code)
    ref = oracle_attention.paged_prefill_attention(q.numpy().astype(np.float64), k.numpy(), v.numpy(),
                                                   w.block_tables, w.context_lens, qs, scale)
    return out.cpu().numpy().astype(np.float64), ref


PREFILL_LENS = [700, 300, 1030]
PREFILL_NEWS = [700, 41, 300]            # a whole prompt; a short tail; 300 new tokens over 730 cached


@pytest.mark.parametrize("scale", [1.0, 4.0])
def test_prefill_large_scale(cuda_device, scale):
    w = wl.custom(51, PREFILL_LENS, num_heads=3, head_dim=128, block_size=16)
    _, k, v = wl.gaussian_inputs(w, 19)
    q = torch.from_numpy(np.random.default_rng(21).standard_normal((sum(PREFILL_NEWS), 3, 128)).astype(np.float16))
    got, ref = _prefill(w, PREFILL_NEWS, q, k, v, scale, cuda_device)
    assert _err(got, ref) <= ATOL


@pytest.mark.parametrize("first,last", [(0.0, 200.0), (0.0, 5.0), (200.0, 0.0)],
                         ids=["rescales_often", "within_2^8", "max_in_first_tile"])
def test_prefill_logit_ramp(cuda_device, first, last):
    # every new token sees the same ramp of q.k over the keys: rising by 200 units over ~1000
    # positions, the running maximum climbs by ~13 units (in log2, ~18) per 64-key tile, so the
    # kept maximum moves on most tiles; rising by 5 units it never has to; falling, the first tile
    # holds the maximum throughout
    w = wl.custom(53, PREFILL_LENS, num_heads=3, head_dim=128, block_size=16)
    q, k, v = wl.ramp_inputs(w, 23, first, last, rows_per_seq=PREFILL_NEWS)
    got, ref = _prefill(w, PREFILL_NEWS, q, k, v, 1.0, cuda_device)
    assert _err(got, ref) <= ATOL


def test_prefill_wide_values(cuda_device):
    w = wl.custom(54, PREFILL_LENS, num_heads=3, head_dim=128, block_size=16)
    _, k, v = wl.gaussian_inputs(w, 24, k_std=3.0, v_std=20.0)
    q = torch.from_numpy((np.random.default_rng(25).standard_normal((sum(PREFILL_NEWS), 3, 128)) * 3.0)
                         .astype(np.float16))
    got, ref = _prefill(w, PREFILL_NEWS, q, k, v, w.scale, cuda_device)
    assert _err(got, ref, spread=20.0) <= ATOL


def test_shared_prefix_decode_logit_ramp(cuda_device):
    # 16 requests on one 512-token prefix: the prefix part (tensor cores, softmax weights in fp16)
    # and each request's own part are merged; the ramp puts the maximum at the end of the context,
    # tens of units above anything in the prefix
    w = dataclasses.replace(wl.shared_prefix(seed=61, requests=16, prefix_len=512, suffix_lo=40, suffix_hi=700),
                            num_heads=4)
    q, k, v = wl.ramp_inputs(w, 26, -30.0, 30.0)
    dev = cuda_device
    gs = torch.tensor([0, 16], dtype=torch.int32, device=dev)
    pl = torch.tensor([512], dtype=torch.int32, device=dev)
    out = pkv.paged_attention_decode_shared_prefix(q.to(dev), k.to(dev), v.to(dev),
                                                   torch.from_numpy(w.block_tables).to(dev),
                                                   torch.from_numpy(w.context_lens).to(dev), gs, pl, 1.0,
                                                   w.block_size, 16)
    code = pkv.device_error()
    assert code == 0, pkv.DEV_CODES.get(code, code)
    assert _err(out.cpu().numpy().astype(np.float64), _oracle(w, q, k, v, 1.0)) <= ATOL
