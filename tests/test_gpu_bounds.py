"""Caller-stated bounds and devices, checked on the GPU.

* pkv_paged_attention_prefill sizes its grid from max_query_len, and the shared-prefix decode
  entry from max_group_size.  A sequence with more new tokens, or a group with more members,
  than those bounds cover is not fully processed; the kernels record a device check code for it
  (PKV_DEV_BAD_QUERY_RANGE, PKV_DEV_PREFIX_MISMATCH) instead of leaving rows silently unwritten.
* The binding refuses a CUDA tensor that is not on the current device, on the host, before any
  kernel runs (the library launches on the current device; another device's memory would be
  read as a peer's).
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _prefill(w, news, max_query_len, dev):
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    q = wl.dense_tensor((int(qs[-1]), w.num_heads, w.head_dim), 5, wl.STREAM_Q, dev)
    k, v = w.pools(dev)
    pkv.paged_attention_prefill(q, k, v, torch.from_numpy(w.block_tables).to(dev),
                                torch.from_numpy(w.context_lens).to(dev), torch.from_numpy(qs).to(dev), w.scale,
                                w.block_size, max_query_len)
    return pkv.device_error()


def test_prefill_understated_max_query_len_is_recorded(cuda_device):
    w = wl.custom(81, [300, 40], num_heads=2, head_dim=128, block_size=16)
    assert _prefill(w, [300, 40], 300, cuda_device) == 0
    # one CTA covers 256 new tokens: stating 200 leaves rows 256..299 of the first sequence unwritten
    assert _prefill(w, [300, 40], 200, cuda_device) == 6            # PKV_DEV_BAD_QUERY_RANGE
    assert _prefill(w, [300, 40], 300, cuda_device) == 0            # the code was read and cleared


def _shared(w, members, max_group_size, dev):
    k, v = w.pools(dev)
    q = w.q(dev)
    gs = torch.tensor([0, members], dtype=torch.int32, device=dev)
    pl = torch.tensor([64], dtype=torch.int32, device=dev)
    pkv.paged_attention_decode_shared_prefix(q, k, v, torch.from_numpy(w.block_tables).to(dev),
                                             torch.from_numpy(w.context_lens).to(dev), gs, pl, w.scale,
                                             w.block_size, max_group_size)
    return pkv.device_error()


def test_shared_prefix_understated_max_group_size_is_recorded(cuda_device):
    # 300 requests on one 64-token prefix: the prefix part covers 256 members per CTA
    w = wl.shared_prefix(seed=82, requests=300, prefix_len=64, suffix_lo=1, suffix_hi=40, block_size=16)
    assert _shared(w, 300, 300, cuda_device) == 0
    assert _shared(w, 300, 100, cuda_device) == 7                   # PKV_DEV_PREFIX_MISMATCH
    assert _shared(w, 300, 300, cuda_device) == 0


def test_binding_refuses_a_tensor_on_another_device(cuda_device, monkeypatch):
    w = wl.custom(83, [40, 9], num_heads=2, head_dim=64, block_size=16)
    k, v = w.pools(cuda_device)
    q = w.q(cuda_device)
    tables = torch.from_numpy(w.block_tables).to(cuda_device)
    lens = torch.from_numpy(w.context_lens).to(cuda_device)
    out = torch.full_like(q, float("nan"))
    torch.cuda.synchronize()
    # the tensors live on cuda:0; make the binding see another current device
    monkeypatch.setattr(torch.cuda, "current_device", lambda: cuda_device.index + 1)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_decode(q, k, v, tables, lens, w.scale, w.block_size, out=out)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG and "current CUDA device" in str(e.value)
    monkeypatch.undo()
    torch.cuda.synchronize()
    assert torch.isnan(out).all()                                   # nothing ran
    pkv.paged_attention_decode(q, k, v, tables, lens, w.scale, w.block_size, out=out)
    assert pkv.device_error() == 0 and torch.isfinite(out).all()
