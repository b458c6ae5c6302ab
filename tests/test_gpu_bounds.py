"""Caller-stated bounds and devices, checked on the GPU.

* pkv_paged_attention_prefill sizes its grid from max_query_len, and the shared-prefix decode
  entry from max_group_size.  A sequence with more new tokens, or a group with more members,
  than those bounds cover is not fully processed; the kernels record a device check code for it
  (PKV_DEV_BAD_QUERY_RANGE, PKV_DEV_PREFIX_MISMATCH) instead of leaving rows silently unwritten.
* The binding refuses a CUDA tensor that is not on the current device, on the host, before any
  kernel runs (the library launches on the current device; another device's memory would be
  read as a peer's).
* Failure detection without a fault: the one wait of one CTA on others (partition 0 of a cluster
  waiting for the other partitions' partial results) is bounded; a test entry makes it run out on
  a phase nothing completes, and the host reads the recorded code with the context still usable.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oracle_attention
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


def test_cluster_merge_wait_runs_out_and_is_reported(cuda_device):
    # failure detection without a fault: partition 0's bounded wait for the other partitions of its
    # cluster runs out on a phase nothing completes (they skip their stores and arrivals in this
    # test entry); the host reads PKV_DEV_WAIT_TIMEOUT and the context stays usable
    w = wl.custom(84, [2000, 700, 1500, 64], num_heads=8, head_dim=128, block_size=16)
    q, k, v = w.q(cuda_device), *w.pools(cuda_device)
    tables = torch.from_numpy(w.block_tables).to(cuda_device)
    lens = torch.from_numpy(w.context_lens).to(cuda_device)
    assert pkv.paged_attention_plan(4, 8, 128, w.max_blocks_per_seq, 16) == (256, 1)   # 8 partitions, on chip
    out = torch.empty_like(q)
    lib = pkv.load()
    assert lib.pkv_test_cluster_merge_timeout(q.data_ptr(), k.data_ptr(), v.data_ptr(), tables.data_ptr(),
                                              lens.data_ptr(), 4, 8, 128, k.shape[0], w.max_blocks_per_seq,
                                              w.scale, 16, out.data_ptr(), 100, None) == pkv.PKV_OK
    assert pkv.device_error() == 5                                   # PKV_DEV_WAIT_TIMEOUT
    good = pkv.paged_attention_decode(q, k, v, tables, lens, w.scale, 16)
    assert pkv.device_error() == 0
    kc, vc, tabs, lens_h = w.compact_pools([0, 1, 2, 3])
    ref = oracle_attention.paged_decode_attention(w.q("cpu").numpy(), kc.numpy(), vc.numpy(), tabs, lens_h, w.scale)
    assert float(np.max(np.abs(good.cpu().numpy().astype(np.float64) - ref))) <= 2e-3
    # sizes that do not merge on chip are refused
    assert lib.pkv_test_cluster_merge_timeout(q.data_ptr(), k.data_ptr(), v.data_ptr(), tables.data_ptr(),
                                              lens.data_ptr(), 4, 8, 128, k.shape[0], 1, w.scale, 16,
                                              out.data_ptr(), 100, None) == pkv.PKV_ERR_UNSUPPORTED
