"""The allocation-free attention entry point against the ordinary one.

pkv_paged_attention_decode_static_workspace serves callers that cannot
allocate device memory (a C host program or plugin with no device allocator,
an engine whose block pools already hold all device memory, a path that must
not pay for cudaMalloc's device-wide synchronisation): it keeps the scratch in
a fixed array inside the library.  Two calls in a row, through the C ABI,
must match pkv_paged_attention_decode with a caller workspace within the
tolerance of the other attention tests; a batch too large for the array is
refused before anything runs.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_73_gb300 import _build
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = 2e-3


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def _inputs(w, dev):
    k, v = w.pools(dev)
    return (w.q(dev), k, v, torch.from_numpy(w.block_tables).to(dev), torch.from_numpy(w.context_lens).to(dev))


@pytest.mark.parametrize("make", [wl.opt13b, lambda: wl.custom(31, [1, 7, 300, 1000, 2049, 16], 4, 64, 8)],
                         ids=["opt13b_full", "ragged_small"])
def test_static_workspace_matches_caller_workspace(lib, cuda_device, make):
    w = make()
    q, k, v, tables, lens = _inputs(w, cuda_device)
    ref = pkv.paged_attention_decode(q, k, v, tables, lens, w.scale, w.block_size)
    assert pkv.device_error() == 0
    for _ in range(2):                               # the array keeps the previous call's contents
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode_static_workspace(q, k, v, tables, lens, w.scale, w.block_size, out=out)
        assert pkv.device_error() == 0
        err = (out.double() - ref.double()).abs().max().item()
        assert np.isfinite(err) and err <= ATOL, err


def test_static_workspace_refuses_oversized_batch(lib, cuda_device):
    S, H, D, B, max_blocks = 256, 40, 128, 16, 256            # 4096-token capacity: > 16 MiB of partials
    part_tokens, _ = pkv.paged_attention_plan(S, H, D, max_blocks, B)
    need = S * H * (-(-max_blocks * B // part_tokens)) * (D + 2) * 4
    assert need > pkv.paged_attention_static_workspace_bytes() == 16 << 20
    q = torch.zeros((S, H, D), dtype=torch.float16, device=cuda_device)
    kv = torch.zeros((4, H, B, D), dtype=torch.float16, device=cuda_device)
    tables = torch.zeros((S, max_blocks), dtype=torch.int32, device=cuda_device)
    lens = torch.ones(S, dtype=torch.int32, device=cuda_device)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attention_decode_static_workspace(q, kv, kv, tables, lens, 0.1, B)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE and "16777216" in str(e.value)
