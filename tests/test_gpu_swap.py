"""swap_blocks on the GPU: whole blocks between HBM pools and page-locked host pools (Grace
memory over the C2C link), bit-exact against the oracle's host loop."""
import numpy as np
import pytest
import torch

from oracle import cache_ops as oracle_cache_ops
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().numpy().view(np.uint16)


def _pools(L, N, H, B, D, seed, device, pinned=False):
    ks, vs = [], []
    for l in range(L):
        k = wl.dense_tensor((N, H, B, D), seed + l, wl.STREAM_K, "cpu")
        v = wl.dense_tensor((N, H, B, D), seed + l, wl.STREAM_V, "cpu")
        if device == "cpu":
            ks.append(k.pin_memory() if pinned else k)
            vs.append(v.pin_memory() if pinned else v)
        else:
            ks.append(k.to(device))
            vs.append(v.to(device))
    return ks, vs


@pytest.mark.parametrize("L,B,D", [(1, 16, 128), (3, 8, 64), (40, 16, 128)])
def test_swap_out_and_in_bit_exact(cuda_device, L, B, D):
    H, N, M = 4, 48, 20
    dk, dv = _pools(L, N, H, B, D, 500, cuda_device)
    hk, hv = _pools(L, M, H, B, D, 900, "cpu", pinned=True)
    rng = np.random.default_rng(L)
    src = rng.choice(N, size=12, replace=False)
    dst = rng.choice(M, size=12, replace=False)
    out_map = np.stack([src, dst], 1).astype(np.int64)
    want_h = [[_bits(x).copy() for x in side] for side in (hk, hv)]
    dev_bits = [[_bits(x) for x in side] for side in (dk, dv)]
    # swap-out: device pools -> pinned host pools, mapping in pinned host memory
    pkv.swap_blocks(dk, dv, hk, hv, torch.from_numpy(out_map).pin_memory())
    assert pkv.device_error() == 0
    oracle_cache_ops.swap_blocks(dev_bits[0], dev_bits[1], want_h[0], want_h[1], out_map.tolist())
    for l in range(L):
        assert np.array_equal(hk[l].numpy().view(np.uint16), want_h[0][l])
        assert np.array_equal(hv[l].numpy().view(np.uint16), want_h[1][l])
    # swap-in: host -> other device blocks, mapping on the device
    back = np.stack([dst, rng.permutation(np.setdiff1d(np.arange(N), src))[:12]], 1).astype(np.int64)
    want_d = [[x.copy() for x in side] for side in dev_bits]
    pkv.swap_blocks(hk, hv, dk, dv, torch.from_numpy(back).to(cuda_device))
    assert pkv.device_error() == 0
    oracle_cache_ops.swap_blocks(want_h[0], want_h[1], want_d[0], want_d[1], back.tolist())
    for l in range(L):
        assert np.array_equal(_bits(dk[l]), want_d[0][l]) and np.array_equal(_bits(dv[l]), want_d[1][l])


def test_swap_between_device_pools(cuda_device):
    H, B, D = 2, 32, 128
    ak, av = _pools(1, 8, H, B, D, 1, cuda_device)
    bk, bv = _pools(1, 8, H, B, D, 2, cuda_device)
    want = [_bits(bk[0]).copy(), _bits(bv[0]).copy()]
    m = np.array([[0, 7], [5, 2]], dtype=np.int64)
    pkv.swap_blocks(ak, av, bk, bv, torch.from_numpy(m).to(cuda_device))
    oracle_cache_ops.swap_blocks([_bits(ak[0])], [_bits(av[0])], [want[0]], [want[1]], m.tolist())
    assert np.array_equal(_bits(bk[0]), want[0]) and np.array_equal(_bits(bv[0]), want[1])


def test_swap_refuses_pageable_host_memory(cuda_device, lib=None):
    dk, dv = _pools(1, 4, 2, 16, 64, 3, cuda_device)
    hk = [torch.zeros((4, 2, 16, 64), dtype=torch.float16)]      # pageable
    lib = pkv.load()
    kp = (pkv.ctypes.c_void_p * 1)(dk[0].data_ptr())
    vp = (pkv.ctypes.c_void_p * 1)(dv[0].data_ptr())
    hp = (pkv.ctypes.c_void_p * 1)(hk[0].data_ptr())
    m = torch.tensor([[0, 1]], dtype=torch.int64, device=cuda_device)
    cast = lambda a: pkv.ctypes.cast(a, pkv.ctypes.c_void_p)
    rc = lib.pkv_swap_blocks(cast(kp), cast(vp), cast(hp), cast(hp), 1, m.data_ptr(), 1, 2, 64, 16, 4, 4, None)
    assert rc == pkv.PKV_ERR_INVALID_ARG and b"page-locked" in lib.pkv_last_error()


def test_swap_bad_pair_recorded(cuda_device):
    dk, dv = _pools(1, 4, 2, 16, 64, 4, cuda_device)
    hk, hv = _pools(1, 2, 2, 16, 64, 5, "cpu", pinned=True)
    before = hk[0].clone()
    pkv.swap_blocks(dk, dv, hk, hv, torch.tensor([[1, 2]], dtype=torch.int64, device=cuda_device))
    assert pkv.device_error() == 4 and torch.equal(hk[0], before)


def test_preempted_group_round_trip_keeps_attention(cuda_device):
    # a request's four samples are preempted: the block manager moves the group to the host pool's
    # manager, swap_blocks copies the group's blocks out, the freed device blocks are overwritten,
    # and the group comes back into other device blocks; attention over the restored tables is the
    # same, bit for bit (the kernel's result does not depend on physical ids)
    B, H, D, N, M, maxb = 16, 4, 128, 96, 64, 24
    dev_bm = pkv.BlockManager(N, B, np.random.default_rng(1).permutation(N))
    host_bm = pkv.BlockManager(M, B, np.random.default_rng(2).permutation(M))
    dev_bm.add_seq(0, 300)
    for c in (1, 2, 3):
        dev_bm.fork(0, c)
    for s in range(4):
        dev_bm.append_slot(s)                               # copies of the shared partly filled block
    dev_bm.add_seq(10, 200)                                 # another request, left on the device
    group = [0, 1, 2, 3]
    k = wl.dense_tensor((N, H, B, D), 700, wl.STREAM_K, cuda_device)
    v = wl.dense_tensor((N, H, B, D), 700, wl.STREAM_V, cuda_device)
    q = wl.dense_tensor((len(group), H, D), 701, wl.STREAM_Q, cuda_device)
    hk = torch.zeros((M, H, B, D), dtype=torch.float16).pin_memory()
    hv = torch.zeros((M, H, B, D), dtype=torch.float16).pin_memory()

    def attend():
        tables, lens = dev_bm.block_tables(group, maxb)
        return pkv.paged_attention_decode(q, k, v, torch.from_numpy(tables).to(cuda_device),
                                          torch.from_numpy(lens).to(cuda_device), D ** -0.5, B)

    before = attend()
    out_pairs = dev_bm.swap(host_bm, group)
    pkv.swap_blocks([k], [v], [hk], [hv], torch.from_numpy(out_pairs).to(cuda_device))
    freed = torch.from_numpy(out_pairs[:, 0]).to(cuda_device)
    k[freed] = float("nan")                                 # reused by someone else meanwhile
    v[freed] = float("nan")
    dev_bm.add_seq(20, B * 3)
    in_pairs = host_bm.swap(dev_bm, group)
    pkv.swap_blocks([hk], [hv], [k], [v], torch.from_numpy(in_pairs).to(cuda_device))
    after = attend()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert len(out_pairs) == len(in_pairs) == 19 + 3         # 18 shared full blocks + the partial + 3 copies
    assert torch.equal(before, after)
