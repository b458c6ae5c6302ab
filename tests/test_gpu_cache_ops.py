"""reshape_and_cache and copy_blocks on the GPU, bit-exact against the oracle's host loops."""
import numpy as np
import pytest
import torch

from oracle import cache_ops as oracle_cache_ops
from paged_kv_cache_73_gb300 import binding as pkv
from paged_kv_cache_73_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [4, 8, 16, 32])
def test_reshape_and_cache_bit_exact(cuda_device, D, B):
    w = wl.custom(200 + D + B, [30, 7, 64, 1], num_heads=5, head_dim=D, block_size=B, num_blocks=40)
    k, v = w.pools(cuda_device)
    T = 50
    key, value = wl.new_tokens(T, 5, D, w.seed, cuda_device)
    rng = np.random.default_rng(D + B)
    slots = rng.choice(40 * B, size=T, replace=False).astype(np.int64)
    slots[[3, 17, 40]] = -1                                       # padding tokens
    k_ref, v_ref = _bits(k).copy(), _bits(v).copy()
    pkv.reshape_and_cache(key, value, k, v, torch.from_numpy(slots).to(cuda_device))
    assert pkv.device_error() == 0
    oracle_cache_ops.reshape_and_cache(_bits(key), _bits(value), k_ref, v_ref, slots)
    assert np.array_equal(_bits(k), k_ref) and np.array_equal(_bits(v), v_ref)


def test_reshape_and_cache_decode_step_full_size(cuda_device):
    # the OPT-13B-shaped batch's 64 new tokens, at the last slot of each sequence
    w = wl.opt13b()
    k, v = w.pools(cuda_device)
    key, value = wl.new_tokens(w.num_seqs, 40, 128, w.seed, cuda_device)
    last = w.context_lens - 1
    slots = (w.block_tables[np.arange(w.num_seqs), last // 16].astype(np.int64) * 16 + last % 16)
    touched = sorted(set((slots // 16).tolist()))
    before_k = _bits(k[touched]).copy()
    before_v = _bits(v[touched]).copy()
    pkv.reshape_and_cache(key, value, k, v, torch.from_numpy(slots).to(cuda_device))
    assert pkv.device_error() == 0
    # oracle on the touched blocks only (remapped slots)
    remap = {b: i for i, b in enumerate(touched)}
    local = np.array([remap[int(s // 16)] * 16 + int(s % 16) for s in slots])
    oracle_cache_ops.reshape_and_cache(_bits(key), _bits(value), before_k, before_v, local)
    assert np.array_equal(_bits(k[touched]), before_k) and np.array_equal(_bits(v[touched]), before_v)


def test_reshape_and_cache_prefill_fill(cuda_device):
    # a whole prompt batch written at once (bandwidth-bound path): 8 x 2048 tokens
    H, D, B = 40, 128, 16
    N = 8 * 128 + 10
    k = torch.zeros((N, H, B, D), dtype=torch.float16, device=cuda_device)
    v = torch.zeros_like(k)
    T = 8 * 2048
    key, value = wl.new_tokens(T, H, D, 77, cuda_device)
    order = np.random.default_rng(1).permutation(N)[: T // B]
    slots = (order[:, None] * B + np.arange(B)[None, :]).reshape(-1).astype(np.int64)
    pkv.reshape_and_cache(key, value, k, v, torch.from_numpy(slots).to(cuda_device))
    assert pkv.device_error() == 0
    # every block of the permutation now holds B consecutive tokens, heads transposed
    kb = k[torch.from_numpy(order).to(cuda_device)]                 # [T/B, H, B, D]
    want = key.view(T // B, B, H, D).permute(0, 2, 1, 3)
    assert torch.equal(kb, want)
    assert torch.equal(v[torch.from_numpy(order).to(cuda_device)], value.view(T // B, B, H, D).permute(0, 2, 1, 3))


def test_reshape_and_cache_bad_slot_recorded(cuda_device):
    k = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=cuda_device)
    v = torch.zeros_like(k)
    key = torch.ones((2, 2, 64), dtype=torch.float16, device=cuda_device)
    pkv.reshape_and_cache(key, key, k, v, torch.tensor([5, 4 * 16], dtype=torch.int64, device=cuda_device))
    assert pkv.device_error() == 3
    assert torch.all(k[0, :, 5] == 1) and int((k != 0).sum()) == 2 * 64


@pytest.mark.parametrize("layers", [1, 3])
def test_copy_blocks_bit_exact(cuda_device, layers):
    H, D, B, N = 4, 128, 16, 64
    ks, vs = [], []
    for l in range(layers):
        ks.append(wl.dense_tensor((N, H, B, D), 300 + l, wl.STREAM_K, cuda_device))
        vs.append(wl.dense_tensor((N, H, B, D), 300 + l, wl.STREAM_V, cuda_device))
    pairs = np.array([[1, 40], [2, 41], [7, 50], [1, 60], [33, 3]], dtype=np.int64)
    k_ref = [_bits(x).copy() for x in ks]
    v_ref = [_bits(x).copy() for x in vs]
    pkv.copy_blocks(ks, vs, torch.from_numpy(pairs).to(cuda_device))
    assert pkv.device_error() == 0
    oracle_cache_ops.copy_blocks(k_ref, v_ref, pairs.tolist())
    for l in range(layers):
        assert np.array_equal(_bits(ks[l]), k_ref[l]) and np.array_equal(_bits(vs[l]), v_ref[l])


def test_copy_blocks_parallel_sampling_cow_pairs(cuda_device):
    # 32 prompts of 511 tokens, 4 samples each: 3 copies per prompt of the shared 15-token block
    from paged_kv_cache_73_gb300.binding import BlockManager
    B, H, D = 16, 40, 128
    N = 32 * 32 * 4 + 64
    order = wl.free_list_order(N, 1003)
    bm = BlockManager(N, B, order)
    sid = 0
    groups = []
    for p in range(32):
        bm.add_seq(sid, 511)
        for i in range(1, 4):
            bm.fork(sid, sid + i)
        groups += list(range(sid, sid + 4))
        sid += 4
    slots, pairs = bm.append_slots(groups)
    assert pairs.shape == (96, 2)
    k = torch.empty((N, H, B, D), dtype=torch.float16, device=cuda_device)
    v = torch.empty_like(k)
    gen = wl.custom(1003, [1], H, D, B)
    for pool, stream in ((k, wl.STREAM_K), (v, wl.STREAM_V)):
        pool.copy_(wl.dense_tensor(tuple(pool.shape), gen.seed, stream, cuda_device))
    srcs = pairs[:, 0]
    dsts = pairs[:, 1]
    src_k = _bits(k[torch.from_numpy(srcs).to(cuda_device)]).copy()
    other = np.setdiff1d(np.arange(N), dsts)[:200]
    other_before = _bits(k[torch.from_numpy(other).to(cuda_device)]).copy()
    pkv.copy_blocks([k], [v], torch.from_numpy(pairs).to(cuda_device))
    assert pkv.device_error() == 0
    assert np.array_equal(_bits(k[torch.from_numpy(dsts).to(cuda_device)]), src_k)
    assert np.array_equal(_bits(k[torch.from_numpy(other).to(cuda_device)]), other_before)


def test_copy_blocks_bad_pair_recorded(cuda_device):
    k = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=cuda_device)
    v = torch.zeros_like(k)
    pkv.copy_blocks([k], [v], torch.tensor([[0, 9]], dtype=torch.int64, device=cuda_device))
    assert pkv.device_error() == 4


def test_forty_layer_reshape_and_copy_in_one_launch(cuda_device):
    # the OPT-13B layer count: every layer's new tokens and copy-on-write copies in one launch each
    L, H, D, B, N, T = 40, 8, 128, 16, 24, 20
    ks = [wl.dense_tensor((N, H, B, D), 600 + l, wl.STREAM_K, cuda_device) for l in range(L)]
    vs = [wl.dense_tensor((N, H, B, D), 600 + l, wl.STREAM_V, cuda_device) for l in range(L)]
    keys = [wl.dense_tensor((T, H, D), 700 + l, wl.STREAM_NEW_K, cuda_device) for l in range(L)]
    vals = [wl.dense_tensor((T, H, D), 700 + l, wl.STREAM_NEW_V, cuda_device) for l in range(L)]
    rng = np.random.default_rng(40)
    slots = rng.choice(N * B, size=T, replace=False).astype(np.int64)
    slots[5] = -1
    k_ref = [_bits(x).copy() for x in ks]
    v_ref = [_bits(x).copy() for x in vs]
    pkv.reshape_and_cache_layers(keys, vals, ks, vs, torch.from_numpy(slots).to(cuda_device))
    assert pkv.device_error() == 0
    for l in range(L):
        oracle_cache_ops.reshape_and_cache(_bits(keys[l]), _bits(vals[l]), k_ref[l], v_ref[l], slots)
        assert np.array_equal(_bits(ks[l]), k_ref[l]) and np.array_equal(_bits(vs[l]), v_ref[l])
    pairs = np.array([[3, 20], [4, 21], [3, 22]], dtype=np.int64)
    pkv.copy_blocks(ks, vs, torch.from_numpy(pairs).to(cuda_device))
    assert pkv.device_error() == 0
    oracle_cache_ops.copy_blocks(k_ref, v_ref, pairs.tolist())
    for l in range(L):
        assert np.array_equal(_bits(ks[l]), k_ref[l]) and np.array_equal(_bits(vs[l]), v_ref[l])


def test_more_layers_than_one_launch_holds(cuda_device):
    L, H, D, B, N = 70, 2, 64, 8, 6                    # two launches of up to 64 layers
    ks = [wl.dense_tensor((N, H, B, D), 800 + l, wl.STREAM_K, cuda_device) for l in range(L)]
    vs = [wl.dense_tensor((N, H, B, D), 800 + l, wl.STREAM_V, cuda_device) for l in range(L)]
    k_ref = [_bits(x).copy() for x in ks]
    v_ref = [_bits(x).copy() for x in vs]
    pairs = np.array([[0, 5], [2, 4]], dtype=np.int64)
    pkv.copy_blocks(ks, vs, torch.from_numpy(pairs).to(cuda_device))
    oracle_cache_ops.copy_blocks(k_ref, v_ref, pairs.tolist())
    assert all(np.array_equal(_bits(ks[l]), k_ref[l]) for l in range(L))
    assert all(np.array_equal(_bits(vs[l]), v_ref[l]) for l in range(L))
