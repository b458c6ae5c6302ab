"""The bench's multi-rank path on CPU (gloo, world size 2): each rank builds its own
independent decode batch (weak scaling, no data exchange) through the host block
manager, and the whole-job figures are the byte sum over the slowest rank's time."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    seed = bench.SEED + 7919 * rank
    x = bench.build_step_inputs(seed)
    w, slots = x["w"], x["slots"]
    # per-rank step time and bytes: stand-ins with known max / sum
    (step_ms, e2e_ms, attn_ms), (kv_total,) = bench.reduce_over_ranks(
        [1.0 + rank, 3.0 - rank, 0.5], [float(w.logical_kv_bytes())], world, "cpu")
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), lens=w.context_lens, tables=w.block_tables, slots=slots,
             step_ms=step_ms, e2e_ms=e2e_ms, kv_total=kv_total, own=w.logical_kv_bytes())
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_ranks_weak_scaling(tmp_path):
    from paged_kv_cache_73_gb300 import _build
    _build.build()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npz")
    r1 = np.load(tmp_path / "rank1.npz")
    # independent batches: different length draws, each a valid decode batch of 64 sequences
    assert r0["lens"].shape == r1["lens"].shape == (64,)
    assert not np.array_equal(r0["lens"], r1["lens"])
    for r in (r0, r1):
        lens, tables, slots = r["lens"], r["tables"], r["slots"]
        for s in range(64):
            nb = -(-int(lens[s]) // 16)
            assert (tables[s, :nb] >= 0).all() and (tables[s, nb:] == -1).all()
            last = int(lens[s]) - 1
            assert slots[s] == tables[s, last // 16] * 16 + last % 16      # the new token's slot
    # whole job: slowest rank's time, all ranks' bytes
    for r in (r0, r1):
        assert float(r["step_ms"]) == 2.0 and float(r["e2e_ms"]) == 3.0
        assert float(r["kv_total"]) == float(r0["own"]) + float(r1["own"])
