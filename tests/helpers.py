"""Shared helpers of the GPU parity tests: run the CUDA path through the binding,
run the oracle on the same seeded inputs (regenerated on the CPU), compare."""
import numpy as np
import torch

from oracle import attention as oracle_attention
from paged_kv_cache_73_gb300 import binding as pkv

ATOL = 2e-3   # max |o_gpu - o_oracle| for fp16 K/V, fp32 accumulation, fp16 output


def device_inputs(w, dev, num_blocks=None):
    k, v = w.pools(dev, num_blocks=num_blocks)
    q = w.q(dev)
    tables = torch.from_numpy(w.block_tables).to(dev)
    lens = torch.from_numpy(w.context_lens).to(dev)
    return q, k, v, tables, lens


def gpu_attention(w, dev, inputs=None, workspace=None):
    q, k, v, tables, lens = inputs if inputs is not None else device_inputs(w, dev)
    out = pkv.paged_attention_decode(q, k, v, tables, lens, w.scale, w.block_size, workspace=workspace)
    code = pkv.device_error()
    assert code == 0, f"device check {pkv.DEV_CODES.get(code, code)}"
    return out


def oracle_on(w, seqs):
    """Oracle output for sequences ``seqs`` of workload ``w``, from CPU-regenerated blocks."""
    kc, vc, tabs, lens = w.compact_pools(seqs)
    q = w.q("cpu").numpy()[list(seqs)]
    return oracle_attention.paged_decode_attention(q, kc.numpy(), vc.numpy(), tabs, lens, w.scale)


def max_err(gpu_rows, ref):
    g = gpu_rows.detach().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), "non-finite output"
    return float(np.max(np.abs(g - ref))) if ref.size else 0.0


def sample_seqs(w, k=4, seed=0):
    """The longest and shortest sequences plus k-2 random ones."""
    lens = w.context_lens
    rng = np.random.default_rng(seed)
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    while len(pick) < min(k, len(lens)):
        pick.add(int(rng.integers(0, len(lens))))
    return sorted(pick)
