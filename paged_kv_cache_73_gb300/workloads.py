"""Seeded synthetic inputs for the paged decode-attention path.

This module is the one piece shared by the CUDA path's callers (tests, bench,
smoke) and the oracle's callers (tests, the bench's CPU baseline).  It holds
none of the method's arithmetic: no attention, no slot formula, no block
manager.  It only draws numbers:

* element values come from a counter-based generator, so any element of any
  tensor can be produced on its own, on the CPU or on a GPU, with identical
  bits (the oracle regenerates just the blocks it needs at full size);
* context lengths, sample tails and the permutation of physical block ids come
  from ``numpy.random.default_rng(seed)``;
* block tables hand out the permuted ids in order: sequence 0 takes the first
  ceil(ctx/B) ids, sequence 1 the next, and so on, with shared prompt/prefix
  blocks handed out once and referenced by every sharer.

Value recipe (the stand-in for ``K/V/q ~ N(0,1)`` in fp16): for an element with
flat index ``i`` of tensor stream ``s`` under seed ``seed``, two 32-bit
``lowbias32`` hashes (C. Wellons' integer hash) give four 16-bit uniforms
u1..u4; ``x = (u1+u2+u3+u4 - 2*65535) * 7 / 2**18`` is an Irwin-Hall(4) draw
rescaled to standard deviation 1.01, range +-3.5.  Every step is integer
arithmetic except the last, a multiply by a power of two (exact in fp32), and
the fp32->fp16 round-to-nearest-even, so CPU and GPU agree bit for bit.
Positions a table does not hold (unused physical blocks and the slots past the
last token of a sequence's last block) are filled with fp16 NaN, so a kernel
that lets them into a result, even with weight zero, fails parity.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

M32 = 0xFFFFFFFF
FP16_NAN_BITS = 0x7E00

# tensor streams of the counter-based generator
STREAM_Q = 0
STREAM_K = 1
STREAM_V = 2
STREAM_NEW_K = 3
STREAM_NEW_V = 4


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for 0 <= x < 2**32, in int64 without overflow."""
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & M32


def _lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _lowbias32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & M32
    x ^= x >> 16
    return x


def _stream_key(seed: int, stream: int) -> int:
    return _lowbias32_int(_lowbias32_int(seed * 0x9E3779B9 + 0x632BE5AB) ^ (stream * 0x85EBCA77 + 1))


def values_at(seed: int, stream: int, index: torch.Tensor) -> torch.Tensor:
    """fp16 values of stream ``stream`` at flat int64 indices ``index`` (any device)."""
    index = index.to(torch.int64)
    key = _stream_key(seed, stream)
    h1 = _lowbias32((index & M32) ^ key)
    h1 = _lowbias32(h1 ^ ((index >> 32) & M32) ^ 0x5BD1E995)
    h2 = _lowbias32(h1 ^ 0x68E31DA4)
    s = (h1 & 0xFFFF) + (h1 >> 16) + (h2 & 0xFFFF) + (h2 >> 16) - 2 * 65535
    x = (s * 7).to(torch.float32) * torch.tensor(2.0 ** -18, dtype=torch.float32, device=index.device)
    return x.to(torch.float16)


def dense_tensor(shape: Sequence[int], seed: int, stream: int, device="cpu",
                 chunk: int = 1 << 26) -> torch.Tensor:
    """A dense fp16 tensor whose flat element i is ``values_at(seed, stream, i)``."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=torch.float16, device=device)
    for start in range(0, n, chunk):
        stop = min(n, start + chunk)
        idx = torch.arange(start, stop, dtype=torch.int64, device=device)
        out[start:stop] = values_at(seed, stream, idx)
    return out.view(*shape)


def block_values(block_ids: np.ndarray, num_heads: int, block_size: int, head_dim: int,
                 seed: int, stream: int, device="cpu") -> torch.Tensor:
    """Generator contents of whole physical blocks: [len(block_ids), H, B, D] fp16.

    The flat index of element (blk, h, t, d) is its offset in a pool laid out
    [num_blocks, H, B, D], so these are exactly the values ``fill_pool`` puts in
    block ``blk`` (before the unfilled tail is set to NaN).
    """
    per_block = num_heads * block_size * head_dim
    ids = torch.as_tensor(np.asarray(block_ids, dtype=np.int64), device=device)
    idx = ids[:, None] * per_block + torch.arange(per_block, dtype=torch.int64, device=device)[None, :]
    return values_at(seed, stream, idx).view(len(block_ids), num_heads, block_size, head_dim)


@dataclasses.dataclass
class DecodeWorkload:
    """One decode batch over a paged K/V pool.

    ``block_tables`` is [S, max_blocks] int32, padded with -1.  ``block_fill``
    maps every physical block the tables reference to how many of its leading
    token slots hold data (the rest are NaN in the pool).
    """
    name: str
    seed: int
    num_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray
    block_tables: np.ndarray
    block_fill: Dict[int, int]
    notes: str = ""
    shared_blocks: int = 0        # physical blocks referenced by more than one sequence

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def logical_kv_bytes(self) -> int:
        """K and V bytes the batch attends over, counting a shared block once per sharer."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_heads * self.head_dim * 2 * 2

    def physical_kv_bytes(self) -> int:
        """K and V bytes of the distinct filled slots the batch attends over."""
        return int(sum(self.block_fill.values())) * self.num_heads * self.head_dim * 2 * 2

    def q(self, device="cpu") -> torch.Tensor:
        return dense_tensor((self.num_seqs, self.num_heads, self.head_dim), self.seed, STREAM_Q, device)

    def fill_pool(self, pool: torch.Tensor, stream: int, chunk_blocks: int = 256) -> None:
        """Write generator values into every referenced block of ``pool`` and NaN elsewhere."""
        assert pool.dtype == torch.float16 and pool.dim() == 4
        pool.view(torch.int16).fill_(FP16_NAN_BITS)
        ids = np.array(sorted(self.block_fill), dtype=np.int64)
        fills = np.array([self.block_fill[int(b)] for b in ids], dtype=np.int64)
        B = self.block_size
        for start in range(0, len(ids), chunk_blocks):
            sub = ids[start:start + chunk_blocks]
            vals = block_values(sub, self.num_heads, B, self.head_dim, self.seed, stream, pool.device)
            f = torch.as_tensor(fills[start:start + chunk_blocks], device=pool.device)
            keep = torch.arange(B, device=pool.device)[None, :] < f[:, None]          # [n, B]
            nan = torch.full((), float("nan"), dtype=torch.float16, device=pool.device)
            vals = torch.where(keep[:, None, :, None], vals, nan)
            pool[torch.as_tensor(sub, device=pool.device)] = vals

    def pools(self, device="cpu", num_blocks: Optional[int] = None):
        n = self.num_blocks if num_blocks is None else num_blocks
        shape = (n, self.num_heads, self.block_size, self.head_dim)
        k = torch.empty(shape, dtype=torch.float16, device=device)
        v = torch.empty(shape, dtype=torch.float16, device=device)
        self.fill_pool(k, STREAM_K)
        self.fill_pool(v, STREAM_V)
        return k, v

    def compact_pools(self, seqs: Sequence[int], device="cpu"):
        """CPU-sized K/V pools holding only the blocks of ``seqs``, plus their remapped tables.

        Returns (k, v, tables, lens): block i of the compact pools is physical
        block ``ids[i]`` of the full pool, and ``tables`` point into it.  Used
        to check sampled sequences of a batch far too large for the CPU.
        """
        return self.compact_pools_with(seqs, (), device)[:4]

    def compact_pools_with(self, seqs: Sequence[int], extra_blocks: Sequence[int] = (), device="cpu"):
        """compact_pools plus the physical blocks ``extra_blocks`` (e.g. the sources of copies into
        the sequences' blocks); returns (k, v, tables, lens, ids), ``ids`` the sorted physical ids
        of the compact pool's blocks."""
        seqs = list(seqs)
        tabs = self.block_tables[seqs]
        lens = self.context_lens[seqs]
        ids = sorted({int(b) for b in tabs.ravel() if b >= 0} | {int(b) for b in extra_blocks})
        remap = {b: i for i, b in enumerate(ids)}
        k = torch.empty((len(ids), self.num_heads, self.block_size, self.head_dim), dtype=torch.float16)
        v = torch.empty_like(k)
        fills = torch.tensor([self.block_fill.get(b, 0) for b in ids], dtype=torch.int64)   # unmapped: all NaN
        keep = (torch.arange(self.block_size)[None, :] < fills[:, None])[:, None, :, None]
        nan = torch.tensor(float("nan"), dtype=torch.float16)
        # generated with the full pool's flat indices, stored at the compact position
        for dst, stream in ((k, STREAM_K), (v, STREAM_V)):
            vals = block_values(np.array(ids, dtype=np.int64), self.num_heads, self.block_size,
                                self.head_dim, self.seed, stream, "cpu")
            dst.copy_(torch.where(keep, vals, nan))
        new_tabs = np.full_like(tabs, -1)
        for r in range(tabs.shape[0]):
            for j in range(tabs.shape[1]):
                if tabs[r, j] >= 0:
                    new_tabs[r, j] = remap[int(tabs[r, j])]
        return k.to(device), v.to(device), new_tabs, lens.copy(), ids


def _blocks_for(n_tokens: int, block_size: int) -> int:
    return -(-n_tokens // block_size)


class _Handout:
    """Hands out a seeded permutation of physical block ids in order."""

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.perm = rng.permutation(num_blocks).astype(np.int64)
        self.next = 0

    def take(self, n: int) -> List[int]:
        assert self.next + n <= len(self.perm), "pool too small for the workload"
        out = [int(x) for x in self.perm[self.next:self.next + n]]
        self.next += n
        return out


def _assemble(name, seed, H, D, B, num_blocks, rows, notes="") -> DecodeWorkload:
    """rows: list of (context_len, [physical ids]) per sequence."""
    S = len(rows)
    max_blk = max(1, max(len(ids) for _, ids in rows))
    tables = np.full((S, max_blk), -1, dtype=np.int32)
    lens = np.zeros(S, dtype=np.int32)
    fill: Dict[int, int] = {}
    refs: Dict[int, int] = {}
    for s, (ctx, ids) in enumerate(rows):
        lens[s] = ctx
        tables[s, :len(ids)] = ids
        for j, b in enumerate(ids):
            f = min(B, ctx - j * B)
            fill[b] = max(fill.get(b, 0), f)
            refs[b] = refs.get(b, 0) + 1
    shared = sum(1 for r in refs.values() if r > 1)
    return DecodeWorkload(name, seed, H, D, B, num_blocks, lens, tables, fill, notes, shared)


def tiny(seed: int = 1001) -> DecodeWorkload:
    """3 sequences with context lengths 7, 5, 12; B=4; 2 heads x 64; 32-block pool, permuted ids."""
    rng = np.random.default_rng(seed)
    H, D, B, N = 2, 64, 4, 32
    hand = _Handout(N, rng)
    rows = [(c, hand.take(_blocks_for(c, B))) for c in (7, 5, 12)]
    return _assemble("tiny", seed, H, D, B, N, rows)


def opt13b(seed: int = 1002, num_seqs: int = 64, lo: int = 128, hi: int = 2048,
           block_size: int = 16, pool_factor: float = 1.25) -> DecodeWorkload:
    """OPT-13B-shaped single layer: 40 heads x 128, B=16, batch 64, ctx ~ U[128, 2048]."""
    rng = np.random.default_rng(seed)
    H, D, B = 40, 128, block_size
    ctx = rng.integers(lo, hi + 1, size=num_seqs)
    need = int(sum(_blocks_for(int(c), B) for c in ctx))
    N = int(math.ceil(need * pool_factor))
    hand = _Handout(N, rng)
    rows = [(int(c), hand.take(_blocks_for(int(c), B))) for c in ctx]
    return _assemble("opt13b", seed, H, D, B, N, rows,
                     f"S={num_seqs} ctx~U[{lo},{hi}] B={B} pool={N} blocks ({pool_factor}x need)")


def parallel_sampling(seed: int = 1003, prompts: int = 32, prompt_len: int = 512, n: int = 4,
                      tail_lo: int = 1, tail_hi: int = 256, block_size: int = 16,
                      pool_factor: float = 1.25) -> DecodeWorkload:
    """``prompts`` prompts, each with ``n`` samples sharing the prompt's blocks.

    Each sample then holds ``tail ~ U[tail_lo, tail_hi]`` tokens of its own.
    Where the prompt's last block is partial, sample 0..n-2 hold a private
    copy of it (the state after copy-on-write) and sample n-1 keeps the
    original; the tables here are that post-copy state.
    """
    rng = np.random.default_rng(seed)
    H, D, B = 40, 128, block_size
    tails = rng.integers(tail_lo, tail_hi + 1, size=prompts * n)
    full, part = divmod(prompt_len, B)
    need = prompts * (full + (1 if part else 0))
    for t in tails:
        need += _blocks_for(part + int(t), B) if part else _blocks_for(int(t), B)
    N = int(math.ceil(need * pool_factor))
    hand = _Handout(N, rng)
    rows = []
    for p in range(prompts):
        shared = hand.take(full)
        last = hand.take(1) if part else []
        for i in range(n):
            t = int(tails[p * n + i])
            ctx = prompt_len + t
            own_last = last if (not part or i == n - 1) else hand.take(1)
            rest = _blocks_for(ctx, B) - full - len(own_last)
            rows.append((ctx, shared + own_last + hand.take(rest)))
    return _assemble("parallel_sampling" if not part else "parallel_sampling_cow", seed, H, D, B, N, rows,
                     f"{prompts} prompts x {prompt_len} tok, n={n}, tails~U[{tail_lo},{tail_hi}]")


def shared_prefix(seed: int = 1004, requests: int = 256, prefix_len: int = 1024,
                  suffix_lo: int = 32, suffix_hi: int = 512, block_size: int = 16,
                  pool_factor: float = 1.25) -> DecodeWorkload:
    """``requests`` sequences sharing one prefix's blocks, each with a private suffix."""
    rng = np.random.default_rng(seed)
    H, D, B = 40, 128, block_size
    suf = rng.integers(suffix_lo, suffix_hi + 1, size=requests)
    full, part = divmod(prefix_len, B)
    need = full + (1 if part else 0) + sum(_blocks_for(prefix_len + int(s), B) - full for s in suf)
    N = int(math.ceil(need * pool_factor))
    hand = _Handout(N, rng)
    prefix = hand.take(full)
    rows = []
    for s in suf:
        ctx = prefix_len + int(s)
        rows.append((ctx, prefix + hand.take(_blocks_for(ctx, B) - full)))
    return _assemble("shared_prefix", seed, H, D, B, N, rows,
                     f"{requests} requests, prefix {prefix_len} tok, suffix~U[{suffix_lo},{suffix_hi}]")


def capacity(seed: int = 1005, num_seqs: int = 64, block_size: int = 16, ctx: int = 2048,
             num_blocks: Optional[int] = None) -> DecodeWorkload:
    """Every sequence at ``ctx`` tokens, ids drawn from a permutation of a pool of ``num_blocks``."""
    rng = np.random.default_rng(seed)
    H, D, B = 40, 128, block_size
    need = num_seqs * _blocks_for(ctx, B)
    N = need if num_blocks is None else int(num_blocks)
    assert N >= need
    hand = _Handout(N, rng)
    rows = [(ctx, hand.take(_blocks_for(ctx, B))) for _ in range(num_seqs)]
    return _assemble(f"capacity_S{num_seqs}_B{B}", seed, H, D, B, N, rows,
                     f"S={num_seqs} ctx={ctx} B={B} pool={N} blocks")


def custom(seed: int, context_lens: Sequence[int], num_heads: int, head_dim: int, block_size: int,
           num_blocks: Optional[int] = None, name: str = "custom") -> DecodeWorkload:
    """Independent sequences with the given lengths (edge cases, ragged tails)."""
    rng = np.random.default_rng(seed)
    need = sum(_blocks_for(int(c), block_size) for c in context_lens)
    N = max(1, need) if num_blocks is None else int(num_blocks)
    hand = _Handout(N, rng)
    rows = [(int(c), hand.take(_blocks_for(int(c), block_size))) for c in context_lens]
    return _assemble(name, seed, num_heads, head_dim, block_size, N, rows)


def new_tokens(num_tokens: int, num_heads: int, head_dim: int, seed: int, device="cpu"):
    """Key and value rows [T, H, D] fp16 of the tokens a decode step appends."""
    shape = (num_tokens, num_heads, head_dim)
    return (dense_tensor(shape, seed, STREAM_NEW_K, device),
            dense_tensor(shape, seed, STREAM_NEW_V, device))


def free_list_order(num_blocks: int, seed: int) -> np.ndarray:
    """The seeded order in which a block manager hands out physical ids (the 'shuffled pool')."""
    return np.random.default_rng(seed).permutation(num_blocks).astype(np.int32)


def from_tables(name: str, seed: int, num_heads: int, head_dim: int, block_size: int, num_blocks: int,
                block_tables: np.ndarray, context_lens: np.ndarray, notes: str = "") -> DecodeWorkload:
    """A workload over tables made elsewhere (e.g. by a block manager); -1 pads each row."""
    rows = []
    for s in range(block_tables.shape[0]):
        ctx = int(context_lens[s])
        nb = _blocks_for(ctx, block_size)
        rows.append((ctx, [int(b) for b in block_tables[s, :nb]]))
    w = _assemble(name, seed, num_heads, head_dim, block_size, num_blocks, rows, notes)
    w.block_tables = np.ascontiguousarray(block_tables.astype(np.int32))
    return w


# ---- inputs for the hard regimes of the softmax ------------------------------------------------------
#
# These draw ordinary Gaussian numbers (numpy, seeded) at a chosen spread instead of the counter
# stream, on the CPU, for batches small enough to build there: spreads far above 1 (logits spanning
# tens or hundreds of units), far below the fp16 normal range (subnormal keys or values), and keys
# laid along each query's direction with a coefficient that follows the token's position, so that
# q.k_t moves steadily from one end of the context to the other.

def _nan_outside(w: DecodeWorkload, pool: np.ndarray) -> np.ndarray:
    """NaN in every slot of ``pool`` that no table row maps (as fill_pool does)."""
    keep = np.zeros(pool.shape[0] * w.block_size, dtype=bool)
    for b, f in w.block_fill.items():
        keep[b * w.block_size: b * w.block_size + f] = True
    flat = pool.reshape(pool.shape[0], pool.shape[1], w.block_size, -1).transpose(0, 2, 1, 3)
    flat = flat.reshape(pool.shape[0] * w.block_size, pool.shape[1], -1)
    flat[~keep] = np.nan
    return flat.reshape(pool.shape[0], w.block_size, pool.shape[1], -1).transpose(0, 2, 1, 3).copy()


def gaussian_inputs(w: DecodeWorkload, seed: int, q_std: float = 1.0, k_std: float = 1.0, v_std: float = 1.0):
    """(q [S, H, D], k pool, v pool) as CPU fp16 tensors: independent N(0, std^2) draws rounded to
    fp16 (tiny spreads give fp16 subnormals), NaN in the slots no table maps."""
    rng = np.random.default_rng(seed)
    S, H, D, B, N = w.num_seqs, w.num_heads, w.head_dim, w.block_size, w.num_blocks
    q = (rng.standard_normal((S, H, D)) * q_std).astype(np.float16)
    k = _nan_outside(w, (rng.standard_normal((N, H, B, D)) * k_std).astype(np.float16))
    v = _nan_outside(w, (rng.standard_normal((N, H, B, D)) * v_std).astype(np.float16))
    return torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v)


def ramp_inputs(w: DecodeWorkload, seed: int, first: float, last: float, q_norm: float = 8.0,
                noise: float = 0.02, rows_per_seq: Optional[Sequence[int]] = None):
    """q and K/V pools in which q[s, h] . k_t runs linearly from about ``first`` (t = 0) to about
    ``last`` (t = ctx_s - 1): q[s, h] = q_norm * u with u a random unit vector per (s, h), and
    k_t = c_t / q_norm * u + N(0, noise^2) per element with c_t the ramp value; v ~ N(0, 1).  All
    fp16 on the CPU, NaN in unmapped slots.  With ``rows_per_seq``, q has that many rows per
    sequence (prefill: every new token of a sequence shares its u), stacked in sequence order."""
    rng = np.random.default_rng(seed)
    S, H, D, B, N = w.num_seqs, w.num_heads, w.head_dim, w.block_size, w.num_blocks
    u = rng.standard_normal((S, H, D))
    u /= np.linalg.norm(u, axis=2, keepdims=True)
    k = rng.standard_normal((N, H, B, D)) * noise
    for s in range(S):
        ctx = int(w.context_lens[s])
        for t in range(ctx):
            c = first + (last - first) * (t / max(ctx - 1, 1))
            k[int(w.block_tables[s, t // B]), :, t % B, :] += (c / q_norm) * u[s]
    v = rng.standard_normal((N, H, B, D))
    rows = [1] * S if rows_per_seq is None else [int(r) for r in rows_per_seq]
    q = np.concatenate([np.repeat((q_norm * u[s])[None], rows[s], axis=0) for s in range(S)], axis=0)
    return (torch.from_numpy(q.astype(np.float16)), torch.from_numpy(_nan_outside(w, k.astype(np.float16))),
            torch.from_numpy(_nan_outside(w, v.astype(np.float16))))
