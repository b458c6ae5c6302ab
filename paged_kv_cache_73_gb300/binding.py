"""Thin Python binding of libpkv.so (include/pkv.h): argument marshalling only.

Each function here calls the C entry point of the same name without the
``pkv_`` prefix (``paged_attention_decode`` -> ``pkv_paged_attention_decode``).
Torch supplies device memory and the stream; every step of the computation
runs in the library's kernels.  There is no fallback: if libpkv.so is missing
or a call fails, a ``PkvError`` is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

from . import _build

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_CUDA = -3
PKV_ERR_WORKSPACE = -4
PKV_ERR_OOM = -5
PKV_ERR_DEVICE_CHECK = -6
PKV_ERR_NOT_FOUND = -7

DEV_CODES = {0: "ok", 1: "bad block id", 2: "bad context length", 3: "bad slot", 4: "bad copy pair",
             5: "wait timeout", 6: "bad query range", 7: "shared prefix mismatch"}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkv status {status}: {message}")
        self.status = status


class PkvOutOfBlocks(PkvError, MemoryError):
    pass


_c = ctypes
_P = _c.c_void_p
_I = _c.c_int
_I64 = _c.c_int64
_SZ = _c.c_size_t

_SIGNATURES = {
    "pkv_last_error": (_c.c_char_p, []),
    "pkv_version": (_I, []),
    "pkv_device_error": (_I, [_P, _I, _c.POINTER(_I)]),
    "pkv_paged_attention_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "pkv_paged_attention_plan": (_I, [_I, _I, _I, _I, _I, _c.POINTER(_I), _c.POINTER(_I)]),
    "pkv_paged_attention_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _c.c_float, _I, _P, _P, _SZ, _P]),
    "pkv_paged_attention_decode_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _c.c_float, _I,
                                               _P, _P, _SZ, _P]),
    "pkv_paged_attention_shared_prefix_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "pkv_paged_attention_decode_shared_prefix": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                                      _c.c_float, _I, _P, _P, _SZ, _P]),
    "pkv_paged_attention_static_workspace_bytes": (_SZ, []),
    "pkv_paged_attention_decode_static_workspace": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _c.c_float, _I,
                                                         _P, _P]),
    "pkv_paged_attention_prefill": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _c.c_float, _I, _P,
                                         _P]),
    "pkv_test_cluster_merge_timeout": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _c.c_float, _I, _P, _I, _P]),
    "pkv_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "pkv_reshape_and_cache_layers": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P]),
    "pkv_copy_blocks": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _P]),
    "pkv_swap_blocks": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pkv_bm_create": (_P, [_I, _I, _P]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_add_seq": (_I, [_P, _I64, _I, _P]),
    "pkv_bm_fork": (_I, [_P, _I64, _I64]),
    "pkv_bm_append_slot": (_I, [_P, _I64, _c.POINTER(_I64), _c.POINTER(_c.c_int32), _c.POINTER(_c.c_int32)]),
    "pkv_bm_append_slots": (_I, [_P, _P, _I, _P, _P, _c.POINTER(_I)]),
    "pkv_bm_free": (_I, [_P, _I64]),
    "pkv_bm_register_prefix": (_I, [_P, _I64, _I, _P]),
    "pkv_bm_add_seq_with_prefix": (_I, [_P, _I64, _I64, _I, _P, _P, _c.POINTER(_I)]),
    "pkv_bm_extend": (_I, [_P, _I64, _I, _P, _P, _c.POINTER(_I)]),
    "pkv_bm_drop_prefix": (_I, [_P, _I64]),
    "pkv_bm_block_table": (_I, [_P, _I64, _P, _I, _c.POINTER(_I), _c.POINTER(_I)]),
    "pkv_bm_block_tables": (_I, [_P, _P, _I, _P, _I, _P]),
    "pkv_bm_beam_step": (_I, [_P, _P, _P, _I, _P, _I, _P, _P, _c.POINTER(_I)]),
    "pkv_bm_swap": (_I, [_P, _P, _P, _I, _P, _I, _c.POINTER(_I)]),
    "pkv_bm_ref_histogram": (_I, [_P, _P, _I]),
    "pkv_bm_counters": (_I, [_P, _P, _I]),
    "pkv_bm_ref_count": (_I, [_P, _c.c_int32]),
    "pkv_bm_stats": (_I, [_P, _c.POINTER(_I), _c.POINTER(_I64), _c.POINTER(_I64)]),
}

_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libpkv.so (building it first only if asked); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise PkvError(PKV_ERR_CUDA, f"{path} is missing: build it with __graft_entry__.build() "
                                         "or python -m paged_kv_cache_73_gb300._build")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != PKV_OK:
        msg = load().pkv_last_error().decode(errors="replace")
        if status == PKV_ERR_OOM:
            raise PkvOutOfBlocks(status, msg)
        raise PkvError(status, msg)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, dim: int, cuda: bool = True,
          host_ok: bool = False) -> None:
    """dtype, rank and contiguity; on the device, or (host_ok) in page-locked host memory, which
    the kernels read or write directly across the host link."""
    placed = t.is_cuda or (host_ok and t.is_pinned())
    if t.dtype != dtype or t.dim() != dim or not t.is_contiguous() or (cuda and not placed):
        where = "CUDA or page-locked host " if host_ok else ("CUDA " if cuda else "")
        raise PkvError(PKV_ERR_INVALID_ARG,
                       f"{name}: want a contiguous {where}{dtype} tensor of rank {dim}, "
                       f"got {t.dtype} {tuple(t.shape)} contiguous={t.is_contiguous()} device={t.device}")
    if t.is_cuda and t.device.index != torch.cuda.current_device():
        # the library launches on the current device; another device's memory would be a peer read
        raise PkvError(PKV_ERR_INVALID_ARG,
                       f"{name}: on {t.device}, but the current CUDA device is cuda:{torch.cuda.current_device()} "
                       f"(make it current, e.g. with torch.cuda.device({t.device}))")


def _out_like(q: torch.Tensor) -> torch.Tensor:
    """A result buffer shaped as q: on the device, or page-locked if q is page-locked host memory."""
    if q.is_cuda:
        return torch.empty_like(q)
    return torch.empty(tuple(q.shape), dtype=q.dtype).pin_memory()


# ---- device entry points -------------------------------------------------------------------

def version() -> int:
    return load().pkv_version()


def device_error(stream=None, reset: bool = True) -> int:
    """Synchronise the stream; return the first recorded device-check code (0 = none)."""
    code = _c.c_int(0)
    st = load().pkv_device_error(_stream(stream), int(reset), _c.byref(code))
    if st not in (PKV_OK, PKV_ERR_DEVICE_CHECK):
        _check(st)
    return code.value


def paged_attention_workspace_size(num_seqs: int, num_heads: int, head_dim: int, max_blocks_per_seq: int,
                                   block_size: int) -> int:
    return int(load().pkv_paged_attention_workspace_size(num_seqs, num_heads, head_dim, max_blocks_per_seq,
                                                         block_size))


def paged_attention_plan(num_seqs: int, num_heads: int, head_dim: int, max_blocks_per_seq: int,
                         block_size: int) -> Tuple[int, int]:
    """(partition tokens, kernels per call) that paged_attention_decode will use on this device."""
    pt = _c.c_int(0)
    nk = _c.c_int(0)
    _check(load().pkv_paged_attention_plan(num_seqs, num_heads, head_dim, max_blocks_per_seq, block_size,
                                           ctypes.byref(pt), ctypes.byref(nk)))
    return pt.value, nk.value


def workspace_for(num_seqs: int, num_heads: int, head_dim: int, max_blocks_per_seq: int, block_size: int,
                  device) -> Optional[torch.Tensor]:
    n = paged_attention_workspace_size(num_seqs, num_heads, head_dim, max_blocks_per_seq, block_size)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device) if n else None


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           block_size: int, out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[s, h] = softmax attention of q[s, h] over the sequence's paged K/V (fp32 accumulate, fp16 out).

    q, block_tables, context_lens and out may be page-locked host tensors: the kernels read and
    write them across the host link (no staging copy).  The pools and the workspace are device memory."""
    _need(q, "q", torch.float16, 3, host_ok=True)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(block_tables, "block_tables", torch.int32, 2, host_ok=True)
    _need(context_lens, "context_lens", torch.int32, 1, host_ok=True)
    S, H, D = q.shape
    N = k_cache.shape[0]
    if tuple(k_cache.shape) != (N, H, block_size, D) or v_cache.shape != k_cache.shape:
        raise PkvError(PKV_ERR_INVALID_ARG, f"cache shape {tuple(k_cache.shape)} does not match "
                                            f"[N, {H}, {block_size}, {D}]")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise PkvError(PKV_ERR_INVALID_ARG, "block_tables / context_lens rows != num_seqs")
    if out is None:
        out = _out_like(q)
    else:
        _need(out, "out", torch.float16, 3, host_ok=True)
    max_blocks = block_tables.shape[1]
    if workspace is None:
        workspace = workspace_for(S, H, D, max_blocks, block_size, k_cache.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_attention_decode(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
        S, H, D, N, max_blocks, float(scale), block_size, out.data_ptr(), _ptr(workspace), ws_bytes,
        _stream(stream)))
    return out


def paged_attention_decode_append(q: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                                  slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                  block_size: int, out: Optional[torch.Tensor] = None,
                                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """reshape_and_cache(key, value, slot_mapping) then paged_attention_decode, in one launch: each
    sequence's new K/V row is stored at its slot and attended to in the same kernel.  The step
    inputs (q, key, value, slot_mapping, tables, lengths) and out may be page-locked host tensors."""
    _need(q, "q", torch.float16, 3, host_ok=True)
    _need(key, "key", torch.float16, 3, host_ok=True)
    _need(value, "value", torch.float16, 3, host_ok=True)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, host_ok=True)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(block_tables, "block_tables", torch.int32, 2, host_ok=True)
    _need(context_lens, "context_lens", torch.int32, 1, host_ok=True)
    S, H, D = q.shape
    N = k_cache.shape[0]
    if tuple(k_cache.shape) != (N, H, block_size, D) or v_cache.shape != k_cache.shape:
        raise PkvError(PKV_ERR_INVALID_ARG, f"cache shape {tuple(k_cache.shape)} does not match "
                                            f"[N, {H}, {block_size}, {D}]")
    if key.shape != q.shape or value.shape != q.shape or slot_mapping.shape[0] != S:
        raise PkvError(PKV_ERR_INVALID_ARG, "key / value must be [num_seqs, H, D] and slot_mapping [num_seqs]")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise PkvError(PKV_ERR_INVALID_ARG, "block_tables / context_lens rows != num_seqs")
    if out is None:
        out = _out_like(q)
    else:
        _need(out, "out", torch.float16, 3, host_ok=True)
    max_blocks = block_tables.shape[1]
    if workspace is None:
        workspace = workspace_for(S, H, D, max_blocks, block_size, k_cache.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_attention_decode_append(
        q.data_ptr(), key.data_ptr(), value.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(), S, H, D, N, max_blocks,
        float(scale), block_size, out.data_ptr(), _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def paged_attention_shared_prefix_workspace_size(num_seqs: int, num_heads: int, head_dim: int,
                                                 max_blocks_per_seq: int, block_size: int) -> int:
    return int(load().pkv_paged_attention_shared_prefix_workspace_size(num_seqs, num_heads, head_dim,
                                                                       max_blocks_per_seq, block_size))


def paged_attention_decode_shared_prefix(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                         block_tables: torch.Tensor, context_lens: torch.Tensor,
                                         group_start: torch.Tensor, prefix_lens: torch.Tensor, scale: float,
                                         block_size: int, max_group_size: int, out: Optional[torch.Tensor] = None,
                                         workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """As paged_attention_decode, for sequences grouped by a shared prefix (read once per group).
    block_tables, context_lens, group_start, prefix_lens and out may be page-locked host tensors;
    q must be on the device (the prefix part loads it by TMA)."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(block_tables, "block_tables", torch.int32, 2, host_ok=True)
    _need(context_lens, "context_lens", torch.int32, 1, host_ok=True)
    _need(group_start, "group_start", torch.int32, 1, host_ok=True)
    _need(prefix_lens, "prefix_lens", torch.int32, 1, host_ok=True)
    S, H, D = q.shape
    N = k_cache.shape[0]
    G = prefix_lens.shape[0]
    if tuple(k_cache.shape) != (N, H, block_size, D) or v_cache.shape != k_cache.shape:
        raise PkvError(PKV_ERR_INVALID_ARG, f"cache shape {tuple(k_cache.shape)} does not match "
                                            f"[N, {H}, {block_size}, {D}]")
    if block_tables.shape[0] != S or context_lens.shape[0] != S or group_start.shape[0] != G + 1:
        raise PkvError(PKV_ERR_INVALID_ARG, "block_tables / context_lens rows != num_seqs or group_start != groups + 1")
    if out is None:
        out = _out_like(q)
    else:
        _need(out, "out", torch.float16, 3, host_ok=True)
    max_blocks = block_tables.shape[1]
    if workspace is None:
        n = paged_attention_shared_prefix_workspace_size(S, H, D, max_blocks, block_size)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=k_cache.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().pkv_paged_attention_decode_shared_prefix(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
        group_start.data_ptr(), prefix_lens.data_ptr(), G, int(max_group_size), S, H, D, N, max_blocks,
        float(scale), block_size, out.data_ptr(), _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def paged_attention_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, query_start: torch.Tensor,
                            scale: float, block_size: int, max_query_len: int,
                            out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The new tokens of each sequence over its cached context plus, causally, themselves."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(query_start, "query_start", torch.int32, 1)
    T, H, D = q.shape
    S = context_lens.shape[0]
    if query_start.shape[0] != S + 1 or block_tables.shape[0] != S:
        raise PkvError(PKV_ERR_INVALID_ARG, "query_start must have num_seqs + 1 entries")
    if tuple(k_cache.shape[1:]) != (H, block_size, D) or v_cache.shape != k_cache.shape:
        raise PkvError(PKV_ERR_INVALID_ARG, "cache shape does not match [N, H, B, D]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.float16, 3)
    _check(load().pkv_paged_attention_prefill(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
        query_start.data_ptr(), S, T, int(max_query_len), H, D, k_cache.shape[0], block_tables.shape[1],
        float(scale), block_size, out.data_ptr(), _stream(stream)))
    return out


def paged_attention_static_workspace_bytes() -> int:
    return int(load().pkv_paged_attention_static_workspace_bytes())


def paged_attention_decode_static_workspace(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                            block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                            block_size: int, out: Optional[torch.Tensor] = None,
                                            stream=None) -> torch.Tensor:
    """paged_attention_decode for callers that cannot allocate device memory: the library's
    fixed scratch array replaces the workspace (see include/pkv.h for its limit and sharing)."""
    _need(q, "q", torch.float16, 3)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    S, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.float16, 3)
    _check(load().pkv_paged_attention_decode_static_workspace(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
        S, H, D, k_cache.shape[0], block_tables.shape[1], float(scale), block_size, out.data_ptr(),
        _stream(stream)))
    return out


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, stream=None) -> None:
    """Store key[t], value[t] at slot_mapping[t] (negative = skip) in the paged pools.
    key, value and slot_mapping may be page-locked host tensors (read across the host link)."""
    _need(key, "key", torch.float16, 3, host_ok=True)
    _need(value, "value", torch.float16, 3, host_ok=True)
    _need(k_cache, "k_cache", torch.float16, 4)
    _need(v_cache, "v_cache", torch.float16, 4)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, host_ok=True)
    T, H, D = key.shape
    N, H2, B, D2 = k_cache.shape
    if value.shape != key.shape or (H2, D2) != (H, D) or v_cache.shape != k_cache.shape or slot_mapping.shape[0] != T:
        raise PkvError(PKV_ERR_INVALID_ARG, "reshape_and_cache: inconsistent shapes")
    _check(load().pkv_reshape_and_cache(key.data_ptr(), value.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                        slot_mapping.data_ptr(), T, H, D, B, N, _stream(stream)))


def reshape_and_cache_layers(keys: Sequence[torch.Tensor], values: Sequence[torch.Tensor],
                             k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor],
                             slot_mapping: torch.Tensor, stream=None) -> None:
    """reshape_and_cache for every layer in one launch (one slot mapping for all layers)."""
    L = len(keys)
    if not (len(values) == len(k_caches) == len(v_caches) == L) or L == 0:
        raise PkvError(PKV_ERR_INVALID_ARG, "reshape_and_cache_layers: need as many keys, values and pools")
    for t in list(keys) + list(values):
        _need(t, "key/value", torch.float16, 3)
        if t.shape != keys[0].shape:
            raise PkvError(PKV_ERR_INVALID_ARG, "reshape_and_cache_layers: keys/values differ in shape")
    for t in list(k_caches) + list(v_caches):
        _need(t, "cache", torch.float16, 4)
        if t.shape != k_caches[0].shape:
            raise PkvError(PKV_ERR_INVALID_ARG, "reshape_and_cache_layers: pools differ in shape")
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    T, H, D = keys[0].shape
    N, H2, B, D2 = k_caches[0].shape
    if (H2, D2) != (H, D) or slot_mapping.shape[0] != T:
        raise PkvError(PKV_ERR_INVALID_ARG, "reshape_and_cache_layers: inconsistent shapes")
    arr = lambda ts: ctypes.cast((ctypes.c_void_p * L)(*[t.data_ptr() for t in ts]), ctypes.c_void_p)
    _check(load().pkv_reshape_and_cache_layers(arr(keys), arr(values), arr(k_caches), arr(v_caches), L,
                                               slot_mapping.data_ptr(), T, H, D, B, N, _stream(stream)))


def copy_blocks(k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor], block_mapping: torch.Tensor,
                stream=None) -> None:
    """For each (src, dst) row of block_mapping and each layer: block dst := block src (K and V).
    block_mapping may be a page-locked host tensor (read across the host link)."""
    if len(k_caches) != len(v_caches) or len(k_caches) == 0:
        raise PkvError(PKV_ERR_INVALID_ARG, "copy_blocks: need as many K as V pools, at least one")
    for t in list(k_caches) + list(v_caches):
        _need(t, "cache", torch.float16, 4)
        if t.shape != k_caches[0].shape:
            raise PkvError(PKV_ERR_INVALID_ARG, "copy_blocks: pools differ in shape")
    _need(block_mapping, "block_mapping", torch.int64, 2, host_ok=True)
    if block_mapping.shape[1] != 2:
        raise PkvError(PKV_ERR_INVALID_ARG, "copy_blocks: block_mapping must be [P, 2]")
    N, H, B, D = k_caches[0].shape
    L = len(k_caches)
    kp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_caches])
    vp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_caches])
    _check(load().pkv_copy_blocks(ctypes.cast(kp, ctypes.c_void_p), ctypes.cast(vp, ctypes.c_void_p), L,
                                  block_mapping.data_ptr(), block_mapping.shape[0], H, D, B, N, _stream(stream)))


def swap_blocks(src_k: Sequence[torch.Tensor], src_v: Sequence[torch.Tensor], dst_k: Sequence[torch.Tensor],
                dst_v: Sequence[torch.Tensor], block_mapping: torch.Tensor, stream=None) -> None:
    """Whole blocks src -> dst between two pools per layer; a pool may be a CUDA tensor or a
    pinned CPU tensor (swap-out: GPU -> pinned host, swap-in: the reverse)."""
    L = len(src_k)
    if not (len(src_v) == len(dst_k) == len(dst_v) == L) or L == 0:
        raise PkvError(PKV_ERR_INVALID_ARG, "swap_blocks: need the same number (>= 1) of pools on each side")
    for t in list(src_k) + list(src_v) + list(dst_k) + list(dst_v):
        _need(t, "pool", torch.float16, 4, cuda=False)
        if not (t.is_cuda or t.is_pinned()):
            raise PkvError(PKV_ERR_INVALID_ARG, "swap_blocks: a CPU pool must be pinned")
    for side in (src_k, src_v):
        if any(t.shape != side[0].shape for t in side):
            raise PkvError(PKV_ERR_INVALID_ARG, "swap_blocks: source pools differ in shape")
    for side in (dst_k, dst_v):
        if any(t.shape != side[0].shape for t in side):
            raise PkvError(PKV_ERR_INVALID_ARG, "swap_blocks: destination pools differ in shape")
    Ns, H, B, D = src_k[0].shape
    Nd = dst_k[0].shape[0]
    if tuple(dst_k[0].shape[1:]) != (H, B, D):
        raise PkvError(PKV_ERR_INVALID_ARG, "swap_blocks: pools differ in [H, B, D]")
    _need(block_mapping, "block_mapping", torch.int64, 2, cuda=False)
    if block_mapping.shape[1] != 2 or not (block_mapping.is_cuda or block_mapping.is_pinned()):
        raise PkvError(PKV_ERR_INVALID_ARG, "swap_blocks: block_mapping must be [P, 2], on the GPU or pinned")
    arr = lambda ts: ctypes.cast((ctypes.c_void_p * L)(*[t.data_ptr() for t in ts]), ctypes.c_void_p)
    _check(load().pkv_swap_blocks(arr(src_k), arr(src_v), arr(dst_k), arr(dst_v), L, block_mapping.data_ptr(),
                                  block_mapping.shape[0], H, D, B, Ns, Nd, _stream(stream)))


# ---- host block manager -----------------------------------------------------------------------

def _np_ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class BlockManager:
    """Host block manager (pkv_bm_*): block tables, FIFO free list, reference counts, copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        lib = load()
        self._lib = lib
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
            if order.shape != (num_blocks,):
                raise PkvError(PKV_ERR_INVALID_ARG, "free_order must have num_blocks entries")
        h = lib.pkv_bm_create(num_blocks, block_size, None if order is None else _np_ptr(order))
        if not h:
            raise PkvError(PKV_ERR_INVALID_ARG, lib.pkv_last_error().decode())
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def add_seq(self, seq_id: int, prompt_len: int) -> np.ndarray:
        slots = np.empty(max(prompt_len, 1), dtype=np.int64)
        _check(self._lib.pkv_bm_add_seq(self._h, seq_id, prompt_len, _np_ptr(slots)))
        return slots[:prompt_len]

    def fork(self, parent: int, child: int) -> None:
        _check(self._lib.pkv_bm_fork(self._h, parent, child))

    def append_slot(self, seq_id: int) -> Tuple[int, int, int]:
        slot = _I64(0)
        src = ctypes.c_int32(0)
        dst = ctypes.c_int32(0)
        _check(self._lib.pkv_bm_append_slot(self._h, seq_id, ctypes.byref(slot), ctypes.byref(src),
                                            ctypes.byref(dst)))
        return slot.value, src.value, dst.value

    def append_slots(self, seq_ids: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.shape[0]
        slots = np.empty(max(n, 1), dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        nc = _c.c_int(0)
        _check(self._lib.pkv_bm_append_slots(self._h, _np_ptr(ids), n, _np_ptr(slots), _np_ptr(pairs),
                                             ctypes.byref(nc)))
        return slots[:n], pairs[:nc.value]

    def free(self, seq_id: int) -> None:
        _check(self._lib.pkv_bm_free(self._h, seq_id))

    def register_prefix(self, prefix_id: int, length: int) -> np.ndarray:
        slots = np.empty(max(length, 1), dtype=np.int64)
        _check(self._lib.pkv_bm_register_prefix(self._h, prefix_id, length, _np_ptr(slots)))
        return slots[:length]

    def add_seq_with_prefix(self, seq_id: int, prefix_id: int, suffix_len: int = 0) -> Tuple[np.ndarray, np.ndarray]:
        """Map the prefix's blocks, then place ``suffix_len`` own tokens (all or nothing).
        Returns the suffix slots [suffix_len] and the copies [0 or 1, 2] (src, dst) to run first."""
        slots = np.empty(max(suffix_len, 1), dtype=np.int64)
        pair = np.empty(2, dtype=np.int64)
        nc = _c.c_int(0)
        _check(self._lib.pkv_bm_add_seq_with_prefix(self._h, seq_id, prefix_id, suffix_len, _np_ptr(slots),
                                                    _np_ptr(pair), ctypes.byref(nc)))
        return slots[:suffix_len], pair.reshape(1, 2)[:nc.value]

    def extend(self, seq_id: int, n: int) -> Tuple[np.ndarray, np.ndarray]:
        """Slots of the sequence's next n tokens in one all-or-nothing call, and the copy
        [0 or 1, 2] (src, dst) that must run before they are written."""
        slots = np.empty(max(n, 1), dtype=np.int64)
        pair = np.empty(2, dtype=np.int64)
        nc = _c.c_int(0)
        _check(self._lib.pkv_bm_extend(self._h, seq_id, n, _np_ptr(slots), _np_ptr(pair), ctypes.byref(nc)))
        return slots[:n], pair.reshape(1, 2)[:nc.value]

    def drop_prefix(self, prefix_id: int) -> None:
        _check(self._lib.pkv_bm_drop_prefix(self._h, prefix_id))

    def block_table(self, seq_id: int, cap: int = 1 << 16) -> Tuple[list, int]:
        out = np.empty(cap, dtype=np.int32)
        nb = _c.c_int(0)
        ctx = _c.c_int(0)
        _check(self._lib.pkv_bm_block_table(self._h, seq_id, _np_ptr(out), cap, ctypes.byref(nb), ctypes.byref(ctx)))
        return [int(x) for x in out[:nb.value]], ctx.value

    def block_tables(self, seq_ids: Sequence[int], max_blocks: int) -> Tuple[np.ndarray, np.ndarray]:
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.shape[0]
        tables = np.empty((n, max_blocks), dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        _check(self._lib.pkv_bm_block_tables(self._h, _np_ptr(ids), n, _np_ptr(tables), max_blocks, _np_ptr(lens)))
        return tables, lens

    def beam_step(self, parents: Sequence[int], children: Sequence[int],
                  retire: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
        """Fork children from parents, free the retired beam, append one token per child."""
        par = np.ascontiguousarray(np.asarray(parents, dtype=np.int64))
        chi = np.ascontiguousarray(np.asarray(children, dtype=np.int64))
        ret = np.ascontiguousarray(np.asarray(retire, dtype=np.int64))
        k = chi.shape[0]
        if par.shape[0] != k:
            raise PkvError(PKV_ERR_INVALID_ARG, "parents and children differ in length")
        slots = np.empty(max(k, 1), dtype=np.int64)
        pairs = np.empty((max(k, 1), 2), dtype=np.int64)
        nc = _c.c_int(0)
        _check(self._lib.pkv_bm_beam_step(self._h, _np_ptr(par), _np_ptr(chi), k, _np_ptr(ret), ret.shape[0],
                                          _np_ptr(slots), _np_ptr(pairs), ctypes.byref(nc)))
        return slots[:k], pairs[:nc.value]

    def swap(self, dst: "BlockManager", seq_ids: Sequence[int]) -> np.ndarray:
        """Move the group ``seq_ids`` to ``dst`` (pkv_bm_swap).  Returns the [P, 2] int64 block moves
        (this manager's block, dst's block): the block_mapping for swap_blocks."""
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        cap = sum(len(self.block_table(int(s))[0]) for s in ids)       # an upper bound on distinct blocks
        pairs = np.empty((max(cap, 1), 2), dtype=np.int64)
        n = _c.c_int(0)
        _check(self._lib.pkv_bm_swap(self._h, dst._h, _np_ptr(ids), ids.shape[0], _np_ptr(pairs), cap,
                                     ctypes.byref(n)))
        return pairs[:n.value]

    COUNTERS = ("cow_copies", "prefix_seqs", "prefix_blocks", "groups_out", "blocks_out", "groups_in", "blocks_in")

    def ref_histogram(self, cap: int = 8) -> np.ndarray:
        """[cap] int64: blocks with reference count r (r < cap - 1), the last entry counting the rest."""
        hist = np.empty(cap, dtype=np.int64)
        _check(self._lib.pkv_bm_ref_histogram(self._h, _np_ptr(hist), cap))
        return hist

    def counters(self) -> dict:
        """Copy-on-write copies, prefix hits (sequences and block references) and swap traffic."""
        out = np.zeros(len(self.COUNTERS), dtype=np.int64)
        n = self._lib.pkv_bm_counters(self._h, _np_ptr(out), out.shape[0])
        if n < 0:
            _check(n)
        return {k: int(v) for k, v in zip(self.COUNTERS, out)}

    def ref_count(self, block: int) -> int:
        r = self._lib.pkv_bm_ref_count(self._h, block)
        if r < 0:
            _check(r)
        return r

    def stats(self) -> Tuple[int, int, int]:
        fb = _c.c_int(0)
        tw = _I64(0)
        cc = _I64(0)
        _check(self._lib.pkv_bm_stats(self._h, ctypes.byref(fb), ctypes.byref(tw), ctypes.byref(cc)))
        return fb.value, tw.value, cc.value
