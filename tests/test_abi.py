"""The C-ABI library builds, loads without a GPU, exports every declared symbol,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_73_gb300 import _build
from paged_kv_cache_73_gb300 import binding as pkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pkv.h but not exported"


def test_version(lib):
    assert pkv.version() == 100


def _decode(lib, **kw):
    a = dict(q=16, k=16, v=16, tables=16, lens=16, S=2, H=2, D=64, N=8, maxb=4, scale=0.125, B=16, out=16,
             ws=None, ws_bytes=0)
    a.update(kw)
    return lib.pkv_paged_attention_decode(a["q"], a["k"], a["v"], a["tables"], a["lens"], a["S"], a["H"], a["D"],
                                          a["N"], a["maxb"], a["scale"], a["B"], a["out"], a["ws"], a["ws_bytes"],
                                          None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), pkv.PKV_ERR_UNSUPPORTED),
    (dict(B=12), pkv.PKV_ERR_UNSUPPORTED),
    (dict(H=0), pkv.PKV_ERR_INVALID_ARG),
    (dict(S=-1), pkv.PKV_ERR_INVALID_ARG),
    (dict(q=None), pkv.PKV_ERR_INVALID_ARG),
    (dict(q=24), pkv.PKV_ERR_INVALID_ARG),                 # not 16-byte aligned
    (dict(scale=float("inf")), pkv.PKV_ERR_INVALID_ARG),
    (dict(S=0), pkv.PKV_OK),                               # empty batch: nothing to do
])
def test_attention_host_validation(lib, kw, status):
    assert _decode(lib, **kw) == status
    if status != pkv.PKV_OK:
        assert lib.pkv_last_error()


def _decode_append(lib, **kw):
    a = dict(q=16, key=16, value=16, slots=16, k=16, v=16, tables=16, lens=16, S=2, H=2, D=64, N=8, maxb=4,
             scale=0.125, B=16, out=16, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.pkv_paged_attention_decode_append(a["q"], a["key"], a["value"], a["slots"], a["k"], a["v"],
                                                 a["tables"], a["lens"], a["S"], a["H"], a["D"], a["N"], a["maxb"],
                                                 a["scale"], a["B"], a["out"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(key=None), pkv.PKV_ERR_INVALID_ARG),
    (dict(value=None), pkv.PKV_ERR_INVALID_ARG),
    (dict(slots=None), pkv.PKV_ERR_INVALID_ARG),
    (dict(key=40), pkv.PKV_ERR_INVALID_ARG),               # not 16-byte aligned
    (dict(value=8), pkv.PKV_ERR_INVALID_ARG),
    (dict(q=None), pkv.PKV_ERR_INVALID_ARG),               # the decode checks follow
    (dict(D=96), pkv.PKV_ERR_UNSUPPORTED),
    (dict(B=12), pkv.PKV_ERR_UNSUPPORTED),
    (dict(S=0, key=None, value=None, slots=None), pkv.PKV_OK),   # empty batch: nothing to do
])
def test_decode_append_host_validation(lib, kw, status):
    assert _decode_append(lib, **kw) == status
    if status != pkv.PKV_OK:
        assert lib.pkv_last_error()


def _prefill(lib, **kw):
    a = dict(q=16, k=16, v=16, tables=16, lens=16, qs=16, S=2, T=8, maxq=4, H=2, D=64, N=8, maxb=4, scale=0.125,
             B=16, out=16)
    a.update(kw)
    return lib.pkv_paged_attention_prefill(a["q"], a["k"], a["v"], a["tables"], a["lens"], a["qs"], a["S"], a["T"],
                                           a["maxq"], a["H"], a["D"], a["N"], a["maxb"], a["scale"], a["B"],
                                           a["out"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), pkv.PKV_ERR_UNSUPPORTED),
    (dict(B=12), pkv.PKV_ERR_UNSUPPORTED),
    (dict(H=0), pkv.PKV_ERR_INVALID_ARG),
    (dict(T=-1), pkv.PKV_ERR_INVALID_ARG),
    (dict(qs=None), pkv.PKV_ERR_INVALID_ARG),
    (dict(out=None), pkv.PKV_ERR_INVALID_ARG),
    (dict(k=40), pkv.PKV_ERR_INVALID_ARG),                 # not 16-byte aligned
    (dict(scale=0.0), pkv.PKV_ERR_INVALID_ARG),            # the causal max needs scale > 0
    (dict(scale=float("nan")), pkv.PKV_ERR_INVALID_ARG),
    (dict(T=0), pkv.PKV_OK),                               # no new tokens: nothing to do
])
def test_prefill_host_validation(lib, kw, status):
    assert _prefill(lib, **kw) == status
    if status != pkv.PKV_OK:
        assert lib.pkv_last_error()


def _shared_prefix(lib, **kw):
    a = dict(q=16, k=16, v=16, tables=16, lens=16, gs=16, pl=16, G=1, maxg=2, S=2, H=2, D=64, N=8, maxb=4,
             scale=0.125, B=16, out=16, ws=16, ws_bytes=1 << 20)
    a.update(kw)
    return lib.pkv_paged_attention_decode_shared_prefix(a["q"], a["k"], a["v"], a["tables"], a["lens"], a["gs"],
                                                        a["pl"], a["G"], a["maxg"], a["S"], a["H"], a["D"], a["N"],
                                                        a["maxb"], a["scale"], a["B"], a["out"], a["ws"],
                                                        a["ws_bytes"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), pkv.PKV_ERR_UNSUPPORTED),
    (dict(B=2), pkv.PKV_ERR_UNSUPPORTED),
    (dict(G=0), pkv.PKV_ERR_INVALID_ARG),
    (dict(maxg=0), pkv.PKV_ERR_INVALID_ARG),
    (dict(gs=None), pkv.PKV_ERR_INVALID_ARG),
    (dict(ws=None), pkv.PKV_ERR_INVALID_ARG),              # the prefix partials always need a workspace
    (dict(ws=24), pkv.PKV_ERR_INVALID_ARG),
    (dict(scale=-1.0), pkv.PKV_ERR_INVALID_ARG),
    (dict(S=0), pkv.PKV_OK),
])
def test_shared_prefix_host_validation(lib, kw, status):
    assert _shared_prefix(lib, **kw) == status
    if status != pkv.PKV_OK:
        assert lib.pkv_last_error()


def test_multi_layer_reshape_host_validation(lib):
    ptrs = lambda *xs: ctypes.cast((ctypes.c_void_p * len(xs))(*xs), ctypes.c_void_p)
    good = ptrs(16, 32)
    call = lambda k=good, L=2, T=4, D=64: lib.pkv_reshape_and_cache_layers(k, good, good, good, L, 16, T, 2, D, 16, 8,
                                                                          None)
    assert call(D=80) == pkv.PKV_ERR_UNSUPPORTED
    assert call(T=-1) == pkv.PKV_ERR_INVALID_ARG
    assert call(T=0) == pkv.PKV_OK and call(L=0) == pkv.PKV_OK
    assert call(k=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(k=ptrs(16, 40)) == pkv.PKV_ERR_INVALID_ARG              # layer 1's key not 16-byte aligned
    assert call(k=ptrs(16, 0)) == pkv.PKV_ERR_INVALID_ARG               # layer 1's key null


def test_workspace_size(lib):
    # one partition (<= 128 tokens of capacity) needs no workspace
    assert pkv.paged_attention_workspace_size(4, 2, 64, 8, 16) == 0
    # 2048 tokens of capacity: 16 partitions of 128 tokens, (D + 2) floats each
    assert pkv.paged_attention_workspace_size(64, 40, 128, 128, 16) == 64 * 40 * 16 * 130 * 4


@pytest.mark.parametrize("S,H,D,max_blocks,want,kernels", [
    (1, 40, 128, 128, 512, 1),      # ctx 2048: 1024-token partitions would leave SMs idle (80 CTAs);
                                    # 160 CTAs, one wave: the 4 partitions merge in a cluster
    (4, 40, 128, 128, 1024, 1),     # 320 CTAs of 1024 tokens already cover every SM; one wave
    (64, 40, 128, 128, 1024, 2),    # the OPT-13B-shaped batch: 5120 CTAs, a merge kernel follows
    (1, 2, 64, 256, 128, 2),        # too few (sequence, head) pairs to fill the GPU: 32 partitions of
                                    # 128 tokens, more than one cluster merges
    (2, 2, 64, 40, 128, 1),         # 5 partitions, 20 CTAs: merged in clusters
    (8, 8, 64, 8, 128, 1),          # one partition: no merge
])
def test_partition_plan(lib, S, H, D, max_blocks, want, kernels):
    # the longest partition that still gives every SM a CTA (the rule holds for 148-160 SMs, and
    # without a device the library assumes 148); the partitions merge inside thread-block clusters
    # when a sequence has at most 8 and the grid is at most one wave of 3 CTAs per SM
    part, got = pkv.paged_attention_plan(S, H, D, max_blocks, 16)
    assert part == want
    assert got == kernels


def test_cache_ops_host_validation(lib):
    assert lib.pkv_reshape_and_cache(16, 16, 16, 16, 16, 4, 2, 80, 16, 8, None) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.pkv_reshape_and_cache(16, 16, 16, 16, 16, 0, 2, 64, 16, 8, None) == pkv.PKV_OK
    assert lib.pkv_reshape_and_cache(None, 16, 16, 16, 16, 4, 2, 64, 16, 8, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(None, None, 1, 16, 0, 2, 64, 16, 8, None) == pkv.PKV_OK
    assert lib.pkv_copy_blocks(None, None, 1, 16, 3, 2, 64, 16, 8, None) == pkv.PKV_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 1)(24)
    assert lib.pkv_copy_blocks(ctypes.cast(arr, ctypes.c_void_p), ctypes.cast(arr, ctypes.c_void_p), 1, 16, 3, 2,
                               64, 16, 8, None) == pkv.PKV_ERR_INVALID_ARG


def test_binding_refuses_missing_library(monkeypatch, tmp_path):
    monkeypatch.setattr(pkv, "_lib", None)
    monkeypatch.setattr(pkv, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(pkv.PkvError):
        pkv.load()
