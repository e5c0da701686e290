"""The C-ABI library loads, exports every symbol include/moe.h declares, and
rejects bad arguments on the host before touching a GPU (CPU only: none of these
calls reaches the CUDA runtime)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import expert_routing_dispatch_gb300 as m

    m.build()
    return m


def header_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_and_binding_agree(moe):
    assert header_symbols() == sorted(moe.EXPORTED)


def test_library_exports_every_declared_symbol(moe):
    L = ctypes.CDLL(moe.LIB_PATH)
    for name in header_symbols():
        assert hasattr(L, name), name


def test_status_strings(moe):
    for code in range(7):
        assert moe.moe_status_string(code) != "unknown status"
    assert moe.moe_status_string(99) == "unknown status"


def test_workspace_sizes(moe):
    d = moe.Dims(6000, 4096, 1536, 128, 8, 0, 32)
    P = 6000 * 8
    assert moe.moe_expert_ffn_workspace_size(d) >= P * 1536 * 2 * 2  # h as bf16 hi and lo terms
    assert moe.moe_dispatch_workspace_size(d) >= -(-6000 // 32) * 32 * 4  # per-chunk histograms
    total = moe.moe_workspace_size(d)
    assert total >= P * 4096 * 2 + P * 4096 * 4 + P * 1536 * 4 + 4 * P * 4
    assert total % 256 == 0


@pytest.mark.parametrize("bad", [
    dict(T=0), dict(k=0), dict(k=33, E=64), dict(k=9, E=8), dict(e0=-1), dict(e1=0), dict(e0=5, e1=5),
    dict(e1=200), dict(H=100), dict(I=96), dict(H=0), dict(E=2000), dict(T=600000000),
])
def test_invalid_dims_rejected_without_gpu(moe, bad):
    base = dict(T=64, H=256, I=128, E=16, k=4, e0=0, e1=16)
    base.update(bad)
    d = moe.Dims.of(base)
    assert moe.moe_workspace_size(d) == 0
    fake = 1 << 20  # a 16-byte aligned address that is never dereferenced
    st = moe.lib().moe_route(ctypes.byref(d), fake, fake, fake, None, None)
    assert st == 1  # MOE_ERR_INVALID_ARG


def test_misaligned_or_null_pointers_rejected(moe):
    d = moe.Dims(64, 256, 128, 16, 4, 0, 16)
    L = moe.lib()
    ok = 1 << 20
    assert L.moe_route(ctypes.byref(d), ok + 4, ok, ok, None, None) == 1
    assert L.moe_route(ctypes.byref(d), None, ok, ok, None, None) == 1
    assert L.moe_combine(ctypes.byref(d), ok, ok, ok + 8, ok, None) == 1
    assert L.moe_layer(ctypes.byref(d), ok, ok, ok, ok, ok, ok + 2, None, None, ok, 1 << 40, None, None) == 1


def test_missing_workspace_rejected(moe):
    d = moe.Dims(64, 256, 128, 16, 4, 0, 16)
    L = moe.lib()
    ok = 1 << 20
    need = moe.moe_workspace_size(d)
    assert L.moe_layer(ctypes.byref(d), ok, ok, ok, ok, ok, ok, None, None, None, need, None, None) == 3
    assert L.moe_layer(ctypes.byref(d), ok, ok, ok, ok, ok, ok, None, None, ok, need - 1, None, None) == 3
    assert L.moe_layer(ctypes.byref(d), ok, ok, ok, ok, ok, ok, None, None, ok + 16, need, None, None) == 3
    nd = moe.moe_dispatch_workspace_size(d)
    assert L.moe_dispatch(ctypes.byref(d), ok, ok, ok, ok, ok, ok, ok, None, nd, None) == 3
    nf = moe.moe_expert_ffn_workspace_size(d)
    assert L.moe_expert_ffn(ctypes.byref(d), ok, ok, ok, ok, ok, ok, ok, nf - 256, None, None) == 3


def test_mxfp8_entries_reject_bad_arguments_without_gpu(moe):
    L = moe.lib()
    ok = 1 << 20
    # H or I not a multiple of 128: unsupported by the MXFP8 entries (fine for the bf16 ones)
    for dims in ((64, 192, 128, 8, 2, 0, 8), (64, 256, 192, 8, 2, 0, 8)):
        d = moe.Dims(*dims)
        assert moe.moe_workspace_size(d) > 0
        assert moe.moe_layer_mxfp8_workspace_size(d) == 0 and moe.moe_expert_ffn_mxfp8_workspace_size(d) == 0
        assert L.moe_layer_mxfp8(ctypes.byref(d), *([ok] * 9), None, None, ok, 1 << 40, None, None) == 2
        assert L.moe_expert_ffn_mxfp8(ctypes.byref(d), *([ok] * 10), ok, 1 << 40, None, None) == 2
    d = moe.Dims(64, 256, 128, 16, 4, 0, 16)
    need = moe.moe_layer_mxfp8_workspace_size(d)
    assert need > moe.moe_expert_ffn_mxfp8_workspace_size(d) > 0
    assert L.moe_layer_mxfp8(ctypes.byref(d), *([ok] * 9), None, None, ok, need - 1, None, None) == 3
    assert L.moe_layer_mxfp8(ctypes.byref(d), ok + 4, *([ok] * 8), None, None, ok, need, None, None) == 1
    # quantiser: K a positive multiple of 32, aligned pointers
    assert L.moe_quantize_mxfp8(ok, 4, 48, ok, ok, None) == 1
    assert L.moe_quantize_mxfp8(ok, -1, 64, ok, ok, None) == 1
    assert L.moe_quantize_mxfp8(ok + 2, 4, 64, ok, ok, None) == 1
    assert L.moe_quantize_mxfp8(ok, 0, 64, ok, ok, None) == 0  # nothing to do, no launch


def test_layer_gather_rejects_split_sizes_without_gpu(moe):
    # dispatch by TMA row gather exists on the fused path only: T*k above the fused limit is unsupported
    L = moe.lib()
    ok = 1 << 20
    d = moe.Dims(moe.FUSED_MAX_PAIRS // 4 + 1, 256, 128, 16, 4, 0, 16)
    assert L.moe_layer_gather(ctypes.byref(d), ok, ok, ok, ok, ok, ok, None, None, ok, 1 << 40, None, None) == 2
    d = moe.Dims(64, 256, 128, 16, 4, 0, 16)
    need = moe.moe_workspace_size(d)
    assert L.moe_layer_gather(ctypes.byref(d), ok, ok, ok, ok, ok, ok + 2, None, None, ok, need, None, None) == 1
    assert L.moe_layer_gather(ctypes.byref(d), ok, ok, ok, ok, ok, ok, None, None, ok, need - 1, None, None) == 3
