"""The C ABI library loads and exports every function include/msk.h
declares; argument validation answers without a GPU (no compute calls)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from moe_decode_step_persistent_gb300 import build as B
    import moe_decode_step_persistent_gb300 as M
    B.build()
    return M.load_library()


def declared_functions():
    with open(os.path.join(ROOT, "include", "msk.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msk_[a-z0-9_]+)\s*\(", text)))


def test_header_lists_the_entry_points():
    names = declared_functions()
    for n in ("msk_create", "msk_load_layer", "msk_layer_step", "msk_decode_step", "msk_get_timeline",
              "msk_debug_dequant", "msk_status_string", "msk_destroy"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    import moe_decode_step_persistent_gb300 as M
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(M.SYMBOLS) == names  # the binding wraps exactly the header's entry points


def test_status_strings(lib):
    for s in range(10):
        assert lib.msk_status_string(s)
    assert b"time budget" in lib.msk_status_string(8)


def test_create_validates_before_touching_the_device(lib):
    import moe_decode_step_persistent_gb300 as M
    h = ctypes.c_void_p()
    cfg = M.ModelConfig()
    assert lib.msk_create(ctypes.byref(cfg), ctypes.byref(h)) == 1  # no layers
    glob = (ctypes.c_uint8 * 1)(0)
    cfg = M.ModelConfig(1, 4096, 32, 8, 96, 2048, 256, 8, 1024, 16, 100, 14, glob, 2048, 1e-6, 1e6, 0)
    assert lib.msk_create(ctypes.byref(cfg), ctypes.byref(h)) == 2  # head_dim 96 unsupported
    cfg = M.ModelConfig(1, 4096, 32, 8, 128, 2048, 256, 8, 1024, 17, 100, 14, glob, 2048, 1e-6, 1e6, 0)
    assert lib.msk_create(ctypes.byref(cfg), ctypes.byref(h)) == 2  # 17 verify tokens
    assert not h.value
    assert lib.msk_layer_step(None, 0, None, None, None, None, None, 0, None) == 1
    assert lib.msk_decode_step(None, None, None, None, None, None, None) == 1
    lib.msk_destroy(None)


def test_binding_rejects_mixed_sliding_windows():
    import msk_synth as S
    import moe_decode_step_persistent_gb300 as M
    with pytest.raises(ValueError):
        M.Model(S.scaled(S.WORKLOADS["tiny"], windows=(2048, 8)))


def test_noalloc_validates_before_touching_the_device(lib):
    # argument checks answer before any CUDA call; the addresses are never
    # dereferenced (a valid call would go on to query the device)
    q, kv, out = 0x10000, 0x20000, 0x30000
    call = lib.msk_attention_noalloc
    assert call(None, kv, 16, 32, 8, 128, 20000, 16384, 0, out, None) == 1      # null query
    assert call(q, kv, 16, 32, 8, 96, 20000, 16384, 0, out, None) == 2          # head_dim 96
    assert call(q, kv, 17, 32, 8, 128, 20000, 16384, 0, out, None) == 2         # 17 tokens
    assert call(q, kv, 16, 32, 4, 128, 20000, 16384, 0, out, None) == 2         # 8 q heads x 16 tokens per kv head
    assert call(q, kv, 16, 30, 8, 128, 20000, 16384, 0, out, None) == 2         # q heads not a multiple of kv heads
    assert call(q, kv, 16, 32, 8, 128, 16390, 16384, 0, out, None) == 1         # rows past max_seq
    assert call(q, kv, 16, 32, 8, 128, 20000, 16384, -1, out, None) == 1        # negative window
    assert call(q + 8, kv, 16, 32, 8, 128, 20000, 16384, 0, out, None) == 3     # misaligned query
    assert call(q, kv, 16, 32, 8, 128, 20000, 16384, 0, out + 4, None) == 3     # misaligned output
