"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point include/blk.h declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

import decode_qwen2_block_gb300 as blk
from decode_qwen2_block_gb300 import build as gpu_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gpu_build.build()
    return blk.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(blk_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"blk_create", "blk_prefill", "blk_prefill_kv", "blk_decode"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(blk.EXPORTED) <= names


def test_status_strings(lib):
    codes = [blk.BLK_OK, blk.BLK_ERR_NULL, blk.BLK_ERR_ALIGN, blk.BLK_ERR_SHAPE,
             blk.BLK_ERR_CACHE_OVERFLOW, blk.BLK_ERR_WORKSPACE, blk.BLK_ERR_CUDA,
             blk.BLK_ERR_DEVICE_TIMEOUT, blk.BLK_ERR_POSITION, blk.BLK_ERR_DEVICE]
    texts = [blk.blk_status_str(c) for c in codes]
    assert len(set(texts)) == len(texts)
    assert blk.blk_status_str(12345) == "unknown status"


def test_null_handle_and_arguments_are_rejected(lib):
    w = blk.BlkWeights()
    assert lib.blk_prefill(None, ctypes.byref(w), 16, 16, 1, 16, 16, 16, None, None, 16, 1 << 20, None) == blk.BLK_ERR_NULL
    assert lib.blk_decode(None, ctypes.byref(w), 16, 16, 0, 16, 16, 16, None, None, 16, 1 << 20, None) == blk.BLK_ERR_NULL
    assert lib.blk_workspace_bytes(None, 4) == 0
    assert lib.blk_check(None, None) == blk.BLK_ERR_NULL
    assert lib.blk_set_flags(None, 1) == blk.BLK_ERR_NULL
    lib.blk_destroy(None)
    h = ctypes.c_void_p()
    assert lib.blk_create(None, ctypes.byref(h)) == blk.BLK_ERR_NULL


@pytest.mark.parametrize("bad", [
    dict(head_dim=96), dict(n_heads=5), dict(hidden=200), dict(intermediate=100), dict(intermediate=684),
    dict(max_ctx=0), dict(n_heads=12, n_kv_heads=1), dict(hidden=32768), dict(rope_theta=0.0),
])
def test_bad_shapes_rejected_before_any_device_call(lib, bad):
    base = dict(hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, intermediate=688,
                rms_eps=1e-6, rope_theta=1e4, max_ctx=64, has_qkv_bias=0)
    base.update(bad)
    cfg = blk.BlkConfig(**base)
    h = ctypes.c_void_p()
    assert lib.blk_create(ctypes.byref(cfg), ctypes.byref(h)) == blk.BLK_ERR_SHAPE
    assert h.value is None


def test_missing_library_fails_loudly(tmp_path):
    saved = blk._lib
    blk._lib = None
    try:
        with pytest.raises(RuntimeError, match="no fallback"):
            blk.load(str(tmp_path / "libblk.so"))
    finally:
        blk._lib = saved


def test_batched_entry_points_reject_a_null_handle(lib):
    w = blk.BlkWeights()
    assert lib.blk_decode_batch(None, ctypes.byref(w), 16, 16, 16, 1, 0, 16, 16, 16, None, None,
                                16, 1 << 20, None) == blk.BLK_ERR_NULL
    assert lib.blk_decode_batch_stack(None, ctypes.byref(w), 1, None, None, 16, 16, 16, 1, 0, 16,
                                      16, 1 << 20, None) == blk.BLK_ERR_NULL
    assert lib.blk_decode_batch_workspace_bytes(None, 4) == 0
    assert lib.blk_decode_batch_stack_workspace_bytes(None, 4) == 0
    assert lib.blk_wait_probe(None, 16, 1_000_000, None) == blk.BLK_ERR_NULL
