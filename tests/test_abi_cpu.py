"""The C-ABI library loads and exports every declared entry point; host-side
argument validation runs without a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

from w4a16_compact_expert_gb300 import build_ext, moe_w4a16

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return moe_w4a16.load_library()


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"MOE_W4A16_API\s+[\w\s\*]+?\b(moe_w4a16_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert set(moe_w4a16.EXPORTED) <= set(names)


def _create(lib, **kw):
    cfg = dict(hidden=256, inter=128, num_experts=8, top_k=2, num_slots=8, max_tokens=16, device=0)
    cfg.update(kw)
    c = moe_w4a16.Config(**cfg)
    h = ctypes.c_void_p(123)
    st = lib.moe_w4a16_create(ctypes.byref(c), ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("kw,expect", [
    (dict(hidden=255), moe_w4a16.ERR_INVALID_ARG),
    (dict(inter=0), moe_w4a16.ERR_INVALID_ARG),
    (dict(hidden=96), moe_w4a16.ERR_UNSUPPORTED),
    (dict(inter=1000), moe_w4a16.ERR_UNSUPPORTED),
    (dict(num_experts=0), moe_w4a16.ERR_INVALID_ARG),
    (dict(num_experts=300), moe_w4a16.ERR_INVALID_ARG),
    (dict(top_k=9), moe_w4a16.ERR_INVALID_ARG),
    (dict(top_k=0), moe_w4a16.ERR_INVALID_ARG),
    (dict(num_slots=0), moe_w4a16.ERR_INVALID_ARG),
    (dict(max_tokens=0), moe_w4a16.ERR_INVALID_ARG),
    (dict(device=-1), moe_w4a16.ERR_INVALID_ARG),
])
def test_create_rejects_bad_config(lib, kw, expect):
    st, h = _create(lib, **kw)
    assert st == expect
    assert h.value is None
    assert lib.moe_w4a16_last_error(None)


def test_create_null_args(lib):
    c = moe_w4a16.Config(256, 128, 8, 2, 8, 16, 0)
    assert lib.moe_w4a16_create(None, ctypes.byref(ctypes.c_void_p())) == moe_w4a16.ERR_INVALID_ARG
    assert lib.moe_w4a16_create(ctypes.byref(c), None) == moe_w4a16.ERR_INVALID_ARG


def test_null_handle_calls(lib):
    assert lib.moe_w4a16_destroy(None) == moe_w4a16.OK
    assert lib.moe_w4a16_forward(None, None, 0, None, None, 0, None, None, None, None, None, None) == \
        moe_w4a16.ERR_INVALID_ARG
    assert lib.moe_w4a16_get_status(None, None) == moe_w4a16.ERR_INVALID_ARG
    assert lib.moe_w4a16_slot_bytes(None) == 0
    assert lib.moe_w4a16_offload_enable(None, 4) == moe_w4a16.ERR_INVALID_ARG
    assert lib.moe_w4a16_forward_host(None, None, 0, None, None, 0, None, None) == moe_w4a16.ERR_INVALID_ARG
    assert lib.moe_w4a16_forward_host_async(None, None, 0, None, None, 0, None, None) == moe_w4a16.ERR_INVALID_ARG


def test_no_device_is_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = _create(lib)
    assert st == moe_w4a16.ERR_CUDA and h.value is None


def test_last_path_null_handle(lib):
    n = ctypes.c_int32(7)
    assert lib.moe_w4a16_last_path(None, ctypes.byref(n)) == -1
    assert n.value == 7
