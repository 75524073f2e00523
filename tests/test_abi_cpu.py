"""The C ABI library builds, loads and exports every function include/moe.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes

import pytest

import expert_routed_ffn_moe_gb300 as moe


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.lib()


def test_every_declared_function_is_exported(lib):
    names = moe.header_functions()
    assert {"moe_init", "moe_route", "moe_forward", "moe_status", "moe_strerror", "moe_destroy"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_covers_codes(lib):
    seen = {moe.moe_strerror(c) for c in range(8)}
    assert len(seen) == 8 and moe.moe_strerror(99) == "unknown error"


def _cfg(**kw):
    base = dict(d=512, n_experts=256, inter=128, shared_inter=128, top_k=8, max_tokens=32, x_dtype=moe.MOE_F32,
                has_router_bias=0, has_shared=1)
    base.update(kw)
    return moe.moe_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(d=0), moe.MOE_ERR_ARG),
    (dict(top_k=0), moe.MOE_ERR_ARG),
    (dict(top_k=33, n_experts=256), moe.MOE_ERR_ARG),
    (dict(top_k=9, n_experts=8), moe.MOE_ERR_ARG),
    (dict(max_tokens=0), moe.MOE_ERR_ARG),
    (dict(x_dtype=7), moe.MOE_ERR_ARG),
    (dict(d=500), moe.MOE_ERR_UNSUPPORTED),
    (dict(inter=100, shared_inter=100), moe.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=300), moe.MOE_ERR_UNSUPPORTED),
    (dict(shared_inter=256), moe.MOE_ERR_UNSUPPORTED),
    (dict(bias_select_only=2), moe.MOE_ERR_ARG),
    (dict(shared_gate=2), moe.MOE_ERR_ARG),
    (dict(shared_gate=1, has_shared=0), moe.MOE_ERR_ARG),
    (dict(weight_format=2), moe.MOE_ERR_ARG),
    (dict(weight_format=moe.MOE_W_Q4G64), moe.MOE_ERR_UNSUPPORTED),  # 4-bit needs inter % 256 == 0
])
def test_init_rejects_bad_configs_before_any_device_call(lib, kw, code):
    h = ctypes.c_void_p()
    assert lib.moe_init(ctypes.byref(_cfg(**kw)), ctypes.byref(h)) == code
    assert not h.value


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.moe_init(None, ctypes.byref(h)) == moe.MOE_ERR_ARG
    assert lib.moe_init(ctypes.byref(_cfg()), None) == moe.MOE_ERR_ARG
    assert lib.moe_forward(None, None, 1, None, None, None, None, None, 8, None, None) == moe.MOE_ERR_ARG
    assert lib.moe_route(None, None, 1, None, None, 8, None, None, None, None, None, None) == moe.MOE_ERR_ARG
    assert lib.moe_set_path(None, 0) == moe.MOE_ERR_ARG
    assert lib.moe_status(None) == moe.MOE_ERR_ARG
    lib.moe_destroy(None)


def test_binding_config_matches_header():
    # the ctypes mirror of moe_config lists the header's int fields in order
    import os
    import re

    hdr = open(os.path.join(os.path.dirname(moe.__file__), "..", "include", "moe.h")).read()
    body = re.search(r"typedef struct moe_config \{(.*?)\} moe_config;", hdr, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\bint\s+(\w+)\s*;", body)
    assert [n for n, _ in moe.moe_config._fields_] == fields
    assert all(t is ctypes.c_int for _, t in moe.moe_config._fields_)


def test_q4_row_layout():
    # MOE_W_Q4G64 (moe.h): each row is its code words, then its scales, then its biases
    import numpy as np

    import moe_workloads as mw

    words = np.array([[0x76543210], [0xFEDCBA98]], dtype=np.uint32)  # 2 rows of 8 codes
    scales = np.array([[0x3F80], [0x4000]], dtype=np.uint16)
    biases = np.array([[0xBF80], [0xC000]], dtype=np.uint16)
    b = mw.pack_q4(words, scales, biases)
    assert b.dtype == np.uint8 and b.size == 2 * (4 + 2 + 2)
    row0, row1 = b[:8], b[8:]
    assert row0[:4].tolist() == [0x10, 0x32, 0x54, 0x76]  # little-endian word, nibble 0 lowest
    assert row0[4:].view(np.uint16).tolist() == [0x3F80, 0xBF80]  # then its scale, then its bias
    assert row1[:4].tolist() == [0x98, 0xBA, 0xDC, 0xFE]
    assert row1[4:].view(np.uint16).tolist() == [0x4000, 0xC000]
