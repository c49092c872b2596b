"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every declared entry point; config validation and sizes."""
import ctypes
import os
import re

import fp4_block_scaled_gb300 as moe
import synth
from conftest import ROOT


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_ffn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = moe.lib()
    names = declared_functions()
    assert "moe_ffn_forward" in names and "moe_stack_forward" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(moe.EXPORTS)
    assert os.path.exists(moe.library_path())


def test_packed_sizes_equal_published_sizes():
    cfg = moe.config(384, 4096, 2880, 6, 1)
    nc, ns = synth.expert_sizes(4096, 2880)
    assert nc == 17694720 and ns == 1105920
    # every published code and scale byte once; the scale atom of the 64-wide
    # half unit of each 128-row down tile is padded from 256 to 512 bytes
    assert moe.moe_ffn_packed_expert_bytes(cfg) == nc + ns + (4096 // 128) * 256 == 18808832
    cfg = moe.config(8, 256, 128, 2, 1)
    assert moe.moe_ffn_packed_expert_bytes(cfg) == 3 * 256 * 128 // 2 + 3 * 256 * 128 // 32


def test_invalid_configs_are_rejected_on_the_host():
    bad = [
        moe.config(0, 4096, 2880, 6, 1),
        moe.config(8, 4096, 2880, 0, 1),
        moe.config(8, 4096, 2880, 9, 1),        # topk > E
        moe.config(8, 4000, 2880, 6, 1),        # H % 128
        moe.config(8, 4160, 2880, 6, 1),        # H % 128 (a multiple of 64)
        moe.config(8, 4096, 2850, 6, 1),        # I % 64
        moe.config(8, 4096, 2880, 6, -1),
        moe.config(8, 4096, 2880, 6, 1, act_mode=7),
        moe.config(8, 4096, 2880, 6, 1, out_dtype=3),
    ]
    for c in bad:
        assert moe.moe_ffn_packed_expert_bytes(c) == 0
    h = ctypes.c_void_p()
    assert moe.lib().moe_ffn_create(ctypes.byref(h), ctypes.byref(bad[0]), 0) == moe.MOE_ERR_INVALID_ARG
    assert moe.lib().moe_ffn_create(ctypes.byref(h), ctypes.byref(bad[3]), 0) == moe.MOE_ERR_UNSUPPORTED
    assert h.value is None


def test_null_handle_and_strerror():
    L = moe.lib()
    assert L.moe_ffn_forward(None, None, None, None, None, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_ffn_status(None, None) == moe.MOE_ERR_INVALID_ARG
    L.moe_ffn_destroy(None)
    for code in range(-6, 1):
        assert moe.strerror(code) and moe.strerror(code) != "unknown error code"
    assert moe.strerror(-99) == "unknown error code"


def test_binding_constants_match_the_header():
    import re

    text = open(os.path.join(ROOT, "include", "moe_ffn.h"), encoding="utf-8").read()
    m = re.search(r"#define MOE_DEFAULT_GEMM_MIN_TOKENS (\d+)", text)
    assert m and int(m.group(1)) == moe.DEFAULT_GEMM_MIN_TOKENS
