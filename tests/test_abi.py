"""The C-ABI library builds for sm_103a, loads, and exports every symbol include/ftmoe.h
declares; host-side argument checks need no GPU."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ftmoe.h")


@pytest.fixture(scope="module")
def ft():
    from expert_cached_sparse_top_b300 import build
    build.build()
    from expert_cached_sparse_top_b300 import ftmoe
    ftmoe.lib()
    return ftmoe


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FT_API\s+[\w\s\*]+?\b(ft_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("ft_moe_create", "ft_moe_forward", "ft_cache_resize", "ft_cache_stats",
                     "ft_cache_snapshot", "ft_moe_destroy", "ft_status_str"):
        assert required in names


def test_library_exports_every_declared_symbol(ft):
    names = _declared()
    out = subprocess.run(["nm", "-D", "--defined-only", ft.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if " T " in line)
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert set(names) == set(ft.EXPORTS)
    for n in names:
        assert hasattr(ft.lib(), n)


def test_library_is_built_for_sm_103a(ft):
    out = subprocess.run(["cuobjdump", "--list-elf", ft.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_status_strings(ft):
    L = ft.lib()
    assert L.ft_status_str(0) == b"FT_OK"
    assert L.ft_status_str(4) == b"FT_ERR_TIMEOUT"
    assert L.ft_status_str(99) == b"FT_ERR_UNKNOWN"


def test_blob_bytes_agree_with_oracle_and_generator(ft):
    import workloads as W
    from oracle import formats
    for name in ("tiny", "decode_bf16", "decode_mxfp4", "elastic_nvfp4"):
        c = W.config(name)
        cfg = ft.make_config(c.layers, c.experts, c.hidden, c.inter, c.top_k, 16, c.wfmt, 4)
        got = ft.blob_bytes(cfg)
        assert got == formats.blob_bytes(c.fmt, c.hidden, c.inter)
        assert got == W.blob_layout(c.fmt, c.hidden, c.inter)[1]
    assert ft.blob_bytes(ft.make_config(1, 8, 2048, 768, 8, 16, "bf16", 4)) == 9437184
    assert ft.blob_bytes(ft.make_config(1, 8, 4096, 2048, 6, 8, "mxfp4", 4)) == 13369344
    assert ft.blob_bytes(ft.make_config(1, 8, 100, 768, 8, 16, "bf16", 4)) == 0


@pytest.mark.parametrize("field,value", [
    ("layers", 0), ("experts", 0), ("experts", 2000), ("top_k", 0), ("top_k", 9),
    ("max_tokens", 0), ("wfmt", 7), ("hidden", 100), ("inter", 32), ("cache_slots", -1),
    ("flags", 3), ("flags", 0x200), ("flags", 0x101 | 0x400),
])
def test_create_rejects_bad_config_before_touching_the_device(ft, field, value):
    cfg = ft.make_config(1, 8, 256, 128, 2, 16, "bf16", 4)
    setattr(cfg, field, value)
    n = max(cfg.layers * max(cfg.experts, 0), 1)
    ptrs = (ctypes.c_void_p * n)(*([1] * n))
    h = ctypes.c_void_p()
    st = ft.lib().ft_moe_create(ctypes.byref(cfg), ptrs, None, ctypes.byref(h))
    assert st == ft.FT_ERR_INVALID
    assert not h.value
    msg = ft.lib().ft_moe_last_error(None)
    assert msg and b"no such CUDA device" not in msg      # the config check itself refused it


def test_create_rejects_null_blob_pointer(ft):
    cfg = ft.make_config(1, 8, 256, 128, 2, 16, "bf16", 4)
    ptrs = (ctypes.c_void_p * 8)(*([1] * 7 + [None]))
    h = ctypes.c_void_p()
    assert ft.lib().ft_moe_create(ctypes.byref(cfg), ptrs, None, ctypes.byref(h)) == ft.FT_ERR_INVALID


def test_stage_entry_points_validate_arguments(ft):
    L = ft.lib()
    assert L.ft_topk_softmax(None, 4, 8, 9, None, None, None) == ft.FT_ERR_INVALID
    assert L.ft_topk_softmax(None, 4, 2048, 2, None, None, None) == ft.FT_ERR_INVALID
    assert L.ft_topk_softmax(None, 0, 8, 2, None, None, None) == ft.FT_OK      # empty
    assert L.ft_router_logits(None, 4, 100, None, 8, None, None) == ft.FT_ERR_INVALID
    assert L.ft_router_logits(None, 0, 64, None, 8, None, None) == ft.FT_OK
    assert L.ft_moe_forward(None, 0, None, 1, None, None, None, None, None) == ft.FT_ERR_INVALID
    L.ft_moe_destroy(None)
