"""The C-ABI library loads and exports every entry point include/ftmoe.h declares (no device needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "ftmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"FT_API\s+[\w\s\*]+?\b(ft_\w+)\s*\(", src)))


def test_header_declares_the_layer_step_calls():
    names = declared_symbols()
    for n in ("ft_moe_route", "ft_moe_permute", "ft_moe_expert_ffn_nvfp4_decode", "ft_moe_combine",
              "ft_expert_cache_lookup", "ft_expert_cache_fill", "ft_moe_layer_decode"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib_path = os.path.join(ROOT, "quantized_expert_ffn_06_b300", "libftmoe.so")
    if not os.path.exists(lib_path):
        pytest.skip("library not built")
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing
