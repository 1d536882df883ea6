"""The C-ABI library builds for sm_103a, loads, and exports every entry point that
include/kvq8attn.h declares (no kernel is launched: this runs without a GPU)."""
import ctypes
import os
import re

from speculative_verify_attention_gb300 import EXPORTED, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvq8attn.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+([a-z][a-z0-9_]*)\s*\(", text, re.M)))


def test_header_declares_the_binding_names():
    assert sorted(EXPORTED) == _declared()


def test_library_exports_every_declared_symbol():
    path = build.build()
    lib = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(lib, name), name
    lib.kvq8_status_str.restype = ctypes.c_char_p
    assert lib.kvq8_status_str(0) == b"ok"
    assert lib.kvq8_status_str(4) == b"workspace missing or too small"
