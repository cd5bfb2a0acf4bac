"""The C-ABI library builds for sm_103a, loads without a GPU and exports every symbol whead.h declares."""
import os
import re

from speculative_decoding_serial_gb300 import build, whead

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "whead.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(whead_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(whead.EXPORTS)


def test_library_exports_every_declared_symbol():
    build.build()
    L = whead.load()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_strerror_needs_no_device():
    build.build()
    assert whead.strerror(whead.ERR_TIMEOUT).startswith("a device-side wait")
    assert whead.strerror(12345) == "unknown error"
