"""CPU checks of the C-ABI library: it builds, loads, and exports every symbol include/pck.h declares.
No compute call is made here (there is no GPU in this environment)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pck.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pck_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib_path():
    from prefix_cached_kv_gb300 import build
    return build.build()


def test_header_declarations_match_binding():
    from prefix_cached_kv_gb300 import binding
    assert _declared() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pck_[a-z0-9_]+)$", out, flags=re.M))
    assert set(_declared()) <= exported


def test_binding_loads_and_sets_signatures(lib_path):
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library(lib_path)
    assert lib.pck_last_error(None) == b"no context"
    # host-side argument checks that return before touching the device
    assert lib.pck_quantize_mlx4g32(None, 0, 1, 64, None, None) == binding.EINVAL
    assert lib.pck_store(None, b"s", 0, 1, 1, 64, 0, None, None, 0, None) == binding.EINVAL


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-fsyntax-only", "-Wall", "-Werror", "-x", "c", HEADER], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
