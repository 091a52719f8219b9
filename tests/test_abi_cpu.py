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


def test_noalloc_rejects_bad_arguments_before_any_device_call(lib_path):
    """pck_attend_records_noalloc checks its arguments before its first CUDA call. Every case
    below breaks exactly one rule and must be refused with that rule's code. The pointer values
    are never dereferenced: a case that slipped through would stop at the device query, which
    has no device here (PCK_ECUDA) and fails the test. Skipped where a GPU is present, where the
    GPU tests cover this entry point with real buffers."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("covered with real buffers by the GPU tests")
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library(lib_path)
    P = ctypes.c_void_p(1 << 20)          # 16-byte aligned stand-ins, never read
    P2 = ctypes.c_void_p((1 << 20) + 2)   # not 4-byte aligned
    P4 = ctypes.c_void_p((1 << 20) + 4)   # 4- but not 16-byte aligned
    good = dict(H_kv=2, N=64, D=64, K=P, V=P, H_q=4, qdt=binding.DT_F32, Q=P, S=0, Ks=None, Vs=None, O=P, L=P)

    def call(**kw):
        a = dict(good, **kw)
        return lib.pck_attend_records_noalloc(a["H_kv"], a["N"], a["D"], a["K"], a["V"], a["H_q"], a["qdt"],
                                              a["Q"], None, a["S"], a["Ks"], a["Vs"], a["O"], a["L"], None)

    cases = [
        (dict(K=None), binding.EINVAL), (dict(Q=None), binding.EINVAL), (dict(O=None), binding.EINVAL),
        (dict(O=P4), binding.EINVAL), (dict(Q=P4), binding.EINVAL),
        (dict(H_kv=0), binding.EINVAL), (dict(H_q=65), binding.EINVAL), (dict(N=0), binding.EINVAL),
        (dict(S=-1), binding.EINVAL), (dict(D=96), binding.EUNSUPPORTED), (dict(qdt=7), binding.EINVAL),
        (dict(S=4), binding.EINVAL), (dict(S=4, Ks=P), binding.EINVAL), (dict(K=P2), binding.EINVAL),
    ]
    for kw, want in cases:
        assert call(**kw) == want, kw
    assert call() == binding.ECUDA        # well-formed: the next step is the device query


def test_quantizer_rejects_bad_arguments_before_any_device_call(lib_path):
    """pck_quantize_mlx4g32 refuses malformed calls, and returns at once for zero rows, before it
    touches the device; no case below launches anything, so the stand-in pointers are never used."""
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library(lib_path)
    P, P8, P2 = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 8), ctypes.c_void_p((1 << 20) + 2)
    q = lambda X=P, dt=binding.DT_F16, rows=4, kv=64, out=P: lib.pck_quantize_mlx4g32(X, dt, rows, kv, out, None)
    for kw in (dict(X=None), dict(out=None), dict(rows=-1), dict(kv=16), dict(kv=48), dict(dt=5), dict(X=P8),
               dict(out=P2)):
        assert q(**kw) == binding.EINVAL, kw
    assert q(rows=0) == binding.OK
