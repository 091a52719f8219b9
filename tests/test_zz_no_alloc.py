"""pck_attend_records_noalloc: the entry point for callers that cannot allocate device memory at
call time (a request path that must not touch the allocator, code under another framework's
memory budget, a process without a pck context). Called through the C ABI (ctypes, raw device
pointers) and compared with the oracle, which dequantises the same records itself, within the
parity tolerances, on two calls in a row (its scratch is shared device memory that keeps the
previous call's contents), and once more against the context path. pck_noalloc_status, the way
such a caller learns that a kernel reported an error, is checked to stay quiet on good calls and
to report (and then clear) the Q-range code. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import pck_oracle as orc
from prefix_cached_kv_gb300 import synth
from tests.gpu_util import LSE_ATOL, O_ATOL, assert_close_o_lse, ctx_factory, dev, host, need_gpu

pytestmark = pytest.mark.gpu


def _vp(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _status(lib):
    code = ctypes.c_int(-1)
    rc = lib.pck_noalloc_status(_stream(), ctypes.byref(code))
    return rc, code.value


def _records(seed, H_kv, N, D):
    K, V = synth.gen_kv(seed, H_kv, N, D)
    tok = lambda X: X.transpose(1, 0, 2).reshape(N, H_kv * D)
    return orc.quantize_records(tok(K)), orc.quantize_records(tok(V))


CASES = [
    # H_q, H_kv, N, D, S_suf, q fp16, explicit head_map, LSE wanted
    (32, 8, 8192, 64, 16, False, False, True),     # the GQA decode layer shape
    (16, 4, 1000, 128, 0, False, False, True),
    (64, 4, 1500, 128, 32, True, True, False),     # 16 q heads per kv head: two work groups, two column blocks
    (6, 3, 333, 256, 5, True, True, True),         # q heads of a kv head not adjacent, D = 256
]


@pytest.mark.parametrize("H_q,H_kv,N,D,S,q16,custom_hm,want_lse", CASES)
def test_noalloc_matches_oracle_twice(H_q, H_kv, N, D, S, q16, custom_hm, want_lse):
    need_gpu()
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library()
    Krec_h, Vrec_h = _records(31 + D, H_kv, N, D)
    Krec, Vrec = dev(Krec_h), dev(Vrec_h)
    Ko, Vo = orc.records_to_heads(Krec_h, H_kv, D), orc.records_to_heads(Vrec_h, H_kv, D)
    if custom_hm:
        hm = np.array([(5 * h + 1) % H_kv for h in range(H_q)], dtype=np.int32)
    else:
        hm = synth.default_head_map(H_q, H_kv)
    hm_c = (ctypes.c_int32 * H_q)(*hm.tolist()) if custom_hm else None
    assert _status(lib) == (binding.OK, 0)
    for call in range(2):   # the second call reuses the scratch the first one left behind
        Q = synth.gen_q(40 + call, H_q, 1, D, dtype=np.float16 if q16 else np.float32)
        Ks = Vs = None
        if S:
            Ks, Vs = synth.gen_suffix(40 + call, H_kv, S, D)
        O = torch.full((H_q, D), float("nan"), device="cuda")
        L = torch.full((H_q,), float("nan"), device="cuda") if want_lse else None
        Qd = dev(Q[:, 0])   # kept alive until the kernels have read it
        Ksd, Vsd = (dev(Ks), dev(Vs)) if S else (None, None)
        rc = lib.pck_attend_records_noalloc(H_kv, N, D, _vp(Krec), _vp(Vrec), H_q,
                                            binding.DT_F16 if q16 else binding.DT_F32, _vp(Qd),
                                            hm_c, S, _vp(Ksd), _vp(Vsd), _vp(O), _vp(L), _stream())
        assert rc == binding.OK
        assert _status(lib) == (binding.OK, 0)
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs)
        o = host(O)
        if want_lse:
            assert_close_o_lse(o, host(L), O_ref[:, 0], L_ref[:, 0], f"call {call}")
        else:
            assert np.isfinite(o).all() and np.abs(o - O_ref[:, 0]).max() <= O_ATOL


def test_noalloc_agrees_with_context_path():
    """The same records through pck_store_records + pck_query_fused: both paths plan the same
    split of the work, so the results agree far inside the tolerance."""
    need_gpu()
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library()
    H_q, H_kv, N, D, S = 32, 8, 4096, 64, 16
    Krec_h, Vrec_h = _records(77, H_kv, N, D)
    Krec, Vrec = dev(Krec_h), dev(Vrec_h)
    Q = dev(synth.gen_q(78, H_q, 1, D))
    Ks, Vs = [dev(a) for a in synth.gen_suffix(78, H_kv, S, D)]
    ctx = ctx_factory()
    ctx.store_records("na", 0, H_kv, N, D, Krec, Vrec)
    O = torch.empty((H_q, D), device="cuda")
    L = torch.empty((H_q,), device="cuda")
    rc = lib.pck_attend_records_noalloc(H_kv, N, D, _vp(Krec), _vp(Vrec), H_q, binding.DT_F32, _vp(Q[:, 0]), None,
                                        S, _vp(Ks), _vp(Vs), _vp(O), _vp(L), _stream())
    assert rc == binding.OK
    O_ref, L_ref = ctx.query_fused("na", 0, Q, Ks, Vs)
    ctx.sync()
    assert _status(lib) == (binding.OK, 0)
    assert np.abs(host(O) - host(O_ref)[:, 0]).max() <= O_ATOL / 100
    assert np.abs(host(L) - host(L_ref)[:, 0]).max() <= LSE_ATOL / 100
    ctx.close()


def test_noalloc_status_reports_a_kernel_error_once():
    """An fp32 Q element beyond the M=1 kernels' range (code 7) is the one kernel-side error that
    well-formed inputs can cause without a fault or a hang: the call returns OK, the status call
    reports PCK_ECUDA with the code and clears it, and the next good call is correct and quiet."""
    need_gpu()
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library()
    H_q, H_kv, N, D = 8, 2, 200, 64
    Krec_h, Vrec_h = _records(5, H_kv, N, D)
    Krec, Vrec = dev(Krec_h), dev(Vrec_h)
    Q = synth.gen_q(6, H_q, 1, D)
    bad = Q.copy()
    bad[1, 0, 0] = 1.0e6
    O = torch.empty((H_q, D), device="cuda")
    L = torch.empty((H_q,), device="cuda")
    args = lambda q: (H_kv, N, D, _vp(Krec), _vp(Vrec), H_q, binding.DT_F32, _vp(q), None, 0, None, None,
                      _vp(O), _vp(L), _stream())
    qb = dev(bad[:, 0])
    assert lib.pck_attend_records_noalloc(*args(qb)) == binding.OK
    assert _status(lib) == (binding.ECUDA, 7)
    assert _status(lib) == (binding.OK, 0)
    qg = dev(Q[:, 0])
    assert lib.pck_attend_records_noalloc(*args(qg)) == binding.OK
    assert _status(lib) == (binding.OK, 0)
    O_ref, L_ref = orc.prefix_query(Q, orc.records_to_heads(Krec_h, H_kv, D), orc.records_to_heads(Vrec_h, H_kv, D))
    assert_close_o_lse(host(O), host(L), O_ref[:, 0], L_ref[:, 0], "after the error")


def test_noalloc_rejects_oversize_before_launch():
    need_gpu()
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library()
    big = torch.zeros(16, dtype=torch.uint8, device="cuda")
    # 8 kv heads x 65536 tokens x D=128 needs 8 x 4096 x 2560 B = 80 MiB of tiles > 16 MiB
    rc = lib.pck_attend_records_noalloc(8, 65536, 128, _vp(big), _vp(big), 32, binding.DT_F32, _vp(big), None, 0,
                                        None, None, _vp(big), None, None)
    assert rc == binding.EUNSUPPORTED
    rc = lib.pck_attend_records_noalloc(8, 16, 96, _vp(big), _vp(big), 32, binding.DT_F32, _vp(big), None, 0,
                                        None, None, _vp(big), None, None)
    assert rc == binding.EUNSUPPORTED
