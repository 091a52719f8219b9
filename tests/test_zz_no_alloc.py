"""pck_attend_records_noalloc: the entry point for callers that cannot allocate device memory
at call time. Called through the C ABI (ctypes, raw device pointers) and compared with the
context-based path (pck_store_records + pck_query_fused) within the parity tolerances, on two
calls in a row (its scratch is shared device memory that keeps the previous call's contents).
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import pck_oracle as orc
from prefix_cached_kv_gb300 import synth
from tests.gpu_util import LSE_ATOL, O_ATOL, ctx_factory, dev, host, need_gpu

pytestmark = pytest.mark.gpu


def _vp(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


@pytest.mark.parametrize("H_q,H_kv,N,D,S", [(32, 8, 8192, 64, 16), (16, 4, 1000, 128, 0)])
def test_noalloc_matches_context_path_twice(H_q, H_kv, N, D, S):
    need_gpu()
    from prefix_cached_kv_gb300 import binding
    lib = binding.load_library()
    K, V = synth.gen_kv(31 + D, H_kv, N, D)
    tok = lambda X: X.transpose(1, 0, 2).reshape(N, H_kv * D)
    Krec, Vrec = dev(orc.quantize_records(tok(K))), dev(orc.quantize_records(tok(V)))
    ctx = ctx_factory()
    ctx.store_records("na", 0, H_kv, N, D, Krec, Vrec)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):   # second call reuses the scratch left by the first
        Q = dev(synth.gen_q(40 + call, H_q, 1, D))
        Ks = Vs = None
        if S:
            Ks, Vs = [dev(a) for a in synth.gen_suffix(40 + call, H_kv, S, D)]
        O = torch.full((H_q, D), float("nan"), device="cuda")
        L = torch.full((H_q,), float("nan"), device="cuda")
        rc = lib.pck_attend_records_noalloc(H_kv, N, D, _vp(Krec), _vp(Vrec), H_q, binding.DT_F32, _vp(Q), None, S,
                                            _vp(Ks), _vp(Vs), _vp(O), _vp(L), stream)
        assert rc == binding.OK
        if S:
            O_ref, L_ref = ctx.query_fused("na", 0, Q, Ks, Vs)
        else:
            O_ref, L_ref = ctx.query("na", 0, Q)
        ctx.sync()
        o, l = host(O), host(L)
        assert np.isfinite(o).all() and np.isfinite(l).all()
        assert np.abs(o - host(O_ref)[:, 0]).max() <= O_ATOL
        assert np.abs(l - host(L_ref)[:, 0]).max() <= LSE_ATOL
    ctx.close()


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
