"""Shared helpers of the GPU parity tests (the oracle supplies every expected value)."""
import numpy as np
import pytest
import torch

# Tolerances fixed for this path: fp32 outputs within max-abs 2e-3, LSE within 1e-3.
O_ATOL = 2e-3
LSE_ATOL = 1e-3
TIE_EPS = 1e-5       # top-K exemption: oracle K-th vs (K+1)-th score gap below this


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def ctx_factory():
    from prefix_cached_kv_gb300 import binding
    return binding.Context(0)


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def assert_close_o_lse(O, LSE, O_ref, LSE_ref, what=""):
    O = np.asarray(O, dtype=np.float64).reshape(np.shape(O_ref))
    LSE = np.asarray(LSE, dtype=np.float64).reshape(np.shape(LSE_ref))
    assert np.isfinite(O).all() and np.isfinite(LSE).all(), f"{what}: non-finite output"
    eo = np.abs(O - O_ref).max()
    el = np.abs(LSE - LSE_ref).max()
    assert eo <= O_ATOL, f"{what}: max |O - O_ref| = {eo:.3e} > {O_ATOL}"
    assert el <= LSE_ATOL, f"{what}: max |LSE - LSE_ref| = {el:.3e} > {LSE_ATOL}"
    return eo, el
