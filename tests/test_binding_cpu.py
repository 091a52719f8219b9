"""Argument checks of the Python binding, on the CPU. The library trusts the sizes a call
implies, so the binding checks every tensor it hands over: dtype and size first, then
contiguity and the device. A context whose library fails the test when called shows that a bad
argument never reaches it; well-formed CPU tensors get as far as the device check."""
import pytest
import torch

from prefix_cached_kv_gb300 import binding


class _NoLib:
    def __getattr__(self, name):
        raise AssertionError(f"{name} was called with arguments the binding should have rejected")


def _ctx():
    c = binding.Context.__new__(binding.Context)   # no device: never created in the library
    c.lib, c.h = _NoLib(), None
    return c


def _raises(fn, text):
    with pytest.raises(ValueError) as e:
        fn()
    assert text in str(e.value), str(e.value)


H_q, H_kv, M, D, S = 4, 2, 3, 64, 5
f32 = dict(dtype=torch.float32)
f16 = dict(dtype=torch.float16)


def test_query_outputs_and_device():
    c = _ctx()
    Q = torch.zeros((H_q, M, D), **f16)
    _raises(lambda: c.query("s", 0, Q, O=torch.zeros((H_q, M, D), dtype=torch.float64)), "O: dtype")
    _raises(lambda: c.query("s", 0, Q, O=torch.zeros((H_q, M, D - 1), **f32)), "O: ")
    _raises(lambda: c.query("s", 0, Q, LSE=torch.zeros((H_q, M - 1), **f32)), "LSE: ")
    _raises(lambda: c.query("s", 0, Q, O=torch.zeros((D, M, H_q), **f32).transpose(0, 2)), "O: must be contiguous")
    _raises(lambda: c.query("s", 0, Q[0]), "Q must be [H_q, M, D]")
    _raises(lambda: c.query("s", 0, Q.to(torch.int32)), "Q: dtype")
    _raises(lambda: c.query("s", 0, Q), "must be on the CUDA device")


def test_query_fused_suffix():
    c = _ctx()
    Q = torch.zeros((H_q, M, D), **f32)
    Ks = torch.zeros((H_kv, S, D), **f16)
    _raises(lambda: c.query_fused("s", 0, Q, Ks.float(), Ks.float()), "K_suf: dtype")
    _raises(lambda: c.query_fused("s", 0, Q, Ks, Ks[:, :-1]), "one shape")
    _raises(lambda: c.query_fused("s", 0, Q, Ks[..., :32], Ks[..., :32]), "does not match")
    _raises(lambda: c.query_fused("s", 0, Q, None, None), "needs K_suf and V_suf")
    _raises(lambda: c.query_fused("s", 0, Q, Ks, Ks.clone()), "must be on the CUDA device")


def test_query_sparse_outputs():
    c = _ctx()
    Q = torch.zeros((H_q, D), **f32)
    _raises(lambda: c.query_sparse_auto("s", 0, Q, 64, 4, H_kv, idx=torch.zeros((H_q, 4), dtype=torch.int64)),
            "idx: dtype")
    _raises(lambda: c.query_sparse_auto("s", 0, torch.zeros((H_q, 2, D), **f32), 64, 4, H_kv), "Q: ")
    Ks = torch.zeros((H_kv + 1, S, D), **f16)
    _raises(lambda: c.query_sparse_auto("s", 0, Q, 64, 4, H_kv, K_suf=Ks, V_suf=Ks), "does not match")
    _raises(lambda: c.query_sparse_auto("s", 0, Q, 64, 4, H_kv), "must be on the CUDA device")


def test_store_shapes_and_records():
    c = _ctx()
    K = torch.zeros((H_kv, 16, D), **f16)
    _raises(lambda: c.store("s", 0, K, K.float()), "one shape and dtype")
    _raises(lambda: c.store("s", 0, K, K[:, :8]), "one shape and dtype")
    _raises(lambda: c.store("s", 0, K, K.clone()), "must be on the CUDA device")
    rec = 16 * (H_kv * D // 2 + H_kv * D // 8)
    small = torch.zeros(rec - 1, dtype=torch.uint8)
    _raises(lambda: c.store_records("s", 0, H_kv, 16, D, small, small), "K_rec: ")
    ok = torch.zeros(rec, dtype=torch.uint8)
    _raises(lambda: c.store_records("s", 0, H_kv, 16, D, ok, ok), "must be on the CUDA device")


def _desc(**kw):
    d = dict(sid="s", layer=0, Q=torch.zeros((H_q, D), **f32), O=torch.zeros((H_q, D), **f32),
             LSE=torch.zeros((H_q,), **f32), K_suf=torch.zeros((H_kv, S, D), **f16),
             V_suf=torch.zeros((H_kv, S, D), **f16), idx=torch.zeros((H_q, 4), dtype=torch.int32))
    d.update(kw)
    return d


def test_batch_descriptors():
    c = _ctx()
    dense = lambda d, **kw: c.batch_caller([_desc(), d], H_q, H_kv, D, S_suf=S, **kw)
    _raises(lambda: dense(_desc(Q=torch.zeros((H_q, D), **f16))), "descs[1].Q: dtype")
    _raises(lambda: dense(_desc(), q_dtype=binding.DT_F16), "descs[0].Q: dtype")
    _raises(lambda: dense(_desc(O=torch.zeros((H_q, D - 1), **f32))), "descs[1].O: ")
    _raises(lambda: dense(_desc(K_suf=torch.zeros((H_kv, S - 1, D), **f16))), "descs[1].K_suf: ")
    _raises(lambda: dense(_desc(V_suf=torch.zeros((H_kv, S, D), **f32))), "descs[1].V_suf: dtype")
    _raises(lambda: c.query_batch([_desc(LSE=torch.zeros((H_q - 1,), **f32))], H_q, H_kv, D, S_suf=S),
            "descs[0].LSE: ")
    _raises(lambda: c.sparse_batch_caller([_desc(idx=torch.zeros((H_q, 4), dtype=torch.int64))], H_q, H_kv, D,
                                          64, 4, S_suf=S), "descs[0].idx: dtype")
    _raises(lambda: dense(_desc()), "must be on the CUDA device")
    _raises(lambda: c.batch_caller([_desc()], H_q, H_kv, D, q_dtype=7), "q_dtype")


def test_quantizer_output_size():
    x = torch.zeros((3, 64), **f16)
    _raises(lambda: binding.quantize_mlx4g32(x, out=torch.zeros((3, 39), dtype=torch.uint8)), "out: ")
    _raises(lambda: binding.quantize_mlx4g32(x[0]), "x must be [rows, kv_dim]")
    _raises(lambda: binding.quantize_mlx4g32(x), "must be on the CUDA device")
