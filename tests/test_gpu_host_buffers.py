"""pck_query_batch_host: the batched M=1 query over page-locked HOST buffers (the library copies
the inputs in and writes O and LSE back itself). Against the same batch over device buffers
(bit-identical: the same kernels on the same bytes) and the oracle, inside a CUDA graph replayed
with new host inputs, and the rejection of pointers that are not page-locked host memory."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import pck_oracle as orc
from prefix_cached_kv_gb300 import synth
from tests.gpu_util import assert_close_o_lse, ctx_factory, dev, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = ctx_factory()
    yield c
    c.close()


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


@pytest.mark.parametrize("fmt,H_q,H_kv,D,S,q16", [
    (1, 32, 8, 64, 16, False),    # the GQA decode layer shape, mlx4g32
    (0, 8, 8, 128, 0, False),     # fp16 slots, no suffix
    (0, 12, 2, 96, 24, True),     # fp16 Q, a head dim of the second set
])
def test_host_batch_matches_device_batch_and_oracle(ctx, fmt, H_q, H_kv, D, S, q16):
    from prefix_cached_kv_gb300 import binding
    hm = synth.default_head_map(H_q, H_kv)
    qdt = np.float16 if q16 else np.float32
    hdescs, ddescs, refs = [], [], []
    for r, N in enumerate((700, 2048, 33, 1500, 4096, 16)):
        K, V = synth.gen_kv(300 + r, H_kv, N, D)
        Q = synth.gen_q(300 + r, H_q, 1, D, dtype=qdt)[:, 0]
        sid = f"hb{fmt}{r}"
        ctx.store(sid, 0, dev(K), dev(V), fmt=fmt)
        Ko, Vo = K.astype(np.float64), V.astype(np.float64)
        if fmt == 1:
            Ko, Vo = [orc.dequantize_mlx4g32(*orc.quantize_mlx4g32(X.reshape(H_kv * N, D))).reshape(H_kv, N, D)
                      for X in (K, V)]
        hd = dict(sid=sid, layer=0, Q=_pinned(Q), O=torch.empty((H_q, D)).pin_memory(), LSE=torch.empty((H_q,)).pin_memory())
        dd = dict(sid=sid, layer=0, Q=dev(Q), O=torch.empty((H_q, D), device="cuda"), LSE=torch.empty((H_q,), device="cuda"))
        if S:
            Ks, Vs = synth.gen_suffix(300 + r, H_kv, S, D)
            hd["K_suf"], hd["V_suf"] = _pinned(Ks), _pinned(Vs)
            dd["K_suf"], dd["V_suf"] = dev(Ks), dev(Vs)
            refs.append(orc.prefix_query(Q[:, None], Ko, Vo, hm, Ks, Vs))
        else:
            refs.append(orc.prefix_query(Q[:, None], Ko, Vo, hm))
        hdescs.append(hd)
        ddescs.append(dd)
    qd = binding.DT_F16 if q16 else binding.DT_F32
    ctx.batch_caller(hdescs, H_q, H_kv, D, S_suf=S, q_dtype=qd, host=True)()
    ctx.batch_caller(ddescs, H_q, H_kv, D, S_suf=S, q_dtype=qd)()
    ctx.sync()
    torch.cuda.synchronize()
    for r, (hd, dd, (O_ref, L_ref)) in enumerate(zip(hdescs, ddescs, refs)):
        assert torch.equal(hd["O"], dd["O"].cpu()) and torch.equal(hd["LSE"], dd["LSE"].cpu()), f"session {r}"
        assert_close_o_lse(hd["O"].numpy(), hd["LSE"].numpy(), O_ref[:, 0], L_ref[:, 0], f"host batch {r}")
    for r in range(6):
        ctx.drop(f"hb{fmt}{r}")


def test_host_batch_in_a_cuda_graph_follows_new_host_inputs(ctx):
    """The call captured once and replayed twice; the host writes a new Q into the same pinned
    buffer before the second replay, and the outputs follow it."""
    H_q, H_kv, N, D, S = 32, 8, 1024, 64, 16
    hm = synth.default_head_map(H_q, H_kv)
    K, V = synth.gen_kv(5, H_kv, N, D)
    ctx.store("hbg", 0, dev(K), dev(V), fmt=1)
    Ko, Vo = [orc.dequantize_mlx4g32(*orc.quantize_mlx4g32(X.reshape(H_kv * N, D))).reshape(H_kv, N, D) for X in (K, V)]
    Ks, Vs = synth.gen_suffix(5, H_kv, S, D)
    d = dict(sid="hbg", layer=0, Q=torch.empty((H_q, D)).pin_memory(), O=torch.empty((H_q, D)).pin_memory(),
             LSE=torch.empty((H_q,)).pin_memory(), K_suf=_pinned(Ks), V_suf=_pinned(Vs))
    call = ctx.batch_caller([d], H_q, H_kv, D, S_suf=S, host=True)
    d["Q"].copy_(torch.from_numpy(synth.gen_q(6, H_q, 1, D)[:, 0]))
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=st):
        call()
    torch.cuda.current_stream().wait_stream(st)
    for seed in (7, 8):
        Q = synth.gen_q(seed, H_q, 1, D)
        d["Q"].copy_(torch.from_numpy(Q[:, 0]))
        g.replay()
        torch.cuda.synchronize()
        ctx.sync()
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs)
        assert_close_o_lse(d["O"].numpy(), d["LSE"].numpy(), O_ref[:, 0], L_ref[:, 0], f"replay seed {seed}")
    del g
    ctx.drop("hbg")


def test_host_batch_rejects_memory_that_is_not_page_locked(ctx):
    from prefix_cached_kv_gb300 import binding
    H_q, H_kv, N, D = 8, 2, 256, 64
    K, V = synth.gen_kv(9, H_kv, N, D)
    ctx.store("hbr", 0, dev(K), dev(V))
    good = dict(sid="hbr", layer=0, Q=torch.zeros((H_q, D)).pin_memory(), O=torch.empty((H_q, D)).pin_memory())
    with pytest.raises(ValueError):   # the binding refuses device tensors ...
        ctx.batch_caller([dict(good, Q=torch.zeros((H_q, D), device="cuda"))], H_q, H_kv, D, host=True)
    with pytest.raises(ValueError):   # ... and pageable host tensors
        ctx.batch_caller([dict(good, O=torch.empty((H_q, D)))], H_q, H_kv, D, host=True)
    # the library itself refuses a device pointer and a pageable one (raw C-ABI call)
    lib = binding.load_library()
    for q in (torch.zeros((H_q, D), device="cuda"), torch.zeros((H_q, D))):
        arr = (binding.QueryDesc * 1)()
        sid = b"hbr"
        arr[0] = binding.QueryDesc(sid, 0, q.data_ptr(), good["O"].data_ptr(), None, None, None)
        rc = lib.pck_query_batch_host(ctx.h, 1, arr, H_q, H_kv, D, 0, binding.DT_F32, None, None)
        assert rc == binding.EINVAL
    ctx.drop("hbr")
