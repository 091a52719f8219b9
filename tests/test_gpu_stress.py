"""Parity on inputs that push the online softmax and the number formats to their edges, against
the oracle, on every path: fp16 and mlx4g32 M=1 decode (with and without a fused suffix),
batched-Q (M > 1, causal suffix) and block-mean top-K sparse.

The inputs (prefix_cached_kv_gb300.synth.gen_stress): Q scaled by 30 and by 100 (scaled logits
in the hundreds); scores rising through the whole sequence (the running maximum moves on every
tile or chunk); one dominant key in the prefix, or in the suffix (under the causal mask when
M > 1, where the rows that must not see it are checked to be unaffected); mlx4g32 groups with a
large bias and a tiny scale. Scores stay below ~500 in magnitude, where fp32 can still meet the
absolute LSE tolerance. An fp32 Q element outside the documented range is reported by the
device error word (code 7) instead of producing silent infinities."""
import numpy as np
import pytest
import torch

from oracle import pck_oracle as orc
from prefix_cached_kv_gb300 import synth
from tests.gpu_util import TIE_EPS, assert_close_o_lse, ctx_factory, dev, host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = ctx_factory()
    yield c
    c.close()


def _oracle_kv(K, V, fmt):
    if fmt == 0:
        return K.astype(np.float64), V.astype(np.float64)
    H, N, D = K.shape
    return [orc.dequantize_mlx4g32(*orc.quantize_mlx4g32(X.reshape(H * N, D))).reshape(H, N, D) for X in (K, V)]


M1_KINDS = ["q30", "q100", "monotone", "dominant_prefix", "dominant_suffix", "bias_scale"]
M1_SHAPES = [
    # H_q, H_kv, N, D, S_suf
    (32, 8, 600, 64, 16),      # GQA 4, the headline head shape
    (16, 2, 400, 128, 24),     # GQA 8: two 4-head column blocks
    (8, 4, 300, 256, 8),       # D = 256
]


@pytest.mark.parametrize("kind", M1_KINDS)
@pytest.mark.parametrize("shape", M1_SHAPES)
@pytest.mark.parametrize("fmt", [0, 1])
def test_stress_decode(ctx, kind, shape, fmt):
    H_q, H_kv, N, D, S = shape
    Q, K, V, Ks, Vs = synth.gen_stress(kind, 3 + D, H_q, H_kv, N, D, 1, S)
    hm = synth.default_head_map(H_q, H_kv)
    sid = f"st{kind}{D}{fmt}"
    ctx.store(sid, 0, dev(K), dev(V), fmt=fmt)
    Ko, Vo = _oracle_kv(K, V, fmt)
    O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs))
    O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"decode {kind} {shape} fmt={fmt}")
    if kind != "dominant_suffix":   # the prefix alone (no suffix warps, no suffix merge)
        O1, L1 = ctx.query(sid, 0, dev(Q))
        O1_ref, L1_ref = orc.prefix_query(Q, Ko, Vo, hm)
        ctx.sync()
        assert_close_o_lse(host(O1), host(L1), O1_ref, L1_ref, f"decode prefix-only {kind} {shape} fmt={fmt}")
    ctx.drop(sid)


@pytest.mark.parametrize("kind", M1_KINDS)
def test_stress_decode_batched(ctx, kind):
    """The same inputs through one pck_query_batch launch of 3 sessions (mlx4g32)."""
    H_q, H_kv, N, D, S = 32, 8, 500, 64, 16
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs = [], []
    for r in range(3):
        Q, K, V, Ks, Vs = synth.gen_stress(kind, 50 + r, H_q, H_kv, N, D, 1, S)
        ctx.store(f"stb{r}", 0, dev(K), dev(V), fmt=1)
        Ko, Vo = _oracle_kv(K, V, 1)
        refs.append(orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs))
        descs.append(dict(sid=f"stb{r}", layer=0, Q=dev(Q[:, 0]), O=torch.empty((H_q, D), device="cuda"),
                          LSE=torch.empty((H_q,), device="cuda"), K_suf=dev(Ks), V_suf=dev(Vs)))
    ctx.query_batch(descs, H_q, H_kv, D, S_suf=S)
    ctx.sync()
    for r, (O_ref, L_ref) in enumerate(refs):
        assert_close_o_lse(host(descs[r]["O"]), host(descs[r]["LSE"]), O_ref[:, 0], L_ref[:, 0], f"batch {kind} {r}")
        ctx.drop(f"stb{r}")


PF_KINDS = ["q30", "q100", "monotone", "dominant_prefix", "dominant_suffix", "bias_scale"]


@pytest.mark.parametrize("kind", PF_KINDS)
@pytest.mark.parametrize("D", [64, 128, 256])
def test_stress_prefill(ctx, kind, D):
    """Batched-Q with a causal suffix (M = S_suf = 64): for the dominant suffix key, the rows that
    the mask hides it from are compared like every other row, so a key leaking through the mask
    would dominate them and fail."""
    H_q, H_kv, N, M, S = 6, 2, 300, 64, 64
    Q, K, V, Ks, Vs = synth.gen_stress(kind, 11 + D, H_q, H_kv, N, D, M, S, rise=0.9, q_dtype=np.float16)
    hm = synth.default_head_map(H_q, H_kv)
    sid = f"stp{kind}{D}"
    ctx.store(sid, 0, dev(K), dev(V))
    O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs), causal=True)
    O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs, causal=True)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"prefill {kind} D={D}")
    ctx.drop(sid)


def test_stress_prefill_dominant_suffix_key_is_masked(ctx):
    """A suffix key that dominates every score it enters: row i (M = S_suf, standard causal) sees
    it only when i >= j*, so rows before j* must equal the attention without that key."""
    H_q, H_kv, N, M, S, D = 4, 1, 200, 96, 96, 128
    Q, K, V, Ks, Vs = synth.gen_stress("dominant_suffix", 5, H_q, H_kv, N, D, M, S, q_dtype=np.float16)
    hm = synth.default_head_map(H_q, H_kv)
    ctx.store("stmask", 0, dev(K), dev(V))
    O, L = ctx.query_fused("stmask", 0, dev(Q), dev(Ks), dev(Vs), causal=True)
    O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs, causal=True)
    ctx.sync()
    o, l = host(O), host(L)
    assert_close_o_lse(o, l, O_ref, L_ref, "prefill dominant suffix")
    # the dominant key: where the oracle's LSE jumps by ~60
    jumps = np.flatnonzero(np.diff(L_ref[0]) > 30)
    assert len(jumps) == 1
    j_star = jumps[0] + 1
    assert 0 < j_star < M
    assert (L_ref[:, :j_star] < L_ref[:, j_star:].min() - 30).all()
    assert (l[:, :j_star] < L_ref[:, j_star:].min() - 30).all()
    ctx.drop("stmask")


SP_KINDS = ["q30", "q100", "monotone", "dominant_prefix"]


@pytest.mark.parametrize("kind", SP_KINDS)
def test_stress_sparse(ctx, kind):
    H_q, H_kv, N, D, B, Kt, S = 8, 2, 2000, 128, 64, 4, 16
    Q, K, V, Ks, Vs = synth.gen_stress(kind, 21, H_q, H_kv, N, D, 1, S)
    Q = Q[:, 0]
    hm = synth.default_head_map(H_q, H_kv)
    sid = f"sts{kind}"
    ctx.store(sid, 0, dev(K), dev(V))
    O, L, idx = ctx.query_sparse_auto(sid, 0, dev(Q), B, Kt, H_kv, K_suf=dev(Ks), V_suf=dev(Vs))
    O_ref, L_ref, idx_ref, scores = orc.sparse_query(Q, K, V, hm, B, Kt, Ks, Vs)
    ok = orc.topk_margin(scores, Kt) >= TIE_EPS
    idx = host(idx)
    assert np.array_equal(idx[ok], idx_ref[ok])
    assert_close_o_lse(host(O)[ok], host(L)[ok], O_ref[ok], L_ref[ok], f"sparse {kind}")
    ctx.drop(sid)


def test_q_out_of_range_is_reported(ctx):
    """An fp32 Q element with |q| log2(e) / sqrt(D) >= 65504 cannot be carried by the M=1 kernels'
    fp16 hi + lo pair: the call still returns OK (it is asynchronous), and pck_sync reports
    PCK_ECUDA naming code 7; the context stays usable and the next in-range query is correct."""
    from prefix_cached_kv_gb300 import binding
    H_q, H_kv, N, D = 8, 2, 100, 64
    K, V = synth.gen_kv(9, H_kv, N, D)
    Q = synth.gen_q(9, H_q, 1, D)
    ctx.store("qr", 0, dev(K), dev(V), fmt=1)
    bad = Q.copy()
    bad[3, 0, 5] = 4.0e5   # 4e5 * 1.4427 / 8 = 72,135 > 65504
    ctx.query("qr", 0, dev(bad))
    with pytest.raises(binding.PckError) as e:
        ctx.sync()
    assert e.value.code == binding.ECUDA and "code 7" in str(e.value)
    O, L = ctx.query("qr", 0, dev(Q))
    ctx.sync()
    Ko, Vo = _oracle_kv(K, V, 1)
    O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, synth.default_head_map(H_q, H_kv))
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, "after the range error")
    ctx.drop("qr")
