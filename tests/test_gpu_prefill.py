"""Batched-Q (M > 1) attention on the tcgen05 kernel vs the oracle: prefix + causal suffix,
GQA packing of q heads into the 128-row tiles, ragged prefix/suffix lengths."""
import numpy as np
import pytest

from oracle import pck_oracle as orc
from prefix_cached_kv_gb300 import synth
from tests.gpu_util import assert_close_o_lse, ctx_factory, dev, host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = ctx_factory()
    yield c
    c.close()


CASES = [
    # H_q, H_kv, N, M, S_suf, D, causal
    (1, 1, 128, 128, 0, 64, True),
    (2, 1, 100, 64, 0, 128, True),
    (4, 2, 300, 130, 40, 64, True),
    (3, 1, 256, 128, 128, 128, True),
    (6, 2, 1000, 96, 200, 128, False),
    (2, 2, 33, 200, 17, 64, True),      # M > S_suf: early rows see no suffix
    (8, 8, 17, 16, 16, 128, True),
    (12, 1, 200, 50, 30, 64, True),     # GQA 12: two work groups on one kv head, 600 + 0 rows
    (2, 1, 1, 2, 3, 128, True),         # N = 1, M = 2: one partial key block, two suffix rows
    (1, 1, 4133, 16, 8, 64, True),      # one row tile: 32 key-range splits over 65 blocks (ragged)
    (4, 1, 500, 129, 0, 128, True),     # 516 rows: four full row tiles and one of 4 rows
    # D = 256: 512 TMEM columns, one CTA per SM, the general merge (two float4 of d per lane)
    (4, 2, 300, 130, 40, 256, True),
    (3, 1, 256, 128, 128, 256, True),
    (6, 2, 1000, 96, 200, 256, False),
    (2, 1, 1, 2, 3, 256, True),
    (1, 1, 4133, 16, 8, 256, True),     # 32 key-range splits
    (12, 1, 200, 50, 30, 256, True),    # GQA 12
]


@pytest.mark.parametrize("H_q,H_kv,N,M,S,D,causal", CASES)
def test_prefill_matches_oracle(ctx, H_q, H_kv, N, M, S, D, causal):
    seed = N + M + S + D + H_q
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, M, D, dtype=np.float16)
    hm = synth.default_head_map(H_q, H_kv)
    sid = f"pf{seed}"
    ctx.store(sid, 0, dev(K), dev(V))
    if S:
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs), causal=causal)
        O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs, causal=causal)
    else:
        O, L = ctx.query(sid, 0, dev(Q))
        O_ref, L_ref = orc.prefix_query(Q, K, V, hm)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"{(H_q, H_kv, N, M, S, D, causal)}")
    ctx.drop(sid)


def test_prefill_batched_q_workload_layer(ctx):
    """One layer of the batched-Q workload: H_q=24, H_kv=8, D=128, N=4096, M=512, causal S_suf=512."""
    w = synth.WORKLOADS["batched_q_prefill"]
    H_q, H_kv, N, D, M, S = w["H_q"], w["H_kv"], w["N"], w["D"], w["M"], w["S_suf"]
    K, V = synth.gen_kv(0, H_kv, N, D)
    Q = synth.gen_q(0, H_q, M, D, dtype=np.float16)
    Ks, Vs = synth.gen_suffix(0, H_kv, S, D)
    hm = synth.default_head_map(H_q, H_kv)
    ctx.store("pfcfg", 0, dev(K), dev(V))
    O, L = ctx.query_fused("pfcfg", 0, dev(Q), dev(Ks), dev(Vs), causal=True)
    O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs, causal=True)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, "batched-Q layer")
    ctx.drop("pfcfg")


@pytest.mark.parametrize("H_q,H_kv,hm", [
    (6, 3, [2, 0, 1, 1, 0, 2]),         # q heads of a kv head not adjacent
    (4, 2, [0, 0, 0, 0]),               # kv head 1 has no q heads
])
def test_prefill_custom_head_map(ctx, H_q, H_kv, hm):
    N, M, S, D = 300, 70, 40, 64
    hm = np.array(hm, dtype=np.int32)
    K, V = synth.gen_kv(21, H_kv, N, D)
    Q = synth.gen_q(21, H_q, M, D, dtype=np.float16)
    Ks, Vs = synth.gen_suffix(21, H_kv, S, D)
    ctx.store("pfhm", 0, dev(K), dev(V))
    O, L = ctx.query_fused("pfhm", 0, dev(Q), dev(Ks), dev(Vs), head_map=hm, causal=True)
    O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs, causal=True)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"batched-Q head_map {hm.tolist()}")
    ctx.drop("pfhm")


MLX_CASES = [
    # H_q, H_kv, N, M, S_suf, D, causal
    (4, 2, 300, 130, 40, 64, True),
    (3, 1, 256, 128, 128, 128, True),
    (6, 2, 1000, 96, 200, 128, False),
    (2, 1, 1, 2, 3, 64, True),
    (1, 1, 4133, 16, 8, 128, True),     # 32 key-range splits: the general merge folds hi and lo
    (1, 1, 4133, 16, 8, 64, True),
    (12, 1, 200, 50, 30, 64, True),
]


@pytest.mark.parametrize("H_q,H_kv,N,M,S,D,causal", MLX_CASES)
def test_prefill_over_mlx4g32_matches_oracle(ctx, H_q, H_kv, N, M, S, D, causal):
    """M > 1 over an mlx4g32 slot: the oracle attends to the dequantised codes of the same fp16
    K/V (the library quantised them itself)."""
    seed = N + M + S + D + H_q + 1
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, M, D, dtype=np.float16)
    hm = synth.default_head_map(H_q, H_kv)
    Ko, Vo = [orc.dequantize_mlx4g32(*orc.quantize_mlx4g32(X.reshape(H_kv * N, D))).reshape(H_kv, N, D) for X in (K, V)]
    sid = f"pfm{seed}"
    ctx.store(sid, 0, dev(K), dev(V), fmt=1)
    if S:
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs), causal=causal)
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs, causal=causal)
    else:
        O, L = ctx.query(sid, 0, dev(Q))
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"mlx4g32 {(H_q, H_kv, N, M, S, D, causal)}")
    ctx.drop(sid)


@pytest.mark.parametrize("kind", ["bias_scale", "q100", "monotone", "dominant_suffix"])
def test_prefill_over_mlx4g32_stress(ctx, kind):
    H_q, H_kv, N, M, S, D = 6, 2, 300, 64, 64, 128
    Q, K, V, Ks, Vs = synth.gen_stress(kind, 17, H_q, H_kv, N, D, M, S, rise=0.9, q_dtype=np.float16)
    hm = synth.default_head_map(H_q, H_kv)
    Ko, Vo = [orc.dequantize_mlx4g32(*orc.quantize_mlx4g32(X.reshape(H_kv * N, D))).reshape(H_kv, N, D) for X in (K, V)]
    ctx.store("pfms", 0, dev(K), dev(V), fmt=1)
    O, L = ctx.query_fused("pfms", 0, dev(Q), dev(Ks), dev(Vs), causal=True)
    O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs, causal=True)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"mlx4g32 prefill {kind}")
    ctx.drop("pfms")


def test_prefill_over_mlx4g32_workload_layer(ctx):
    """One layer of the batched-Q workload (H_q=24, H_kv=8, D=128, N=4096, M=512, causal S_suf=512)
    with the prefix stored as mlx4g32."""
    w = synth.WORKLOADS["batched_q_prefill"]
    H_q, H_kv, N, D, M, S = w["H_q"], w["H_kv"], w["N"], w["D"], w["M"], w["S_suf"]
    K, V = synth.gen_kv(1, H_kv, N, D)
    Q = synth.gen_q(1, H_q, M, D, dtype=np.float16)
    Ks, Vs = synth.gen_suffix(1, H_kv, S, D)
    hm = synth.default_head_map(H_q, H_kv)
    Ko, Vo = [orc.dequantize_mlx4g32(*orc.quantize_mlx4g32(X.reshape(H_kv * N, D))).reshape(H_kv, N, D) for X in (K, V)]
    ctx.store("pfm3", 0, dev(K), dev(V), fmt=1)
    O, L = ctx.query_fused("pfm3", 0, dev(Q), dev(Ks), dev(Vs), causal=True)
    O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs, causal=True)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, "mlx4g32 batched-Q layer")
    ctx.drop("pfm3")
