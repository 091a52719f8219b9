"""The longest prefixes and the largest head counts the kernels take, against the oracle: an M=1
decode over a million-token prefix (fp16 and mlx4g32, ragged tails, a suffix), the batched-Q
kernel over a 65,537-token prefix (many key-range splits and a ragged last block), and 64 q
heads on one kv head."""
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


def _oracle_kv(K, V, fmt):
    if fmt == 0:
        return K.astype(np.float64), V.astype(np.float64)
    H, N, D = K.shape
    return [orc.dequantize_mlx4g32(*orc.quantize_mlx4g32(X.reshape(H * N, D))).reshape(H, N, D) for X in (K, V)]


@pytest.mark.parametrize("fmt,N", [(0, 1_000_003), (1, 600_001)])
def test_decode_million_token_prefix(ctx, fmt, N):
    H_q, H_kv, D, S = 4, 1, 64, 5
    K, V = synth.gen_kv(11 + fmt, H_kv, N, D)
    Q = synth.gen_q(11 + fmt, H_q, 1, D)
    Ks, Vs = synth.gen_suffix(11 + fmt, H_kv, S, D)
    ctx.store("long", 0, dev(K), dev(V), fmt=fmt)
    O, L = ctx.query_fused("long", 0, dev(Q), dev(Ks), dev(Vs))
    Ko, Vo = _oracle_kv(K, V, fmt)
    O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, synth.default_head_map(H_q, H_kv), Ks, Vs)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"N={N} fmt={fmt}")
    ctx.drop("long")


def test_prefill_long_prefix(ctx):
    H_q, H_kv, N, M, S, D = 2, 1, 65_537, 256, 96, 64
    K, V = synth.gen_kv(12, H_kv, N, D)
    Q = synth.gen_q(12, H_q, M, D, dtype=np.float16)
    Ks, Vs = synth.gen_suffix(12, H_kv, S, D)
    ctx.store("longp", 0, dev(K), dev(V))
    O, L = ctx.query_fused("longp", 0, dev(Q), dev(Ks), dev(Vs), causal=True)
    O_ref, L_ref = orc.prefix_query(Q, K, V, synth.default_head_map(H_q, H_kv), Ks, Vs, causal=True)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, "prefill N=65537")
    ctx.drop("longp")


@pytest.mark.parametrize("M", [1, 64])
def test_sixty_four_q_heads_on_one_kv_head(ctx, M):
    """H_q = 64 (the limit) on H_kv = 1: eight work groups of 8 q heads at M = 1, one 128-row tile
    per two heads at M = 64."""
    H_q, H_kv, N, D, S = 64, 1, 3000, 128, 12
    K, V = synth.gen_kv(13 + M, H_kv, N, D)
    Q = synth.gen_q(13 + M, H_q, M, D, dtype=np.float16 if M > 1 else np.float32)
    Ks, Vs = synth.gen_suffix(13 + M, H_kv, S, D)
    ctx.store("wide", 0, dev(K), dev(V))
    O, L = ctx.query_fused("wide", 0, dev(Q), dev(Ks), dev(Vs), causal=True)
    O_ref, L_ref = orc.prefix_query(Q, K, V, synth.default_head_map(H_q, H_kv), Ks, Vs, causal=True)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"H_q=64 M={M}")
    ctx.drop("wide")
