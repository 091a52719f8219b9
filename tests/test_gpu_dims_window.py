"""The head dimensions beyond 64/128/256 (fp16 M=1 decode at D = 32, 96, 160, 192, 512 and
batched-Q at D = 32, 96, 160, 192; mlx4g32 M=1 at D = 192) and the attention window (fa_window,
M = 1) on the GPU, against the oracle."""
import numpy as np
import pytest
import torch

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


DIM_CASES = [
    # H_q, H_kv, N, D, S_suf, fmt
    (8, 8, 1000, 32, 0, 0),
    (32, 8, 777, 32, 16, 0),
    (16, 2, 500, 96, 20, 0),       # GQA 8: two column blocks
    (8, 4, 333, 96, 0, 0),
    (8, 2, 1200, 160, 7, 0),
    (16, 2, 300, 160, 0, 0),
    (8, 8, 900, 192, 16, 0),
    (16, 2, 400, 192, 33, 0),
    (32, 8, 1000, 192, 16, 1),     # mlx4g32 at D = 192
    (16, 2, 257, 192, 5, 1),
    (8, 8, 1000, 512, 0, 0),       # D = 512: q fragments in shared memory, one ring stage
    (32, 8, 777, 512, 16, 0),      # GQA 4: one work group per kv head
    (16, 2, 500, 512, 20, 0),      # GQA 8: two work groups of 4 per kv head
    (12, 1, 2049, 512, 3, 0),      # GQA 12: three work groups, ragged tail
    (2, 1, 1, 512, 0, 0),          # N = 1
]


@pytest.mark.parametrize("H_q,H_kv,N,D,S,fmt", DIM_CASES)
def test_decode_other_head_dims(ctx, H_q, H_kv, N, D, S, fmt):
    seed = N + D + S + fmt
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, 1, D)
    hm = synth.default_head_map(H_q, H_kv)
    sid = f"dim{seed}"
    ctx.store(sid, 0, dev(K), dev(V), fmt=fmt)
    Ko, Vo = _oracle_kv(K, V, fmt)
    if S:
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs))
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs)
    else:
        O, L = ctx.query(sid, 0, dev(Q))
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"D={D} {(H_q, H_kv, N, S, fmt)}")
    ctx.drop(sid)


def test_decode_d512_fp16_q_and_custom_head_map(ctx):
    """D = 512 with fp16 Q and q heads of a kv head that are not adjacent (5 of them: groups of
    4 and 1)."""
    H_q, H_kv, N, D, S = 10, 2, 640, 512, 9
    K, V = synth.gen_kv(51, H_kv, N, D)
    Q = synth.gen_q(51, H_q, 1, D, dtype=np.float16)
    hm = np.array([h % 2 for h in range(H_q)], dtype=np.int32)
    Ks, Vs = synth.gen_suffix(51, H_kv, S, D)
    ctx.store("d512h", 0, dev(K), dev(V))
    O, L = ctx.query_fused("d512h", 0, dev(Q), dev(Ks), dev(Vs), head_map=hm)
    O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, "D=512 fp16 Q, custom head_map")
    ctx.drop("d512h")


def test_decode_d512_batched(ctx):
    """pck_query_batch at D = 512: 5 sessions of different lengths, GQA 8, with a suffix."""
    H_q, H_kv, D, S = 16, 2, 512, 16
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs = [], []
    for r, N in enumerate((1000, 3000, 17, 512, 1601)):
        K, V = synth.gen_kv(90 + r, H_kv, N, D)
        Q = synth.gen_q(90 + r, H_q, 1, D)
        Ks, Vs = synth.gen_suffix(90 + r, H_kv, S, D)
        ctx.store(f"d5b{r}", 0, dev(K), dev(V))
        refs.append(orc.prefix_query(Q, K, V, hm, Ks, Vs))
        descs.append(dict(sid=f"d5b{r}", layer=0, Q=dev(Q[:, 0]), O=torch.empty((H_q, D), device="cuda"),
                          LSE=torch.empty((H_q,), device="cuda"), K_suf=dev(Ks), V_suf=dev(Vs)))
    ctx.query_batch(descs, H_q, H_kv, D, S_suf=S)
    ctx.sync()
    for r, (O_ref, L_ref) in enumerate(refs):
        assert_close_o_lse(host(descs[r]["O"]), host(descs[r]["LSE"]), O_ref[:, 0], L_ref[:, 0], f"D=512 batch {r}")
        ctx.drop(f"d5b{r}")


def test_d512_stress(ctx):
    """Large logits, scores rising through prefix and suffix, and dominant keys at D = 512."""
    for kind in ("q100", "monotone", "dominant_prefix", "dominant_suffix"):
        Q, K, V, Ks, Vs = synth.gen_stress(kind, 512, 8, 2, 700, 512, 1, 16)
        hm = synth.default_head_map(8, 2)
        ctx.store("d5s", 0, dev(K), dev(V))
        O, L = ctx.query_fused("d5s", 0, dev(Q), dev(Ks), dev(Vs))
        O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs)
        ctx.sync()
        assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"D=512 stress {kind}")
    ctx.drop("d5s")


def test_d512_rejections(ctx):
    """D = 512 is built for fp16 slots at M = 1 only: M > 1, an mlx4g32 slot and the block-mean
    sparse forms are refused before launch."""
    from prefix_cached_kv_gb300 import binding
    K, V = synth.gen_kv(4, 2, 300, 512)
    ctx.store("d5r", 0, dev(K), dev(V))
    with pytest.raises(binding.PckError) as e:
        ctx.query("d5r", 0, dev(synth.gen_q(4, 4, 8, 512, dtype=np.float16)))
    assert e.value.code == binding.EUNSUPPORTED
    with pytest.raises(binding.PckError) as e:
        ctx.query_sparse_auto("d5r", 0, dev(synth.gen_q(4, 4, 1, 512)[:, 0]), 64, 2, 2)
    assert e.value.code == binding.EUNSUPPORTED
    with pytest.raises(binding.PckError) as e:
        ctx.store("d5q", 0, dev(K), dev(V), fmt=1)
    assert e.value.code == binding.EUNSUPPORTED
    ctx.drop("d5r")


def test_decode_other_head_dims_batched(ctx):
    """pck_query_batch at D = 160: 6 sessions of different lengths, with a suffix."""
    H_q, H_kv, D, S = 8, 2, 160, 12
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs = [], []
    for r, N in enumerate((1000, 2048, 17, 999, 1600, 640)):
        K, V = synth.gen_kv(80 + r, H_kv, N, D)
        Q = synth.gen_q(80 + r, H_q, 1, D)
        Ks, Vs = synth.gen_suffix(80 + r, H_kv, S, D)
        ctx.store(f"db{r}", 0, dev(K), dev(V))
        refs.append(orc.prefix_query(Q, K, V, hm, Ks, Vs))
        descs.append(dict(sid=f"db{r}", layer=0, Q=dev(Q[:, 0]), O=torch.empty((H_q, D), device="cuda"),
                          LSE=torch.empty((H_q,), device="cuda"), K_suf=dev(Ks), V_suf=dev(Vs)))
    ctx.query_batch(descs, H_q, H_kv, D, S_suf=S)
    ctx.sync()
    for r, (O_ref, L_ref) in enumerate(refs):
        assert_close_o_lse(host(descs[r]["O"]), host(descs[r]["LSE"]), O_ref[:, 0], L_ref[:, 0], f"batch {r}")
        ctx.drop(f"db{r}")


@pytest.mark.parametrize("H_q,H_kv,N,M,S,D", [
    (2, 1, 300, 130, 40, 32),
    (4, 2, 1000, 96, 96, 96),
    (3, 1, 500, 128, 64, 160),
    (6, 2, 700, 64, 64, 192),
    (1, 1, 4133, 16, 8, 192),      # many key-range splits at one CTA per SM
])
def test_prefill_other_head_dims(ctx, H_q, H_kv, N, M, S, D):
    seed = N + M + S + D
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, M, D, dtype=np.float16)
    Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
    hm = synth.default_head_map(H_q, H_kv)
    sid = f"pd{seed}"
    ctx.store(sid, 0, dev(K), dev(V))
    O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs), causal=True)
    O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs, causal=True)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"prefill D={D}")
    ctx.drop(sid)


@pytest.mark.parametrize("D", [96, 192])
def test_other_head_dims_stress(ctx, D):
    """Large logits and a dominant key at the new dims (decode fp16 and batched-Q)."""
    for kind in ("q100", "dominant_prefix"):
        Q, K, V, Ks, Vs = synth.gen_stress(kind, D, 8, 2, 500, D, 1, 16)
        hm = synth.default_head_map(8, 2)
        ctx.store("dst", 0, dev(K), dev(V))
        O, L = ctx.query_fused("dst", 0, dev(Q), dev(Ks), dev(Vs))
        O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs)
        ctx.sync()
        assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"decode stress {kind} D={D}")
        Q, K, V, Ks, Vs = synth.gen_stress(kind, D + 1, 4, 2, 300, D, 64, 64, q_dtype=np.float16)
        hm = synth.default_head_map(4, 2)
        ctx.store("dst", 1, dev(K), dev(V))
        O, L = ctx.query_fused("dst", 1, dev(Q), dev(Ks), dev(Vs), causal=True)
        O_ref, L_ref = orc.prefix_query(Q, K, V, hm, Ks, Vs, causal=True)
        ctx.sync()
        assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"prefill stress {kind} D={D}")
    ctx.drop("dst")


WINDOW_SHAPES = [
    # H_q, H_kv, N, D, S_suf, fmt
    (32, 8, 1000, 64, 16, 1),
    (32, 8, 1000, 64, 16, 0),
    (8, 2, 777, 128, 0, 0),
    (8, 2, 777, 128, 0, 1),
    (16, 4, 300, 256, 40, 0),
    (8, 2, 500, 96, 24, 0),
    (8, 2, 500, 512, 24, 0),
]


@pytest.mark.parametrize("shape", WINDOW_SHAPES)
def test_window_matches_oracle(ctx, shape):
    H_q, H_kv, N, D, S, fmt = shape
    seed = N + D + S + fmt + 5
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, 1, D)
    hm = synth.default_head_map(H_q, H_kv)
    Ko, Vo = _oracle_kv(K, V, fmt)
    Ks = Vs = None
    if S:
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
    sid = f"win{seed}"
    ctx.store(sid, 0, dev(K), dev(V), fmt=fmt)
    windows = sorted({1, 7, 16, 17, max(S, 1), S + 1, S + 15, S + 16, S + 33, 100, N + S - 1, N + S, 10 ** 6})
    for W in windows:
        if S:
            O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs), fa_window=W)
        else:
            O, L = ctx.query(sid, 0, dev(Q), fa_window=W)
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs, window=W)
        ctx.sync()
        assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"window {W} {shape}")
    ctx.drop(sid)


def test_window_rejections(ctx):
    from prefix_cached_kv_gb300 import binding
    K, V = synth.gen_kv(3, 2, 200, 64)
    ctx.store("wr", 0, dev(K), dev(V))
    with pytest.raises(binding.PckError) as e:
        ctx.query("wr", 0, dev(synth.gen_q(3, 4, 1, 64)), fa_window=-1)
    assert e.value.code == binding.EINVAL
    with pytest.raises(binding.PckError) as e:
        ctx.query_sparse_auto("wr", 0, dev(synth.gen_q(3, 4, 1, 64)[:, 0]), 64, 2, 2, fa_window=16)
    assert e.value.code == binding.EUNSUPPORTED
    ctx.drop("wr")


@pytest.mark.parametrize("H_q,H_kv,N,M,S,D,fmt,causal", [
    (4, 2, 1000, 130, 40, 64, 0, True),      # rows span several row tiles; windows end in the suffix
    (6, 2, 700, 64, 64, 128, 0, True),
    (3, 1, 4133, 16, 8, 128, 0, True),       # many key-range splits: whole splits before a row's window
    (4, 2, 900, 96, 32, 64, 1, True),        # mlx4g32 slot (hi/lo pairs at width 2D)
    (2, 2, 500, 40, 24, 96, 0, False),       # no causal bound: the window alone
])
def test_prefill_window_matches_oracle(ctx, H_q, H_kv, N, M, S, D, fmt, causal):
    """fa_window at M > 1: row i sees positions p_i - W + 1 .. p_i (p_i = N + S - M + i), under the
    causal bound when set; windows inside the suffix, across the prefix / suffix border, deep in
    the prefix, wider than everything, and W = 1."""
    seed = N + M + S + D + fmt
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, M, D, dtype=np.float16)
    Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
    hm = synth.default_head_map(H_q, H_kv)
    Ko, Vo = _oracle_kv(K, V, fmt)
    sid = f"pw{seed}"
    ctx.store(sid, 0, dev(K), dev(V), fmt=fmt)
    for W in sorted({1, 17, S, S + 70, M + S, 300, N + S + 5}):
        O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs), causal=causal, fa_window=W)
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs, causal=causal, window=W)
        ctx.sync()
        assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"prefill window {W} {(H_q, H_kv, N, M, S, D, fmt, causal)}")
    ctx.drop(sid)


def test_prefill_window_without_suffix(ctx):
    H_q, H_kv, N, M, D = 4, 2, 1500, 200, 128
    K, V = synth.gen_kv(77, H_kv, N, D)
    Q = synth.gen_q(77, H_q, M, D, dtype=np.float16)
    hm = synth.default_head_map(H_q, H_kv)
    ctx.store("pwn", 0, dev(K), dev(V))
    for W in (1, 64, 250, 10 ** 6):
        O, L = ctx.query("pwn", 0, dev(Q), fa_window=W)
        O_ref, L_ref = orc.prefix_query(Q, K, V, hm, window=W)
        ctx.sync()
        assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"prefill window {W}, no suffix")
    ctx.drop("pwn")
