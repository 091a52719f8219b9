"""M=1 prefix attention (split-K decode) on the GPU vs the oracle, fp16 and mlx4g32 slots,
with GQA, a fused dense suffix, ragged tails, batched launches and the full-size workloads."""
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
    """What the oracle attends to: fp16 values, or the dequantised mlx4g32 codes of them."""
    if fmt == 0:
        return K.astype(np.float64), V.astype(np.float64)
    H, N, D = K.shape
    outs = []
    for X in (K, V):
        c, s, b = orc.quantize_mlx4g32(X.reshape(H * N, D))
        outs.append(orc.dequantize_mlx4g32(c, s, b).reshape(H, N, D))
    return outs


CASES = [
    # H_q, H_kv, N, D, S_suf, fmt
    (8, 8, 2048, 128, 0, 0),        # the single-layer M=1 workload
    (32, 8, 1000, 64, 16, 1),
    (32, 8, 1000, 64, 16, 0),
    (4, 1, 17, 256, 0, 0),
    (4, 1, 17, 256, 5, 1),
    (6, 3, 1, 64, 0, 0),            # N = 1
    (6, 3, 1, 64, 0, 1),
    (16, 2, 333, 128, 33, 1),       # GQA 8
    (16, 2, 333, 128, 33, 0),       # GQA 8, fp16 (two 4-head column blocks)
    (16, 2, 600, 256, 20, 0),       # GQA 8, fp16, D = 256
    (24, 2, 100, 64, 1, 0),         # GQA 12 -> two work groups per kv head
    (1, 1, 4097, 64, 0, 1),
]


@pytest.mark.parametrize("H_q,H_kv,N,D,S,fmt", CASES)
@pytest.mark.parametrize("q16", [False, True])
def test_decode_matches_oracle(ctx, H_q, H_kv, N, D, S, fmt, q16):
    seed = H_q * 7 + N + D + S + fmt
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, 1, D, dtype=np.float16 if q16 else np.float32)
    hm = synth.default_head_map(H_q, H_kv)
    sid = f"d{seed}"
    ctx.store(sid, 0, dev(K), dev(V), fmt=fmt)
    Ko, Vo = _oracle_kv(K, V, fmt)
    if S:
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        O, L = ctx.query_fused(sid, 0, dev(Q), dev(Ks), dev(Vs), causal=True)
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs)
    else:
        O, L = ctx.query(sid, 0, dev(Q))
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"{(H_q, H_kv, N, D, S, fmt, q16)}")
    ctx.drop(sid)


def test_custom_head_map(ctx):
    H_q, H_kv, N, D = 6, 3, 200, 64
    K, V = synth.gen_kv(11, H_kv, N, D)
    Q = synth.gen_q(11, H_q, 1, D)
    hm = np.array([2, 0, 1, 1, 0, 2], dtype=np.int32)
    for fmt in (0, 1):
        ctx.store("hm", fmt, dev(K), dev(V), fmt=fmt)
        O, L = ctx.query("hm", fmt, dev(Q), head_map=hm)
        Ko, Vo = _oracle_kv(K, V, fmt)
        O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, hm)
        assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"head_map fmt={fmt}")


def test_store_records_equals_store(ctx):
    """A slot stored from token-major mlx4g32 records (computed by the oracle) answers like
    the slot the library quantised itself."""
    H_q, H_kv, N, D = 16, 4, 300, 128
    K, V = synth.gen_kv(12, H_kv, N, D)
    Q = synth.gen_q(12, H_q, 1, D)
    tok = lambda X: X.transpose(1, 0, 2).reshape(N, H_kv * D)
    Krec, Vrec = orc.quantize_records(tok(K)), orc.quantize_records(tok(V))
    ctx.store_records("rec", 0, H_kv, N, D, dev(Krec), dev(Vrec))
    ctx.store("rec", 1, dev(K), dev(V), fmt=1)
    O0, L0 = ctx.query("rec", 0, dev(Q))
    O1, L1 = ctx.query("rec", 1, dev(Q))
    Ko = orc.records_to_heads(Krec, H_kv, D)
    Vo = orc.records_to_heads(Vrec, H_kv, D)
    O_ref, L_ref = orc.prefix_query(Q, Ko, Vo, synth.default_head_map(H_q, H_kv))
    assert_close_o_lse(host(O0), host(L0), O_ref, L_ref, "store_records")
    assert np.array_equal(host(O0), host(O1)) and np.array_equal(host(L0), host(L1))


def test_deterministic(ctx):
    K, V = synth.gen_kv(13, 8, 5000, 64)
    Q = synth.gen_q(13, 32, 1, 64)
    Ks, Vs = synth.gen_suffix(13, 8, 16, 64)
    ctx.store("det", 0, dev(K), dev(V), fmt=1)
    a = [host(t) for t in ctx.query_fused("det", 0, dev(Q), dev(Ks), dev(Vs))]
    b = [host(t) for t in ctx.query_fused("det", 0, dev(Q), dev(Ks), dev(Vs))]
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gqa_decode_workload_full(ctx):
    """16 layers, H_q=32, H_kv=8, D=64, N=8192, mlx4g32, S_suf=16: every output vs the oracle,
    through per-layer fused queries and through one batched launch."""
    w = synth.WORKLOADS["gqa_decode_mlx4g32"]
    H_q, H_kv, N, D, S, L = w["H_q"], w["H_kv"], w["N"], w["D"], w["S_suf"], w["layers"]
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs, singles = [], [], []
    for layer in range(L):
        K, V = synth.gen_kv(0, H_kv, N, D, layer=layer)
        Q = synth.gen_q(0, H_q, 1, D, layer=layer)
        Ks, Vs = synth.gen_suffix(0, H_kv, S, D, layer=layer)
        ctx.store("cfg2", layer, dev(K), dev(V), fmt=1)
        Ko, Vo = _oracle_kv(K, V, 1)
        refs.append(orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs))
        Qd, Ksd, Vsd = dev(Q[:, 0]), dev(Ks), dev(Vs)
        O = torch.empty((H_q, D), device="cuda")
        Ld = torch.empty((H_q,), device="cuda")
        descs.append(dict(sid="cfg2", layer=layer, Q=Qd, O=O, LSE=Ld, K_suf=Ksd, V_suf=Vsd))
        singles.append(ctx.query_fused("cfg2", layer, Qd[:, None, :], Ksd, Vsd))
    ctx.query_batch(descs, H_q, H_kv, D, S_suf=S)
    ctx.sync()
    for layer in range(L):
        O_ref, L_ref = refs[layer]
        assert_close_o_lse(host(descs[layer]["O"]), host(descs[layer]["LSE"]), O_ref[:, 0], L_ref[:, 0], f"batch {layer}")
        assert_close_o_lse(host(singles[layer][0]), host(singles[layer][1]), O_ref, L_ref, f"single {layer}")
    for layer in range(L):
        ctx.drop("cfg2", layer)


def test_cartridge_attend_sampled(ctx):
    """Cartridge workload: 64 sessions, each an M=1 GQA query (H_q=32, H_kv=8, D=128) over its own
    8192-token window of a layer of an 86,580-token, 36-layer cartridge stored as mlx4g32. The
    layers needed are generated on the device (N(0,1) fp16), quantised by the library and stored
    per window; a seeded sample of sessions is checked against the oracle, which quantises the
    same fp16 windows itself."""
    w = synth.WORKLOADS["cartridge_mlx4g32"]
    H_q, H_kv, N, D, W, S = w["H_q"], w["H_kv"], w["N"], w["D"], w["window"], w["sessions"]
    hm = synth.default_head_map(H_q, H_kv)
    sample = sorted(set(np.random.default_rng(3).choice(S, size=3, replace=False).tolist()) | {0, S - 1})
    descs, kept = [], {}
    for layer in range(36):
        sess = [s for s in range(S) if s % 36 == layer]
        if not sess:
            continue
        K, V = synth.torch_gen_kv_device(0, H_kv, N, D, "cuda", layer=layer)
        for s in sess:
            o = synth.cartridge_window_start(s, N, W)
            Kw, Vw = K[:, o:o + W].contiguous(), V[:, o:o + W].contiguous()
            ctx.store(f"cart{s}", 0, Kw, Vw, fmt=1)
            Q = synth.gen_q(s, H_q, 1, D)[:, 0]
            Od = torch.empty((H_q, D), device="cuda")
            Ld = torch.empty((H_q,), device="cuda")
            descs.append(dict(sid=f"cart{s}", layer=0, Q=dev(Q), O=Od, LSE=Ld))
            if s in sample:
                kept[s] = (host(Kw), host(Vw), Q)
        del K, V
    descs.sort(key=lambda d: int(d["sid"][4:]))
    ctx.query_batch(descs, H_q, H_kv, D)
    ctx.sync()
    for s in sample:
        Kh, Vh, Q = kept[s]
        Ko, Vo = _oracle_kv(Kh, Vh, 1)
        O_ref, L_ref = orc.prefix_query(Q[:, None], Ko, Vo, hm)
        assert_close_o_lse(host(descs[s]["O"]), host(descs[s]["LSE"]), O_ref[:, 0], L_ref[:, 0], f"session {s}")
    for s in range(S):
        ctx.drop(f"cart{s}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_batch_suffix_computed_by_prefix_workers(ctx, fmt):
    """A batch large enough that every resident warp streams prefix tiles: the suffix pieces (three
    per item here, S_suf = 40) are computed by the prefix workers whose ranges hold the items'
    first tiles. Descriptors of different prefix lengths, GQA 4, against the oracle."""
    H_q, H_kv, D, S = 32, 8, 64, 40
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs = [], []
    for r, N in enumerate((6000, 8192, 4099, 7001, 5555, 8192, 6500, 3001)):
        K, V = synth.gen_kv(70 + r, H_kv, N, D)
        Q = synth.gen_q(70 + r, H_q, 1, D)
        Ks, Vs = synth.gen_suffix(70 + r, H_kv, S, D)
        ctx.store(f"fold{r}", 0, dev(K), dev(V), fmt=fmt)
        Ko, Vo = _oracle_kv(K, V, fmt)
        refs.append(orc.prefix_query(Q, Ko, Vo, hm, Ks, Vs))
        descs.append(dict(sid=f"fold{r}", layer=0, Q=dev(Q[:, 0]), O=torch.empty((H_q, D), device="cuda"),
                          LSE=torch.empty((H_q,), device="cuda"), K_suf=dev(Ks), V_suf=dev(Vs)))
    ctx.query_batch(descs, H_q, H_kv, D, S_suf=S)
    ctx.sync()
    for r, (O_ref, L_ref) in enumerate(refs):
        assert_close_o_lse(host(descs[r]["O"]), host(descs[r]["LSE"]), O_ref[:, 0], L_ref[:, 0], f"fold {fmt} {r}")
        ctx.drop(f"fold{r}")
