"""Block-mean top-K sparse attention on the GPU vs the oracle: selected blocks bit-exact (except
near-ties of the oracle's scores), outputs within tolerance."""
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


def _check_idx(idx, scores, K_top):
    ok_rows = orc.topk_margin(scores, K_top) >= TIE_EPS
    want = orc.select_top_blocks(scores, K_top)
    assert np.array_equal(idx[ok_rows], want[ok_rows])
    assert (np.diff(idx, axis=1) > 0).all()          # strictly ascending everywhere
    return want


@pytest.mark.parametrize("H_q,H_kv,N,D,B,K_top,S", [
    (8, 2, 1000, 64, 64, 3, 0),
    (8, 2, 1000, 64, 64, 3, 7),
    (4, 4, 777, 256, 32, 5, 16),
    (6, 2, 4096, 128, 64, 8, 32),
    (8, 1, 100, 64, 16, 2, 0),
    (8, 2, 4096, 64, 64, 40, 0),      # K_top > 32: arg-max rounds; union lists longer than 32
    (4, 1, 8192, 128, 64, 64, 16),    # the largest K_top
    (2, 1, 1, 64, 16, 1, 0),          # a one-token prefix: one block
    (12, 1, 2000, 64, 64, 4, 5),      # GQA 12: two work groups (two unions) on one kv head
])
def test_sparse_matches_oracle(ctx, H_q, H_kv, N, D, B, K_top, S):
    seed = N + D + K_top
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, 1, D)[:, 0]
    hm = synth.default_head_map(H_q, H_kv)
    sid = f"sp{seed}"
    ctx.store(sid, 0, dev(K), dev(V))
    Ks = Vs = None
    if S:
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
    O, L, idx = ctx.query_sparse_auto(sid, 0, dev(Q), B, K_top, H_kv, K_suf=dev(Ks) if S else None,
                                      V_suf=dev(Vs) if S else None)
    O_ref, L_ref, idx_ref, scores = orc.sparse_query(Q, K, V, hm, B, K_top, Ks, Vs)
    k_eff = min(K_top, (N + B - 1) // B)
    idx = host(idx).reshape(-1)[: H_q * k_eff].reshape(H_q, k_eff)
    _check_idx(idx, scores, K_top)
    near = orc.topk_margin(scores, K_top) < TIE_EPS
    assert_close_o_lse(host(O)[~near], host(L)[~near], O_ref[~near], L_ref[~near], "sparse")
    ctx.drop(sid)


def test_sparse_covering_all_blocks_equals_dense(ctx):
    H_q, H_kv, N, D, B = 8, 2, 300, 64, 64
    K, V = synth.gen_kv(21, H_kv, N, D)
    Q = synth.gen_q(21, H_q, 1, D)
    ctx.store("spall", 0, dev(K), dev(V))
    O, L, idx = ctx.query_sparse_auto("spall", 0, dev(Q[:, 0]), B, 5, H_kv)
    Od, Ld = ctx.query("spall", 0, dev(Q))
    assert (host(idx).reshape(-1)[: H_q * 5].reshape(H_q, 5) == np.arange(5)).all()
    O_ref, L_ref = orc.prefix_query(Q, K, V, synth.default_head_map(H_q, H_kv))
    assert_close_o_lse(host(O), host(L), O_ref[:, 0], L_ref[:, 0], "sparse-all")
    assert_close_o_lse(host(Od), host(Ld), O_ref, L_ref, "dense")


def test_sparse_needle_workload_full(ctx):
    """Sparse long-context workload: N=65,536, D=256, H_q=8, H_kv=2, B=64, K_top=8, S_suf=32, with
    eight seeded needle blocks pulled toward the query (+3 sigma along the GQA-group direction)."""
    w = synth.WORKLOADS["sparse_topk_64k"]
    H_q, H_kv, N, D, B, Kt, S = w["H_q"], w["H_kv"], w["N"], w["D"], w["B"], w["K_top"], w["S_suf"]
    K, V = synth.gen_kv(0, H_kv, N, D)
    Q = synth.gen_q(0, H_q, 1, D)[:, 0]
    hm = synth.default_head_map(H_q, H_kv)
    needles = synth.needle_blocks(0, N // B, Kt)
    K = synth.plant_needles(K, Q, hm, needles, B)
    Ks, Vs = synth.gen_suffix(0, H_kv, S, D)
    ctx.store("needle", 0, dev(K), dev(V))
    O, L, idx = ctx.query_sparse_auto("needle", 0, dev(Q), B, Kt, H_kv, K_suf=dev(Ks), V_suf=dev(Vs))
    O_ref, L_ref, idx_ref, scores = orc.sparse_query(Q, K, V, hm, B, Kt, Ks, Vs)
    idx = host(idx)
    assert (idx_ref == needles[None]).all()
    assert np.array_equal(idx, idx_ref)
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, "needle")
    ctx.drop("needle")


def test_sparse_exact_ties_pick_lowest_indices(ctx):
    """Every block has the same mean (K is the same vector at every token, so the block means are
    bit-identical), so every score ties: each head must select blocks 0..K_top-1 (ties go to the
    lower block index), and attend uniformly over their tokens."""
    H_q, H_kv, N, D, B, Kt = 4, 1, 4096, 64, 64, 8
    rng = np.random.default_rng(5)
    row = rng.standard_normal(D).astype(np.float16)
    K = np.broadcast_to(row, (H_kv, N, D)).copy()
    _, V = synth.gen_kv(5, H_kv, N, D)
    Q = synth.gen_q(5, H_q, 1, D)[:, 0]
    hm = synth.default_head_map(H_q, H_kv)
    ctx.store("ties", 0, dev(K), dev(V))
    O, L, idx = ctx.query_sparse_auto("ties", 0, dev(Q), B, Kt, H_kv)
    idx = host(idx).reshape(-1)[: H_q * Kt].reshape(H_q, Kt)
    assert (idx == np.arange(Kt)[None]).all()
    O_ref, L_ref, idx_ref, _ = orc.sparse_query(Q, K, V, hm, B, Kt)
    assert (idx_ref == np.arange(Kt)[None]).all()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, "sparse-ties")
    ctx.drop("ties")


def test_sparse_more_blocks_than_registers(ctx):
    """2500 blocks per head (more than the selector keeps in registers): scores read from memory."""
    H_q, H_kv, N, D, B, Kt = 4, 2, 40000, 64, 16, 6
    K, V = synth.gen_kv(77, H_kv, N, D)
    Q = synth.gen_q(77, H_q, 1, D)[:, 0]
    hm = synth.default_head_map(H_q, H_kv)
    ctx.store("manyb", 0, dev(K), dev(V))
    O, L, idx = ctx.query_sparse_auto("manyb", 0, dev(Q), B, Kt, H_kv)
    O_ref, L_ref, idx_ref, scores = orc.sparse_query(Q, K, V, hm, B, Kt)
    idx = host(idx).reshape(-1)[: H_q * Kt].reshape(H_q, Kt)
    _check_idx(idx, scores, Kt)
    near = orc.topk_margin(scores, Kt) < TIE_EPS
    assert_close_o_lse(host(O)[~near], host(L)[~near], O_ref[~near], L_ref[~near], "sparse-many")
    ctx.drop("manyb")


def test_sparse_batch_matches_single_calls_and_oracle(ctx):
    """pck_query_sparse_batch over 3 sessions (own data, own suffix): every query selects what its
    own single call selects, and its outputs match the oracle."""
    H_q, H_kv, N, D, B, Kt, S = 8, 2, 3000, 128, 64, 5, 24
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs, singles = [], [], []
    for r in range(3):
        seed = 300 + r
        K, V = synth.gen_kv(seed, H_kv, N, D)
        Q = synth.gen_q(seed, H_q, 1, D)[:, 0]
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        sid = f"spb{r}"
        ctx.store(sid, 0, dev(K), dev(V))
        O1, L1, i1 = ctx.query_sparse_auto(sid, 0, dev(Q), B, Kt, H_kv, K_suf=dev(Ks), V_suf=dev(Vs))
        singles.append(host(i1).reshape(-1)[: H_q * Kt].reshape(H_q, Kt))
        d = dict(sid=sid, layer=0, Q=dev(Q), O=torch.empty((H_q, D), device="cuda"),
                 LSE=torch.empty((H_q,), device="cuda"), K_suf=dev(Ks), V_suf=dev(Vs),
                 idx=torch.empty((H_q, Kt), dtype=torch.int32, device="cuda"))
        descs.append(d)
        refs.append(orc.sparse_query(Q, K, V, hm, B, Kt, Ks, Vs))
    ctx.query_sparse_batch(descs, H_q, H_kv, D, B, Kt, S_suf=S)
    ctx.sync()
    for r, (d, (O_ref, L_ref, idx_ref, scores)) in enumerate(zip(descs, refs)):
        idx = host(d["idx"])
        assert np.array_equal(idx, singles[r])
        _check_idx(idx, scores, Kt)
        near = orc.topk_margin(scores, Kt) < TIE_EPS
        assert_close_o_lse(host(d["O"])[~near], host(d["LSE"])[~near], O_ref[~near], L_ref[~near], f"batch {r}")
    for r in range(3):
        ctx.drop(f"spb{r}")


def test_sparse_batch_rejects_slots_of_different_lengths(ctx):
    from prefix_cached_kv_gb300 import binding
    H_q, H_kv, D = 4, 1, 64
    descs = []
    for r, N in enumerate((512, 640)):
        K, V = synth.gen_kv(r, H_kv, N, D)
        ctx.store(f"spn{r}", 0, dev(K), dev(V))
        descs.append(dict(sid=f"spn{r}", layer=0, Q=dev(synth.gen_q(r, H_q, 1, D)[:, 0]),
                          O=torch.empty((H_q, D), device="cuda")))
    with pytest.raises(binding.PckError) as e:
        ctx.query_sparse_batch(descs, H_q, H_kv, D, 64, 2)
    assert e.value.code == binding.EUNSUPPORTED
    for r in range(2):
        ctx.drop(f"spn{r}")


def test_sparse_batch_many_sessions_uneven_items(ctx):
    """24 sessions x 2 kv heads = 48 work items (more than one 32-item window): the device-side
    split of the selected tiles over the workers (a 32-way search over the items' unit offsets,
    then a window of them per worker), with a ragged last block and a suffix, against the oracle
    per session."""
    H_q, H_kv, N, D, B, Kt, S = 8, 2, 1500, 64, 64, 4, 8
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs = [], []
    for r in range(24):
        seed = 900 + r
        K, V = synth.gen_kv(seed, H_kv, N, D)
        Q = synth.gen_q(seed, H_q, 1, D)[:, 0]
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        sid = f"spm{r}"
        ctx.store(sid, 0, dev(K), dev(V))
        descs.append(dict(sid=sid, layer=0, Q=dev(Q), O=torch.empty((H_q, D), device="cuda"),
                          LSE=torch.empty((H_q,), device="cuda"), K_suf=dev(Ks), V_suf=dev(Vs),
                          idx=torch.empty((H_q, Kt), dtype=torch.int32, device="cuda")))
        refs.append(orc.sparse_query(Q, K, V, hm, B, Kt, Ks, Vs))
    for _ in range(2):   # twice: the launch-to-launch counters must come back to zero
        ctx.query_sparse_batch(descs, H_q, H_kv, D, B, Kt, S_suf=S)
        ctx.sync()
        for r, (d, (O_ref, L_ref, idx_ref, scores)) in enumerate(zip(descs, refs)):
            _check_idx(host(d["idx"]), scores, Kt)
            near = orc.topk_margin(scores, Kt) < TIE_EPS
            assert_close_o_lse(host(d["O"])[~near], host(d["LSE"])[~near], O_ref[~near], L_ref[~near], f"session {r}")
    for r in range(24):
        ctx.drop(f"spm{r}")


def test_sparse_batch_in_a_cuda_graph(ctx):
    """A batch of 9 sessions captured in a CUDA graph and replayed twice: the selector's
    completion counter comes back to zero between replays, and every session matches the oracle
    after each replay."""
    H_q, H_kv, N, D, B, Kt, S = 4, 2, 2000, 128, 64, 3, 16
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs = [], []
    for r in range(9):
        seed = 700 + r
        K, V = synth.gen_kv(seed, H_kv, N, D)
        Q = synth.gen_q(seed, H_q, 1, D)[:, 0]
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        sid = f"sph{r}"
        ctx.store(sid, 0, dev(K), dev(V))
        ctx.build_block_means(sid, 0, B)
        descs.append(dict(sid=sid, layer=0, Q=dev(Q), O=torch.empty((H_q, D), device="cuda"),
                          LSE=torch.empty((H_q,), device="cuda"), K_suf=dev(Ks), V_suf=dev(Vs),
                          idx=torch.empty((H_q, Kt), dtype=torch.int32, device="cuda")))
        refs.append(orc.sparse_query(Q, K, V, hm, B, Kt, Ks, Vs))
    call = ctx.sparse_batch_caller(descs, H_q, H_kv, D, B, Kt, S_suf=S)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=st):
        call()
    torch.cuda.current_stream().wait_stream(st)
    for _ in range(2):
        for d in descs:
            d["O"].fill_(float("nan"))
            d["idx"].fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        ctx.sync()
        for r, (d, (O_ref, L_ref, idx_ref, scores)) in enumerate(zip(descs, refs)):
            _check_idx(host(d["idx"]), scores, Kt)
            near = orc.topk_margin(scores, Kt) < TIE_EPS
            assert_close_o_lse(host(d["O"])[~near], host(d["LSE"])[~near], O_ref[~near], L_ref[~near], f"graph {r}")
    del g
    for r in range(9):
        ctx.drop(f"sph{r}")


def test_block_means_arena_reuse(ctx):
    """The block means live in the context's arena: a dropped slot's means are reused by a later
    slot (after the drop's stream work), a replaced slot gets fresh means, and the slots that stay
    keep theirs. Every query is checked against the oracle."""
    H_q, H_kv, N, D, B, Kt, S = 4, 2, 3000, 128, 64, 4, 8
    hm = synth.default_head_map(H_q, H_kv)

    def put(sid, seed):
        K, V = synth.gen_kv(seed, H_kv, N, D)
        ctx.store(sid, 0, dev(K), dev(V))
        ctx.build_block_means(sid, 0, B)
        return K, V

    def check(sid, seed, K, V):
        Q = synth.gen_q(seed, H_q, 1, D)[:, 0]
        Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        O, L, idx = ctx.query_sparse_auto(sid, 0, dev(Q), B, Kt, H_kv, K_suf=dev(Ks), V_suf=dev(Vs))
        O_ref, L_ref, _, scores = orc.sparse_query(Q, K, V, hm, B, Kt, Ks, Vs)
        _check_idx(host(idx), scores, Kt)
        near = orc.topk_margin(scores, Kt) < TIE_EPS
        assert_close_o_lse(host(O)[~near], host(L)[~near], O_ref[~near], L_ref[~near], sid)

    kv = {r: put(f"ar{r}", 900 + r) for r in range(3)}
    ctx.drop("ar1")
    torch.cuda.synchronize()
    kv[3] = put("ar3", 903)                       # takes the range ar1 freed
    kv[0] = put("ar0", 910)                       # replaced: old means freed, new ones built
    for r, seed in ((0, 910), (2, 902), (3, 903)):
        check(f"ar{r}", seed, *kv[r])
    for r in (0, 2, 3):
        ctx.drop(f"ar{r}")


def test_block_means_not_built_during_capture(ctx):
    """A sparse call whose block means are missing cannot build them while its stream is being
    captured: it returns PCK_EINVAL before launching anything, and works once they are built."""
    from prefix_cached_kv_gb300 import binding
    H_q, H_kv, N, D, B, Kt = 4, 2, 1000, 64, 64, 2
    K, V = synth.gen_kv(950, H_kv, N, D)
    Q = dev(synth.gen_q(950, H_q, 1, D)[:, 0])
    ctx.store("cap", 0, dev(K), dev(V))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        g.capture_begin()
        try:
            with pytest.raises(binding.PckError) as e:
                ctx.query_sparse_auto("cap", 0, Q, B, Kt, H_kv)
        finally:
            g.capture_end()
    assert e.value.code == binding.EINVAL
    del g
    ctx.build_block_means("cap", 0, B)
    O, L, idx = ctx.query_sparse_auto("cap", 0, Q, B, Kt, H_kv)
    O_ref, L_ref, _, scores = orc.sparse_query(host(Q), K, V, synth.default_head_map(H_q, H_kv), B, Kt)
    near = orc.topk_margin(scores, Kt) < TIE_EPS
    assert_close_o_lse(host(O)[~near], host(L)[~near], O_ref[~near], L_ref[~near], "after capture")
    ctx.drop("cap")


@pytest.mark.parametrize("H_q,H_kv,hm", [
    (6, 3, [2, 0, 1, 1, 0, 2]),         # q heads of a kv head not adjacent
    (4, 2, [1, 1, 1, 1]),               # kv head 0 has no q heads: nothing scored or selected there
])
def test_sparse_custom_head_map(ctx, H_q, H_kv, hm):
    N, D, B, K_top, S = 1500, 128, 64, 4, 9
    hm = np.array(hm, dtype=np.int32)
    K, V = synth.gen_kv(23, H_kv, N, D)
    Q = synth.gen_q(23, H_q, 1, D)[:, 0]
    Ks, Vs = synth.gen_suffix(23, H_kv, S, D)
    ctx.store("sphm", 0, dev(K), dev(V))
    O, L, idx = ctx.query_sparse_auto("sphm", 0, dev(Q), B, K_top, H_kv, head_map=hm, K_suf=dev(Ks), V_suf=dev(Vs))
    O_ref, L_ref, idx_ref, scores = orc.sparse_query(Q, K, V, hm, B, K_top, Ks, Vs)
    idx = host(idx).reshape(-1)[: H_q * K_top].reshape(H_q, K_top)
    _check_idx(idx, scores, K_top)
    near = orc.topk_margin(scores, K_top) < TIE_EPS
    assert_close_o_lse(host(O)[~near], host(L)[~near], O_ref[~near], L_ref[~near], f"sparse head_map {hm.tolist()}")
    ctx.drop("sphm")


@pytest.mark.parametrize("H_kv,N,D,B", [(2, 1000, 64, 64), (1, 777, 256, 32), (4, 4096, 128, 16), (1, 5, 64, 16)])
def test_block_means_direct(ctx, H_kv, N, D, B):
    """The slot's block means against the oracle's, value by value (the last block partial)."""
    K, V = synth.gen_kv(N + B, H_kv, N, D)
    ctx.store("bm", 0, dev(K), dev(V))
    got = host(ctx.get_block_means("bm", 0, B, H_kv, N, D))
    want = orc.block_means(K, B)
    assert got.shape == want.shape
    assert np.abs(got - want).max() <= 1e-5
    ctx.drop("bm")


# ---------------------------------------------------------------- the fused single-kernel form
# pck_query_sparse_batch runs the whole query in one kernel (a CTA per (session, group of q
# heads)) once a batch has at least 32 work items and every kv head has at most 1024 blocks;
# these batches are sized to take that path.

FUSED_CASES = [
    # H_q, H_kv, head_map, N, D, B, K_top, S_suf, q fp16, sessions
    (8, 2, None, 3000, 256, 64, 5, 24, False, 16),           # ragged last block, short last suffix tile
    (16, 2, None, 2000, 128, 32, 40, 0, True, 16),           # 8 q heads per group, K_top > 32 (arg-max rounds)
    (6, 3, [2, 0, 1, 1, 0, 2], 1500, 64, 64, 4, 9, False, 12),   # q heads of a kv head not adjacent
    (4, 2, [1, 1, 1, 1], 777, 128, 16, 64, 16, False, 32),   # kv head 0 has no q heads; K_top = 64 > nb
    (8, 1, None, 1100, 256, 64, 3, 32, True, 32),            # 8 q heads of one kv head at D = 256: two groups of 4
]


@pytest.mark.parametrize("H_q,H_kv,hm,N,D,B,Kt,S,q16,R", FUSED_CASES)
def test_sparse_fused_batch_matches_oracle(ctx, H_q, H_kv, hm, N, D, B, Kt, S, q16, R):
    hm = synth.default_head_map(H_q, H_kv) if hm is None else np.array(hm, dtype=np.int32)
    nb = -(-N // B)
    K_eff = min(Kt, nb)
    descs, refs = [], []
    for r in range(R):
        seed = 5000 + 17 * r + D
        K, V = synth.gen_kv(seed, H_kv, N, D)
        Q = synth.gen_q(seed, H_q, 1, D, dtype=np.float16 if q16 else np.float32)[:, 0]
        Ks = Vs = None
        if S:
            Ks, Vs = synth.gen_suffix(seed, H_kv, S, D)
        sid = f"spf{r}"
        ctx.store(sid, 0, dev(K), dev(V))
        d = dict(sid=sid, layer=0, Q=dev(Q), O=torch.full((H_q, D), float("nan"), device="cuda"),
                 LSE=torch.empty((H_q,), device="cuda"), idx=torch.full((H_q, K_eff), -1, dtype=torch.int32, device="cuda"))
        if S:
            d["K_suf"], d["V_suf"] = dev(Ks), dev(Vs)
        descs.append(d)
        refs.append(orc.sparse_query(Q, K, V, hm, B, Kt, Ks, Vs))
    ctx.query_sparse_batch(descs, H_q, H_kv, D, B, Kt, S_suf=S, q_dtype=binding_dt(q16), head_map=hm)
    ctx.sync()
    for r, (d, (O_ref, L_ref, idx_ref, scores)) in enumerate(zip(descs, refs)):
        _check_idx(host(d["idx"]), scores, K_eff)
        near = orc.topk_margin(scores, K_eff) < TIE_EPS
        assert_close_o_lse(host(d["O"])[~near], host(d["LSE"])[~near], O_ref[~near], L_ref[~near],
                           f"fused session {r} {(H_q, H_kv, N, D, B, Kt, S)}")
    for r in range(R):
        ctx.drop(f"spf{r}")


def test_sparse_fused_batch_exact_ties(ctx):
    """Bit-identical block means in every session (every score ties) through the fused form:
    each head selects blocks 0..K_top-1 and attends uniformly over their tokens."""
    H_q, H_kv, N, D, B, Kt, R = 4, 2, 2048, 64, 64, 6, 16
    rng = np.random.default_rng(9)
    row = rng.standard_normal(D).astype(np.float16)
    K = np.broadcast_to(row, (H_kv, N, D)).copy()
    hm = synth.default_head_map(H_q, H_kv)
    descs, refs = [], []
    for r in range(R):
        _, V = synth.gen_kv(60 + r, H_kv, N, D)
        Q = synth.gen_q(60 + r, H_q, 1, D)[:, 0]
        ctx.store(f"spt{r}", 0, dev(K), dev(V))
        descs.append(dict(sid=f"spt{r}", layer=0, Q=dev(Q), O=torch.empty((H_q, D), device="cuda"),
                          LSE=torch.empty((H_q,), device="cuda"), idx=torch.empty((H_q, Kt), dtype=torch.int32, device="cuda")))
        refs.append(orc.sparse_query(Q, K, V, hm, B, Kt))
    ctx.query_sparse_batch(descs, H_q, H_kv, D, B, Kt)
    ctx.sync()
    for r, (d, (O_ref, L_ref, idx_ref, scores)) in enumerate(zip(descs, refs)):
        assert (host(d["idx"]) == np.arange(Kt)[None]).all()
        assert_close_o_lse(host(d["O"]), host(d["LSE"]), O_ref, L_ref, f"ties session {r}")
    for r in range(R):
        ctx.drop(f"spt{r}")


def binding_dt(q16):
    from prefix_cached_kv_gb300 import binding
    return binding.DT_F16 if q16 else binding.DT_F32
