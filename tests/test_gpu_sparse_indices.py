"""ATTEND.PREFIX.QUERY_SPARSE (caller-supplied per-head token indices) on the GPU vs the oracle,
and its host-side rejection of malformed index lists before anything is launched."""
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


def _lists(seed, H_q, N, K_max, min_count=1):
    """Seeded per-head sorted distinct token positions, counts between min_count and K_max."""
    rng = np.random.default_rng(seed)
    idx = np.zeros((H_q, K_max), dtype=np.int32)
    cnt = rng.integers(min_count, K_max + 1, size=H_q).astype(np.int32)
    for h in range(H_q):
        idx[h, :cnt[h]] = np.sort(rng.choice(N, size=int(cnt[h]), replace=False))
        idx[h, cnt[h]:] = -7   # entries past the count are never read
    return idx, cnt


@pytest.mark.parametrize("H_q,H_kv,N,D,K_max,q16,hm", [
    (8, 8, 2048, 128, 256, False, None),      # one q head per kv head, as the wire form
    (8, 2, 3000, 128, 300, False, None),      # GQA: q heads of one kv head pick different tokens
    (6, 3, 1000, 64, 40, True, [2, 0, 1, 1, 0, 2]),
    (4, 1, 700, 256, 97, False, None),
    (3, 1, 50, 64, 1, False, None),           # a single token each
    (2, 2, 17, 64, 17, True, None),           # every token of a ragged prefix
    (4, 2, 900, 512, 130, False, None),       # the widest head dim
    (3, 1, 300, 96, 33, True, None),
])
def test_query_sparse_matches_oracle(ctx, H_q, H_kv, N, D, K_max, q16, hm):
    K, V = synth.gen_kv(N + D, H_kv, N, D)
    Q = synth.gen_q(N + D, H_q, 1, D, dtype=np.float16 if q16 else np.float32)[:, 0]
    idx, cnt = _lists(N + K_max, H_q, N, K_max)
    if K_max == N:
        cnt[:] = N
        idx[:] = np.arange(N)
    hmap = None if hm is None else np.array(hm, dtype=np.int32)
    sid = f"qs{N}{D}"
    ctx.store(sid, 0, dev(K), dev(V))
    O, L = ctx.query_sparse(sid, 0, dev(Q), idx, cnt, head_map=hmap)
    O_ref, L_ref = orc.sparse_query_indices(Q, K, V, idx, cnt, hmap)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, f"query_sparse {(H_q, H_kv, N, D, K_max)}")
    ctx.drop(sid)


def test_query_sparse_of_selected_blocks_equals_auto(ctx):
    """The tokens of the blocks the auto selector picked, given as indices: the same answer."""
    H_q, H_kv, N, D, B, Kt = 8, 2, 4096, 128, 64, 6
    K, V = synth.gen_kv(3, H_kv, N, D)
    Q = synth.gen_q(3, H_q, 1, D)[:, 0]
    ctx.store("qsa", 0, dev(K), dev(V))
    Oa, La, sel = ctx.query_sparse_auto("qsa", 0, dev(Q), B, Kt, H_kv)
    sel = host(sel)
    idx = np.stack([np.concatenate([np.arange(b * B, (b + 1) * B) for b in sel[h]]) for h in range(H_q)]).astype(np.int32)
    O, L = ctx.query_sparse("qsa", 0, dev(Q), idx, np.full(H_q, Kt * B, dtype=np.int32))
    ctx.sync()
    assert np.abs(host(O) - host(Oa)).max() <= 1e-5 and np.abs(host(L) - host(La)).max() <= 1e-5
    ctx.drop("qsa")


def test_query_sparse_stress_dominant_key(ctx):
    H_q, H_kv, N, D = 8, 2, 1000, 128
    Q, K, V, _, _ = synth.gen_stress("dominant_prefix", 4, H_q, H_kv, N, D)
    Q = Q[:, 0]
    idx, cnt = _lists(5, H_q, N, 200, min_count=50)
    ctx.store("qsd", 0, dev(K), dev(V))
    O, L = ctx.query_sparse("qsd", 0, dev(Q), idx, cnt)
    O_ref, L_ref = orc.sparse_query_indices(Q, K, V, idx, cnt)
    ctx.sync()
    assert_close_o_lse(host(O), host(L), O_ref, L_ref, "query_sparse dominant")
    ctx.drop("qsd")


def test_query_sparse_rejects_malformed_lists(ctx):
    from prefix_cached_kv_gb300 import binding
    H_q, H_kv, N, D = 2, 2, 100, 64
    K, V = synth.gen_kv(8, H_kv, N, D)
    ctx.store("qsr", 0, dev(K), dev(V))
    Q = dev(synth.gen_q(8, H_q, 1, D)[:, 0])
    good = np.array([[1, 5, 9], [0, 2, 99]], dtype=np.int32)
    cnt = np.array([3, 3], dtype=np.int32)
    bad_cases = [
        (np.array([[1, 9, 5], [0, 2, 99]]), cnt),       # unsorted
        (np.array([[1, 5, 5], [0, 2, 99]]), cnt),       # duplicate
        (np.array([[1, 5, 9], [0, 2, 100]]), cnt),      # past the prefix
        (np.array([[-1, 5, 9], [0, 2, 99]]), cnt),      # negative
        (good, np.array([0, 3])),                        # empty list
        (good, np.array([3, 4])),                        # count above K_sparse_max
    ]
    for idx, c in bad_cases:
        with pytest.raises(binding.PckError) as e:
            ctx.query_sparse("qsr", 0, Q, idx, c)
        assert e.value.code == binding.EINVAL, (idx, c)
    O, L = ctx.query_sparse("qsr", 0, Q, good, cnt)
    ctx.sync()
    assert np.isfinite(host(O)).all()
    ctx.drop("qsr")
