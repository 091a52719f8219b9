"""Pins of the CPU oracle against facts fixed by the pages and by the mathematics.

Each test checks the oracle against something other than its own formula: values the
pages print or a worked example built from the stated layout (tests/golden/), closed
forms, invariants, brute force with plain Python loops, and special cases that reduce
to a library routine (torch's CPU scaled_dot_product_attention, scipy's logsumexp).
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle import pck_oracle as orc
from prefix_cached_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


# ------------------------------------------------------------------ mlx4g32 layout

def test_layout_worked_example():
    lines = _golden_lines("mlx4g32_layout_example.txt")
    codes = np.array([int(v) for v in lines[0].split(":")[1].split()], dtype=np.uint8)[None, :]
    words = [int(v, 16) for v in lines[1].split(":")[1].split()]
    assert orc.pack_codes(codes)[0].tolist() == words
    assert np.array_equal(orc.unpack_codes(orc.pack_codes(codes), 32), codes)
    for ln in lines[2:]:
        kv = dict(p.split("=") for p in ln.split(":")[1].split())
        j, w, val = int(kv["j"]), int(kv["word"]), int(kv["value"], 16)
        c = np.zeros((1, 32), dtype=np.uint8)
        c[0, j] = 15
        packed = orc.pack_codes(c)[0]
        assert packed[w] == val and packed.sum() == val


def test_record_sizes_printed():
    for ln in _golden_lines("mlx4g32_record_sizes.txt"):
        kv = dict(p.split("=") for p in ln.split())
        d = int(kv["kv_dim"])
        assert orc.record_bytes(d) == int(kv["record_bytes"])
        assert 2 * d == int(kv["fp16_bytes"])
    assert round(2048 / orc.record_bytes(1024), 1) == 3.2


def test_record_byte_order():
    """Record = codes words, then all scales, then all biases, little-endian."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 64)).astype(np.float16)
    codes, s, b = orc.quantize_mlx4g32(x)
    rec = orc.pack_records(codes, s, b)
    assert rec.shape == (3, 40)
    for r in range(3):
        w0 = int(rec[r, 0]) | int(rec[r, 1]) << 8 | int(rec[r, 2]) << 16 | int(rec[r, 3]) << 24
        assert w0 & 0xF == codes[r, 0] and (w0 >> 28) & 0xF == codes[r, 7]
        assert rec[r, 32:34].tobytes() == s[r, 0].tobytes()
        assert rec[r, 34:36].tobytes() == s[r, 1].tobytes()
        assert rec[r, 36:38].tobytes() == b[r, 0].tobytes()
    c2, s2, b2 = orc.unpack_records(rec, 64)
    assert np.array_equal(c2, codes) and np.array_equal(s2, s) and np.array_equal(b2, b)


def test_records_to_heads_lossless_roundtrip():
    """Token-major records [N, H_kv*D] back to [H_kv, N, D]: on a lossless grid (scale 1/8, a bias
    of g + t/8 per kv head g and token t, codes (d + t) mod 16 so every group spans 0..15) every
    value names its own (g, t, d), so the round trip must return K exactly."""
    H_kv, N, D = 3, 5, 64
    g = np.arange(H_kv)[:, None, None]
    t = np.arange(N)[None, :, None]
    d = np.arange(D)[None, None, :]
    K = (g + t / 8.0 + ((d + t) % 16) / 8.0).astype(np.float16)
    assert np.array_equal(K.astype(np.float64), g + t / 8.0 + ((d + t) % 16) / 8.0)   # exact in fp16
    tok = K.transpose(1, 0, 2).reshape(N, H_kv * D)          # the pages' token-major row layout
    back = orc.records_to_heads(orc.quantize_records(tok), H_kv, D)
    assert back.shape == (H_kv, N, D)
    assert np.array_equal(back, K.astype(np.float64))


# ------------------------------------------------------------------ quantiser

def test_quantizer_lossless_on_grid():
    """A group already on an fp16 affine grid {b + k s} comes back exactly."""
    rng = np.random.default_rng(2)
    done = 0
    while done < 50:
        s = np.float16(2.0 ** rng.integers(-6, 2) * (1 + rng.integers(0, 64) / 64))
        b = np.float16(rng.integers(-64, 64) / 8)
        k = rng.integers(0, 16, size=32)
        k[0], k[1] = 0, 15
        x = (np.float64(b) + k * np.float64(s)).astype(np.float16)
        if not np.array_equal(x.astype(np.float64), np.float64(b) + k * np.float64(s)):
            continue  # this (s, b) grid is not exactly representable in fp16; draw again
        done += 1
        codes, sc, bi = orc.quantize_mlx4g32(x[None, :])
        assert sc[0, 0] == s and bi[0, 0] == b
        assert np.array_equal(codes[0], k)
        assert np.array_equal(orc.dequantize_mlx4g32(codes, sc, bi)[0], x.astype(np.float64))


def test_quantizer_constant_group():
    x = np.full((2, 64), np.float16(-1.375))
    x[1, 32:] = np.float16(7.0)
    codes, s, b = orc.quantize_mlx4g32(x)
    assert (codes == 0).all() and (s == 0).all()
    assert np.array_equal(orc.dequantize_mlx4g32(codes, s, b), x.astype(np.float64))


def test_quantizer_error_bound_and_monotone():
    """|x - x^| <= scale/2 (+ fp32 rounding), codes monotone in x, min -> 0 and max -> 15."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((200, 128)) * np.exp(rng.standard_normal((200, 1)))).astype(np.float16)
    codes, s, b = orc.quantize_mlx4g32(x)
    xh = orc.dequantize_mlx4g32(codes, s, b)
    smax = np.repeat(s.astype(np.float64), 32, axis=1)
    err = np.abs(xh - x.astype(np.float64))
    assert (err <= smax * 0.5 * (1 + 1e-6) + 1e-7 * np.abs(x.astype(np.float64))).all()
    xg = x.astype(np.float64).reshape(200, 4, 32)
    cg = codes.reshape(200, 4, 32)
    for r in range(200):
        for g in range(4):
            order = np.argsort(xg[r, g], kind="stable")
            assert (np.diff(cg[r, g][order].astype(int)) >= 0).all()
            assert cg[r, g][np.argmin(xg[r, g])] == 0 and cg[r, g][np.argmax(xg[r, g])] == 15


def test_quantizer_scale_is_fp16_roundtripped():
    """Each code is the nearest point of the grid the reader sees, {b16 + c * s16 : c in 0..15}.

    The page has the scale rounded to fp16 ahead of code selection; codes picked
    against the fp32 scale would miss the nearest reader-grid point for some elements, so the
    test also checks that such elements exist in the sample (the pin can fail)."""
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((400, 64)) * 3).astype(np.float16)
    codes, s, b = orc.quantize_mlx4g32(x)
    xg = x.astype(np.float64).reshape(400, 2, 32)
    grid = b.astype(np.float64)[:, :, None, None] + s.astype(np.float64)[:, :, None, None] * np.arange(16)
    dist = np.abs(xg[:, :, :, None] - grid)                         # [rows, G, 32, 16]
    best = dist.min(axis=3)
    mine = np.take_along_axis(dist, codes.reshape(400, 2, 32, 1).astype(np.int64), axis=3)[..., 0]
    assert (mine <= best + 1e-9 * s.astype(np.float64)[:, :, None]).all()
    # codes chosen against the unrounded fp32 scale disagree somewhere in this sample
    mn = xg.min(axis=2, keepdims=True)
    s32 = ((xg.max(axis=2, keepdims=True) - mn) / 15.0)
    alt = np.clip(np.rint((xg - b.astype(np.float64)[:, :, None]) / s32), 0, 15)
    assert (alt != codes.reshape(400, 2, 32)).any()


# ------------------------------------------------------------------ dense attention

def _naive_attention(q, keys, vals, tau):
    """Pure-Python brute force: explicit loops and math.exp, no max-shift."""
    z = [tau * sum(qd * kd for qd, kd in zip(q, k)) for k in keys]
    w = [math.exp(zi) for zi in z]
    tot = sum(w)
    out = [sum(w[t] * vals[t][d] for t in range(len(keys))) / tot for d in range(len(q))]
    return out, math.log(tot)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(4)
    for N in (1, 2, 3, 5, 8):
        D = 4
        q = rng.standard_normal((1, 1, D))
        K = rng.standard_normal((1, N, D))
        V = rng.standard_normal((1, N, D))
        O, L = orc.prefix_query(q, K, V)
        o2, l2 = _naive_attention(q[0, 0].tolist(), K[0].tolist(), V[0].tolist(), 1 / math.sqrt(D))
        assert np.allclose(O[0, 0], o2, rtol=1e-12, atol=1e-12)
        assert abs(L[0, 0] - l2) < 1e-12


def test_attention_closed_forms():
    rng = np.random.default_rng(5)
    D, N = 64, 37
    q = rng.standard_normal((1, 1, D))
    V = rng.standard_normal((1, N, D))
    # N = 1: output is the single value row, LSE the single scaled logit.
    K1 = rng.standard_normal((1, 1, D))
    O, L = orc.prefix_query(q, K1, V[:, :1])
    assert np.allclose(O[0, 0], V[0, 0]) and np.isclose(L[0, 0], (q[0, 0] @ K1[0, 0]) / 8.0)
    # identical keys: mean of V, LSE = tau q.k + ln N
    K = np.repeat(K1, N, axis=1)
    O, L = orc.prefix_query(q, K, V)
    assert np.allclose(O[0, 0], V[0].mean(axis=0)) and np.isclose(L[0, 0], (q[0, 0] @ K1[0, 0]) / 8 + math.log(N))
    # Q = 0: mean of V, LSE = ln N
    Kr = rng.standard_normal((1, N, D))
    O, L = orc.prefix_query(np.zeros_like(q), Kr, V)
    assert np.allclose(O[0, 0], V[0].mean(axis=0)) and np.isclose(L[0, 0], math.log(N))


def test_attention_matches_scipy_and_torch():
    """LSE equals scipy's logsumexp of the scaled scores; O equals torch's CPU SDPA (float64)."""
    rng = np.random.default_rng(6)
    H, M, N, D = 3, 5, 50, 32
    Q = rng.standard_normal((H, M, D))
    K = rng.standard_normal((H, N, D)) * 2
    V = rng.standard_normal((H, N, D))
    O, L = orc.prefix_query(Q, K, V, head_map=np.arange(H))
    for h in range(H):
        assert np.allclose(L[h], logsumexp(Q[h] @ K[h].T / math.sqrt(D), axis=1), atol=1e-12)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None]).numpy()[0]
    assert np.allclose(O, ref, atol=1e-12)


@pytest.mark.parametrize("M,S", [(1, 16), (4, 4), (3, 7), (8, 5), (512, 512)])
def test_causal_suffix_matches_torch_mask(M, S):
    """Bottom-right causal suffix: the mask built with torch.tril(diagonal=S-M)."""
    rng = np.random.default_rng(7 + M)
    H, N, D = 2, 9, 16
    if M == 512:
        H, N, D = 1, 33, 16
    Q = rng.standard_normal((H, M, D))
    K, V = rng.standard_normal((H, N, D)), rng.standard_normal((H, N, D))
    Ks, Vs = rng.standard_normal((H, S, D)), rng.standard_normal((H, S, D))
    O, L = orc.prefix_query(Q, K, V, np.arange(H), Ks, Vs, causal=True)
    mask = torch.cat([torch.ones(M, N, dtype=torch.bool), torch.ones(M, S, dtype=torch.bool).tril(diagonal=S - M)], 1)
    q = torch.from_numpy(Q)[None]
    k = torch.from_numpy(np.concatenate([K, Ks], 1))[None]
    v = torch.from_numpy(np.concatenate([V, Vs], 1))[None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask).numpy()[0]
    assert np.allclose(O, ref, atol=1e-11)
    sc = (q @ k.transpose(-1, -2))[0] / math.sqrt(D)
    lse = torch.logsumexp(sc.masked_fill(~mask, float("-inf")), dim=-1).numpy()
    assert np.allclose(L, lse, atol=1e-11)
    if M == S:  # standard causal: torch's own is_causal on the suffix-only part
        O2, _ = orc.prefix_query(Q, K[:, :0], V[:, :0], np.arange(H), Ks, Vs, causal=True)
        ref2 = torch.nn.functional.scaled_dot_product_attention(
            q, torch.from_numpy(Ks)[None], torch.from_numpy(Vs)[None], is_causal=True).numpy()[0]
        assert np.allclose(O2, ref2, atol=1e-11)


def test_split_merge_equals_full():
    """Attention over a split prefix merged through the LSE trailer equals full attention."""
    rng = np.random.default_rng(8)
    H, N, D = 4, 100, 64
    Q = rng.standard_normal((H, 2, D))
    K, V = rng.standard_normal((2, N, D)), rng.standard_normal((2, N, D))
    hm = np.array([0, 0, 1, 1])
    O, L = orc.prefix_query(Q, K, V, hm)
    for t in (1, 17, 50, 99):
        O1, L1 = orc.prefix_query(Q, K[:, :t], V[:, :t], hm)
        O2, L2 = orc.prefix_query(Q, K[:, t:], V[:, t:], hm)
        Om, Lm = orc.merge_partials(O1, L1, O2, L2)
        assert np.allclose(Om, O, atol=1e-12) and np.allclose(Lm, L, atol=1e-12)
        Om2, Lm2 = orc.merge_partials(O2, L2, O1, L1)
        assert np.allclose(Om2, Om, atol=1e-14) and np.allclose(Lm2, Lm, atol=1e-14)


def test_fused_suffix_equals_merge_of_parts():
    rng = np.random.default_rng(9)
    H_q, H_kv, N, S, D = 8, 2, 40, 16, 64
    Q = rng.standard_normal((H_q, 1, D))
    K, V = rng.standard_normal((H_kv, N, D)), rng.standard_normal((H_kv, N, D))
    Ks, Vs = rng.standard_normal((H_kv, S, D)), rng.standard_normal((H_kv, S, D))
    hm = synth.default_head_map(H_q, H_kv)
    O, L = orc.prefix_query(Q, K, V, hm, Ks, Vs)
    Op, Lp = orc.prefix_query(Q, K, V, hm)
    Os, Ls = orc.prefix_query(Q, Ks, Vs, hm)
    Om, Lm = orc.merge_partials(Op, Lp, Os, Ls)
    assert np.allclose(O, Om, atol=1e-12) and np.allclose(L, Lm, atol=1e-12)
    # M=1: suffix appended to the prefix is plain dense attention over N + S keys.
    Od, Ld = orc.prefix_query(Q, np.concatenate([K, Ks], 1), np.concatenate([V, Vs], 1), hm)
    assert np.allclose(O, Od, atol=1e-12) and np.allclose(L, Ld, atol=1e-12)


def test_gqa_head_map_and_permutation():
    rng = np.random.default_rng(10)
    H_q, H_kv, N, D = 6, 3, 20, 16
    Q = rng.standard_normal((H_q, 2, D))
    K, V = rng.standard_normal((H_kv, N, D)), rng.standard_normal((H_kv, N, D))
    hm = np.array([2, 0, 1, 1, 0, 2])
    O, L = orc.prefix_query(Q, K, V, hm)
    Kx, Vx = K[hm], V[hm]       # explicit per-q-head copies
    O2, L2 = orc.prefix_query(Q, Kx, Vx, np.arange(H_q))
    assert np.allclose(O, O2) and np.allclose(L, L2)
    perm = rng.permutation(N)
    O3, L3 = orc.prefix_query(Q, K[:, perm], V[:, perm], hm)
    assert np.allclose(O, O3, atol=1e-12) and np.allclose(L, L3, atol=1e-12)


def test_merge_with_empty_partial_is_identity():
    O = np.arange(8.0).reshape(2, 4)
    L = np.array([0.3, -2.0])
    Om, Lm = orc.merge_partials(O, L, np.zeros_like(O), np.full(2, -np.inf))
    assert np.allclose(Om, O) and np.allclose(Lm, L)


# ------------------------------------------------------------------ block means, top-K, sparse

def test_block_means_ramp_closed_form():
    H_kv, N, D, B = 2, 203, 3, 64
    K = np.broadcast_to(np.arange(N, dtype=np.float64)[None, :, None], (H_kv, N, D)).copy()
    K[1] *= -2
    km = orc.block_means(K, B)
    assert km.shape == (2, 4, 3)
    for b in range(4):
        lo, hi = b * B, min(N, (b + 1) * B) - 1
        assert np.allclose(km[0, b], (lo + hi) / 2) and np.allclose(km[1, b], -(lo + hi))


def test_block_scores_closed_form():
    """score[h, b] = tau * q_h . K_mean[head_map[h], b]: unit queries against known block means,
    through a head map that is neither the identity nor the grouped default."""
    D = 16
    tau = 1.0 / np.sqrt(D)
    km = np.zeros((2, 3, D))
    km[0, :, 3] = [1.0, 2.0, 4.0]        # kv head 0: d = 3 carries 1, 2, 4
    km[1, :, 5] = [-8.0, 0.5, 16.0]      # kv head 1: d = 5 carries -8, 0.5, 16
    Q = np.zeros((3, D))
    Q[0, 3] = 2.0                        # head 0 -> kv head 1, but probes d = 3: all zero
    Q[1, 5] = 3.0                        # head 1 -> kv head 1, probes d = 5
    Q[2, 3] = -1.0                       # head 2 -> kv head 0, probes d = 3
    sc = orc.block_scores(Q, km, np.array([1, 1, 0]))
    assert sc.shape == (3, 3)
    assert np.allclose(sc[0], 0.0)
    assert np.allclose(sc[1], tau * 3.0 * np.array([-8.0, 0.5, 16.0]))
    assert np.allclose(sc[2], -tau * np.array([1.0, 2.0, 4.0]))


def test_topk_margin_worked_example():
    """Gap between the K-th and (K+1)-th largest score of a row, by hand: scores 5, 1, 3, 3."""
    s = np.array([[5.0, 1.0, 3.0, 3.0]])
    assert orc.topk_margin(s, 1)[0] == 2.0      # 5 vs 3
    assert orc.topk_margin(s, 2)[0] == 0.0      # 3 vs 3: a tie at the cut
    assert orc.topk_margin(s, 3)[0] == 2.0      # 3 vs 1
    assert np.isinf(orc.topk_margin(s, 4)[0])   # every block kept: no cut


def test_topk_tie_example():
    lines = _golden_lines("topk_tie_example.txt")
    scores = np.array([[float(v) for v in lines[0].split(":")[1].split()]])
    for ln in lines[1:]:
        k = int(ln.split()[0].split("=")[1])
        want = [int(v) for v in ln.split(":")[1].split()]
        assert orc.select_top_blocks(scores, k)[0].tolist() == want


def test_sparse_covering_all_blocks_equals_dense():
    rng = np.random.default_rng(11)
    H_q, H_kv, N, D, B = 4, 2, 300, 32, 64
    Q = rng.standard_normal((H_q, 1, D))
    K, V = rng.standard_normal((H_kv, N, D)), rng.standard_normal((H_kv, N, D))
    Ks, Vs = rng.standard_normal((H_kv, 8, D)), rng.standard_normal((H_kv, 8, D))
    hm = synth.default_head_map(H_q, H_kv)
    for Kt in (5, 9):
        O, L, idx, _ = orc.sparse_query(Q, K, V, hm, B, Kt, Ks, Vs)
        Od, Ld = orc.prefix_query(Q, K, V, hm, Ks, Vs)
        assert (idx == np.arange(5)).all()
        assert np.allclose(O, Od[:, 0], atol=1e-12) and np.allclose(L, Ld[:, 0], atol=1e-12)


def test_sparse_equals_dense_over_selected_tokens():
    rng = np.random.default_rng(12)
    H_q, H_kv, N, D, B = 4, 1, 256, 16, 32
    Q = rng.standard_normal((H_q, D))
    K, V = rng.standard_normal((H_kv, N, D)), rng.standard_normal((H_kv, N, D))
    hm = np.zeros(H_q, dtype=np.int32)
    O, L, idx, scores = orc.sparse_query(Q, K, V, hm, B, 3)
    for h in range(H_q):
        toks = np.concatenate([np.arange(b * B, (b + 1) * B) for b in idx[h]])
        Od, Ld = orc.prefix_query(Q[h][None, None], K[:, toks], V[:, toks], np.zeros(1, dtype=int))
        assert np.allclose(O[h], Od[0, 0]) and np.isclose(L[h], Ld[0, 0])
        # selected blocks really are the top-3 by score
        assert set(idx[h]) == set(np.argsort(-scores[h], kind="stable")[:3])


def test_needle_workload_selects_needles():
    """Sparse workload at reduced length: planted needles are exactly the selected blocks."""
    H_q, H_kv, N, D, B, Kt = 8, 2, 8192, 256, 64, 8
    seed = 0
    K, V = synth.gen_kv(seed, H_kv, N, D)
    Q = synth.gen_q(seed, H_q, 1, D)[:, 0]
    hm = synth.default_head_map(H_q, H_kv)
    needles = synth.needle_blocks(seed, N // B, Kt)
    K = synth.plant_needles(K, Q, hm, needles, B)
    scores = orc.block_scores(Q, orc.block_means(K, B), hm)
    idx = orc.select_top_blocks(scores, Kt)
    assert (idx == needles[None, :]).all()
    assert (orc.topk_margin(scores, Kt) > 0.5).all()


def test_sparse_indices_hand_worked_two_heads():
    """Two heads, D = 2 (tau = 1/sqrt(2)), by hand. Head 0 picks tokens {0, 2} of kv head 0 with
    q = (sqrt(2) ln 3, 0): scores 0 and ln 3, weights 1/4 and 3/4, LSE = ln 4. Head 1 picks
    token {1} of kv head 1 alone: O is that value row, LSE its score."""
    Q = np.array([[math.sqrt(2) * math.log(3), 0.0], [0.5, -1.0]])
    K = np.array([[[0.0, 5.0], [7.0, 7.0], [1.0, -2.0]],
                  [[9.0, 9.0], [2.0, 4.0], [-3.0, 3.0]]])
    V = np.array([[[4.0, 0.0], [100.0, 100.0], [0.0, 8.0]],
                  [[50.0, 50.0], [-1.0, 2.0], [60.0, 60.0]]])
    idx = np.array([[0, 2], [1, 0]])
    cnt = np.array([2, 1])
    O, L = orc.sparse_query_indices(Q, K, V, idx, cnt, head_map=np.array([0, 1]))
    assert np.allclose(O[0], [1.0, 6.0]) and math.isclose(L[0], math.log(4.0))
    assert np.allclose(O[1], [-1.0, 2.0])
    assert math.isclose(L[1], (0.5 * 2.0 - 1.0 * 4.0) / math.sqrt(2))


def test_sparse_indices_all_tokens_equal_dense():
    rng = np.random.default_rng(13)
    H_q, H_kv, N, D = 6, 2, 50, 16
    Q = rng.standard_normal((H_q, 1, D))
    K, V = rng.standard_normal((H_kv, N, D)), rng.standard_normal((H_kv, N, D))
    idx = np.tile(np.arange(N), (H_q, 1))
    O, L = orc.sparse_query_indices(Q, K, V, idx, np.full(H_q, N))
    Od, Ld = orc.prefix_query(Q, K, V)
    assert np.allclose(O, Od[:, 0], atol=1e-12) and np.allclose(L, Ld[:, 0], atol=1e-12)


def test_sparse_indices_of_selected_blocks_equal_auto():
    """The tokens of the blocks the block-mean selector picks, given as indices, give the
    selector's own sparse answer."""
    rng = np.random.default_rng(14)
    H_q, H_kv, N, D, B, Kt = 4, 2, 300, 32, 32, 3
    Q = rng.standard_normal((H_q, D))
    K, V = rng.standard_normal((H_kv, N, D)), rng.standard_normal((H_kv, N, D))
    hm = synth.default_head_map(H_q, H_kv)
    Oa, La, sel, _ = orc.sparse_query(Q, K, V, hm, B, Kt)
    rows = [np.concatenate([np.arange(b * B, min(N, (b + 1) * B)) for b in sel[h]]) for h in range(H_q)]
    kmax = max(len(r) for r in rows)
    idx = np.zeros((H_q, kmax), dtype=np.int64)
    for h, r in enumerate(rows):
        idx[h, :len(r)] = r
    O, L = orc.sparse_query_indices(Q, K, V, idx, [len(r) for r in rows], hm)
    assert np.allclose(O, Oa, atol=1e-12) and np.allclose(L, La, atol=1e-12)


def test_warm_heads_lossless_on_grid_and_rounded_once():
    """Groups that sit exactly on an fp16 grid b + k s come back bit-exact in both output types;
    random groups come back in fp32 within half an fp32 ulp of the exact value."""
    H_kv, N, D = 2, 5, 64
    rng = np.random.default_rng(15)
    b = np.float16(-3.5)
    s = np.float16(0.25)
    x = (np.float32(b) + np.float32(s) * rng.integers(0, 16, size=(N, H_kv * D)).astype(np.float32)).astype(np.float16)
    x[:, ::32] = b                      # every group holds its minimum ...
    x[:, 1::32] = np.float16(b + 15 * s)   # ... and its maximum, so the scale is s exactly
    rec = orc.quantize_records(x)
    want = x.reshape(N, H_kv, D).transpose(1, 0, 2)
    assert np.array_equal(orc.warm_heads(rec, H_kv, D, np.float32), want.astype(np.float32))
    assert np.array_equal(orc.warm_heads(rec, H_kv, D, np.float16), want)
    y = (rng.standard_normal((N, H_kv * D)) * 40 + 200).astype(np.float16)
    rec = orc.quantize_records(y)
    exact = orc.records_to_heads(rec, H_kv, D)
    w32 = orc.warm_heads(rec, H_kv, D, np.float32)
    assert w32.dtype == np.float32
    assert (np.abs(w32.astype(np.float64) - exact) <= np.spacing(np.abs(w32)) / 2).all()


def test_window_equals_attention_over_the_last_keys():
    """A window of W keys at M = 1 equals plain attention over the last W positions of the
    concatenated prefix and suffix, built by slicing (so prefix-only, suffix-only and mixed
    windows are all covered); W = 0 and W >= N + S change nothing."""
    rng = np.random.default_rng(16)
    H_q, H_kv, N, S, D = 4, 2, 40, 9, 16
    Q = rng.standard_normal((H_q, 1, D))
    K, V = rng.standard_normal((H_kv, N, D)), rng.standard_normal((H_kv, N, D))
    Ks, Vs = rng.standard_normal((H_kv, S, D)), rng.standard_normal((H_kv, S, D))
    Kall, Vall = np.concatenate([K, Ks], axis=1), np.concatenate([V, Vs], axis=1)
    full = orc.prefix_query(Q, K, V, None, Ks, Vs)
    for W in (0, N + S, N + S + 7):
        O, L = orc.prefix_query(Q, K, V, None, Ks, Vs, window=W)
        assert np.allclose(O, full[0]) and np.allclose(L, full[1])
    for W in (1, 3, S, S + 1, 25, N + S - 1):
        O, L = orc.prefix_query(Q, K, V, None, Ks, Vs, window=W)
        Or, Lr = orc.prefix_query(Q, Kall[:, -W:], Vall[:, -W:])
        assert np.allclose(O, Or, atol=1e-12) and np.allclose(L, Lr, atol=1e-12)
    # W = 1 at M = 1: the value row of the last suffix key, LSE = its score
    O, L = orc.prefix_query(Q, K, V, None, Ks, Vs, window=1)
    g = np.arange(H_q) // 2
    assert np.allclose(O[:, 0], Vs[g, -1])
    assert np.allclose(L[:, 0], np.einsum("hd,hd->h", Q[:, 0], Ks[g, -1]) / math.sqrt(D))


def test_window_per_row_under_the_causal_mask():
    """M > 1: row i sees positions p_i - W + 1 .. p_i with p_i = N + S - M + i: a hand-built mask
    from positions, compared with suffix_allowed."""
    N, S, M, W = 6, 4, 3, 4
    allowed = orc.suffix_allowed(M, N, S, True, W)
    for i in range(M):
        p_i = N + S - M + i
        want = np.array([(p_i - W + 1) <= t <= p_i for t in range(N + S)])
        assert (allowed[i] == want).all()


# ------------------------------------------------------------------ planted mistakes are caught

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check a pin fails for each."""
    import oracle.pck_oracle as mod
    good = mod.attend_rows

    def no_tau(q, k, v, tau, allowed=None):
        return good(q, k, v, 1.0, allowed)

    def drop_max(q, k, v, tau, allowed=None):
        O, L = good(q, k, v, tau, allowed)
        return O, L - np.max(tau * (np.asarray(q) @ np.asarray(k).T), axis=1)

    for bad in (no_tau, drop_max):
        monkeypatch.setattr(mod, "attend_rows", bad)
        with pytest.raises(AssertionError):
            test_attention_matches_scipy_and_torch()
        monkeypatch.setattr(mod, "attend_rows", good)

    good_q = mod.quantize_mlx4g32

    def symmetric(x):
        c, s, b = good_q(x)
        return c, s, np.zeros_like(b)

    monkeypatch.setattr(mod, "quantize_mlx4g32", symmetric)
    with pytest.raises(AssertionError):
        test_quantizer_lossless_on_grid()
    monkeypatch.setattr(mod, "quantize_mlx4g32", good_q)

    def groups_and_params(x):
        """x as [rows, groups, 32] float64, with the correct fp16 scales and biases."""
        xg = np.asarray(x).astype(np.float64).reshape(np.shape(x)[0], -1, 32)
        _, s16, b16 = good_q(x)
        return xg, s16, b16

    def fp32_scale_codes(x):
        xg, s16, b16 = groups_and_params(x)
        s32 = (xg.max(axis=2) - xg.min(axis=2)) / 15.0
        c = np.clip(np.rint((xg - b16.astype(np.float64)[:, :, None]) / s32[:, :, None]), 0, 15)
        return c.astype(np.uint8).reshape(np.shape(x)), s16, b16

    def truncated_codes(x):
        xg, s16, b16 = groups_and_params(x)
        with np.errstate(divide="ignore", invalid="ignore"):
            t = (xg - b16.astype(np.float64)[:, :, None]) / s16.astype(np.float64)[:, :, None]
        c = np.where((s16 == 0)[:, :, None], 0, np.clip(np.floor(np.nan_to_num(t)), 0, 15))
        return c.astype(np.uint8).reshape(np.shape(x)), s16, b16

    for bad, pin in ((fp32_scale_codes, test_quantizer_scale_is_fp16_roundtripped),
                     (truncated_codes, test_quantizer_error_bound_and_monotone)):
        monkeypatch.setattr(mod, "quantize_mlx4g32", bad)
        with pytest.raises(AssertionError):
            pin()
        monkeypatch.setattr(mod, "quantize_mlx4g32", good_q)

    good_pc = mod.pack_codes

    def wrong_nibble_order(codes):
        return good_pc(codes[:, ::-1].copy())

    monkeypatch.setattr(mod, "pack_codes", wrong_nibble_order)
    with pytest.raises(AssertionError):
        test_layout_worked_example()
    monkeypatch.setattr(mod, "pack_codes", good_pc)

    good_bs = mod.block_scores

    def scores_no_tau(Q, K_mean, head_map):
        return good_bs(Q, K_mean, head_map) * np.sqrt(np.shape(Q)[-1])

    def scores_ignore_map(Q, K_mean, head_map):
        return good_bs(Q, K_mean, np.arange(np.shape(Q)[0]) % K_mean.shape[0])

    for bad in (scores_no_tau, scores_ignore_map):
        monkeypatch.setattr(mod, "block_scores", bad)
        with pytest.raises(AssertionError):
            test_block_scores_closed_form()
        monkeypatch.setattr(mod, "block_scores", good_bs)

    good_tm = mod.topk_margin

    def margin_off_by_one(scores, K_top):
        return good_tm(scores, K_top + 1)

    monkeypatch.setattr(mod, "topk_margin", margin_off_by_one)
    with pytest.raises(AssertionError):
        test_topk_margin_worked_example()
    monkeypatch.setattr(mod, "topk_margin", good_tm)

    good_bm = mod.block_means

    def means_over_full_blocks(K, B):
        K = np.asarray(K, dtype=np.float64)
        nb = (K.shape[1] + B - 1) // B
        pad = np.zeros((K.shape[0], nb * B - K.shape[1], K.shape[2]))
        return np.concatenate([K, pad], axis=1).reshape(K.shape[0], nb, B, K.shape[2]).mean(axis=2)

    monkeypatch.setattr(mod, "block_means", means_over_full_blocks)
    with pytest.raises(AssertionError):
        test_block_means_ramp_closed_form()
    monkeypatch.setattr(mod, "block_means", good_bm)

    good_mask = mod.suffix_allowed

    def top_left_causal(M, N, S, causal, window=0):
        allowed = np.ones((M, N + S), dtype=bool)
        if S and causal:
            for i in range(M):
                allowed[i, N + i + 1:] = False
        return allowed

    def causal_one_short(M, N, S, causal, window=0):
        allowed = good_mask(M, N, S, causal)
        if S and causal:
            for i in range(M):
                j = S - M + i
                if 0 <= j < S:
                    allowed[i, N + j] = False
        return allowed

    for bad in (top_left_causal, causal_one_short):
        monkeypatch.setattr(mod, "suffix_allowed", bad)
        with pytest.raises(AssertionError):
            test_causal_suffix_matches_torch_mask(3, 7)
        monkeypatch.setattr(mod, "suffix_allowed", good_mask)

    good_rh = mod.records_to_heads

    def heads_as_token_blocks(rec, H_kv, D):
        x = mod.dequantize_mlx4g32(*mod.unpack_records(rec, H_kv * D))
        return x.reshape(H_kv, rec.shape[0], D).copy()     # reads the rows as head-major blocks

    monkeypatch.setattr(mod, "records_to_heads", heads_as_token_blocks)
    with pytest.raises(AssertionError):
        test_records_to_heads_lossless_roundtrip()
    monkeypatch.setattr(mod, "records_to_heads", good_rh)

    good_sqi = mod.sparse_query_indices

    def counts_off_by_one(Q, K, V, indices, counts, head_map=None):
        return good_sqi(Q, K, V, indices, np.asarray(counts) + 1, head_map)

    def rows_of_next_head(Q, K, V, indices, counts, head_map=None):
        return good_sqi(Q, K, V, np.roll(np.asarray(indices), 1, axis=0), np.roll(np.asarray(counts), 1), head_map)

    for bad in (counts_off_by_one, rows_of_next_head):
        monkeypatch.setattr(mod, "sparse_query_indices", bad)
        with pytest.raises((AssertionError, IndexError)):
            test_sparse_indices_hand_worked_two_heads()
        monkeypatch.setattr(mod, "sparse_query_indices", good_sqi)

    good_wh = mod.warm_heads

    def warm_without_transpose(rec, H_kv, D, dtype=np.float32):
        x = mod.dequantize_mlx4g32(*mod.unpack_records(rec, H_kv * D)).astype(np.float32)
        x = x.reshape(H_kv, rec.shape[0], D)
        return x if np.dtype(dtype) == np.float32 else x.astype(np.float16)

    monkeypatch.setattr(mod, "warm_heads", warm_without_transpose)
    with pytest.raises(AssertionError):
        test_warm_heads_lossless_on_grid_and_rounded_once()
    monkeypatch.setattr(mod, "warm_heads", good_wh)

    def window_one_short(M, N, S, causal, window=0):
        allowed = good_mask(M, N, S, causal, window)
        if window > 0:
            for i in range(M):
                t = N + S - M + i - window + 1
                if 0 <= t < N + S:
                    allowed[i, t] = False
        return allowed

    monkeypatch.setattr(mod, "suffix_allowed", window_one_short)
    with pytest.raises(AssertionError):
        test_window_equals_attention_over_the_last_keys()
    monkeypatch.setattr(mod, "suffix_allowed", good_mask)
