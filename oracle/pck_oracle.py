"""CPU oracle for prefix-cached KV attention -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy in float64 (float32/float16 only where a step
is defined in those precisions: the mlx4g32 quantiser). Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
module. The CUDA library never imports, links or calls it, and it shares no code,
table or helper with the CUDA library.

What each function follows (page title, section):

* mlx4g32 record layout and quantiser -- "Shared KV Cache Serving -- Pion as LLM
  Memory", section "Quantized tier -- mlx4g32"; the same text is on "V.* -- the
  V-store", section "The mlx4g32 tier": 4-bit codes in groups of 32 values, each
  group affine with its own fp16 scale and fp16 bias. A token's record holds D/8
  32-bit code words, then D/32 fp16 scales, then D/32 fp16 biases; the code of a
  group's j-th value fills the four bits from ``4*(j mod 8)`` of its word. The scale
  is rounded to fp16 first, and the codes are picked against that rounded scale.
* Attention over the resident prefix -- "ATTEND.* and ATTEND.PREFIX.*", section
  "Wire forms" (QUERY, QUERY_FUSED, QUERY_SPARSE_AUTO(_FUSED)), and "Shared KV
  Cache Serving", section "Stage 2: ATTEND.PREFIX.*" (agreement is judged against
  a CPU softmax(QK^T)V).
* LSE trailer and the two-halves merge -- "Shared KV Cache Serving", section
  "Wire-protocol details" (batched-Q returns O followed by one LSE per row; the
  LSE is what the online-softmax merge needs).
* Block-mean top-K selection -- "ATTEND.* and ATTEND.PREFIX.*", section "Wire
  forms" (the server keeps block means of K per slot, scores blocks against Q
  and keeps K_top blocks of size B, GQA-aware).
* Sparse attention over caller-chosen tokens -- "ATTEND.* and ATTEND.PREFIX.*",
  command table, QUERY_SPARSE (per-head indices and counts, at most K_sparse_max
  of them, supplied by the caller, e.g. a learned router).
* Dequantise-and-transpose of stored records -- "Shared KV Cache Serving -- Pion
  as LLM Memory", sections "KV.PREFIX.WARM" and "Cold-tier state machine" (the
  records come back as fp32 and are turned from token-major [N, H*D] into the
  attention layout [H, N, D]); "V.* -- the V-store", V.FETCH RANGE (dequantised
  fp32 values).

Readings taken where the pages are silent:

* Quantiser: mn/mx are the group's min/max as fp32; s32 = fp32(mx-mn)/15 in fp32;
  s16 = fp16(s32); b16 = fp16(mn); code = clamp(rint_half_even(fp32(fp32(x - b16) /
  s16)), 0, 15); a group with s16 == 0 gets all-zero codes. Dequant x^ = s16*c + b16.
* Scores use tau = 1/sqrt(D); LSE is the natural log of sum(exp(tau q.k)).
* Causal suffix mask, bottom-right aligned: query row i of M sees every prefix key
  and suffix keys j <= S_suf - M + i.
* head_map is an int array, q head h reads kv head head_map[h].
* Top-K is per query head; ties go to the lower block index; K_top is clamped to the
  number of blocks; the selected indices are returned sorted ascending. The last
  block may be partial; its mean is over the tokens it has.
* QUERY_SPARSE indices are prefix token positions; q head h attends to the first
  counts[h] entries of its row of indices (kv head head_map[h]).
* fa_window (listed on every QUERY form, never defined): a sliding attention window.
  Query row i sits at absolute position p_i = N + S_suf - M + i (prefix positions
  0..N-1, then the suffix), the last key it may see; with fa_window = W > 0 it sees
  only keys at positions p_i - W + 1 .. p_i. W = 0 means no window.
* The dequantised values are fp32: the exact s*c + b rounded once to fp32. An fp16
  output is that fp32 value rounded to fp16.
"""
from __future__ import annotations

import math

import numpy as np

GROUP = 32  # elements per mlx4g32 group


# ----------------------------------------------------------------------------------
# mlx4g32 tier
# ----------------------------------------------------------------------------------

def record_bytes(kv_dim: int) -> int:
    """Bytes of one token's record: kv_dim/8 u32 words + kv_dim/32 fp16 scales + kv_dim/32 fp16 biases."""
    assert kv_dim % GROUP == 0
    return (kv_dim // 8) * 4 + (kv_dim // GROUP) * 2 * 2


def quantize_mlx4g32(x) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Affine int4, group-32 quantisation of rows of x (fp16 or fp32 values).

    Returns (codes uint8 [rows, kv_dim] in 0..15, scales fp16 [rows, G], biases fp16 [rows, G]).
    Every arithmetic step is an IEEE fp32 operation (numpy float32 scalars/arrays round to
    nearest even after each op), then the fp16 roundings the page describes.
    """
    x = np.asarray(x)
    rows, kv_dim = x.shape
    G = kv_dim // GROUP
    xg = x.astype(np.float32).reshape(rows, G, GROUP)
    mn = xg.min(axis=2)                                              # fp32 [rows, G]
    mx = xg.max(axis=2)
    s32 = ((mx - mn).astype(np.float32) / np.float32(15.0)).astype(np.float32)
    scales = s32.astype(np.float16)                                  # the scale the reader will see
    biases = mn.astype(np.float16)
    a = (xg - biases.astype(np.float32)[:, :, None]).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (a / scales.astype(np.float32)[:, :, None]).astype(np.float32)
    codes = np.clip(np.rint(t), 0, 15)
    codes = np.where((scales == 0)[:, :, None], 0, codes).astype(np.uint8)   # constant group: all codes 0
    return codes.reshape(rows, kv_dim), scales, biases


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [rows, kv_dim] -> uint32 words [rows, kv_dim/8]; code j fills bits 4*(j%8) .. 4*(j%8)+3 of word j//8."""
    rows, kv_dim = codes.shape
    words = np.zeros((rows, kv_dim // 8), dtype=np.uint32)
    for j in range(kv_dim):
        words[:, j // 8] |= codes[:, j].astype(np.uint32) << np.uint32(4 * (j % 8))
    return words


def unpack_codes(words: np.ndarray, kv_dim: int) -> np.ndarray:
    rows = words.shape[0]
    codes = np.zeros((rows, kv_dim), dtype=np.uint8)
    for j in range(kv_dim):
        codes[:, j] = (words[:, j // 8] >> np.uint32(4 * (j % 8))) & np.uint32(0xF)
    return codes


def pack_records(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray) -> np.ndarray:
    """Token-major records, little-endian: [u32 codes x D/8][f16 scales x D/32][f16 biases x D/32]."""
    words = pack_codes(codes)
    rows = codes.shape[0]
    parts = [words.astype("<u4").view(np.uint8).reshape(rows, -1),
             scales.astype("<f2").view(np.uint8).reshape(rows, -1),
             biases.astype("<f2").view(np.uint8).reshape(rows, -1)]
    return np.ascontiguousarray(np.concatenate(parts, axis=1))


def unpack_records(rec: np.ndarray, kv_dim: int):
    """Inverse of pack_records -> (codes, scales, biases)."""
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    rows = rec.shape[0]
    nw, G = kv_dim // 8, kv_dim // GROUP
    words = rec[:, :4 * nw].copy().view("<u4").reshape(rows, nw)
    scales = rec[:, 4 * nw:4 * nw + 2 * G].copy().view("<f2").reshape(rows, G)
    biases = rec[:, 4 * nw + 2 * G:4 * nw + 4 * G].copy().view("<f2").reshape(rows, G)
    return unpack_codes(words, kv_dim), scales.astype(np.float16), biases.astype(np.float16)


def dequantize_mlx4g32(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray) -> np.ndarray:
    """x^ = s * c + b per element, in float64 (exact for fp16 s, b and 4-bit c)."""
    rows, kv_dim = codes.shape
    s = np.repeat(scales.astype(np.float64), GROUP, axis=1)
    b = np.repeat(biases.astype(np.float64), GROUP, axis=1)
    return s * codes.astype(np.float64) + b


def quantize_records(x) -> np.ndarray:
    """Rows of x -> packed mlx4g32 records [rows, record_bytes]."""
    return pack_records(*quantize_mlx4g32(x))


def records_to_heads(rec: np.ndarray, H_kv: int, D: int) -> np.ndarray:
    """Dequantised token-major records [N, H_kv*D] -> float64 [H_kv, N, D]."""
    x = dequantize_mlx4g32(*unpack_records(rec, H_kv * D))
    return x.reshape(rec.shape[0], H_kv, D).transpose(1, 0, 2).copy()


def warm_heads(rec: np.ndarray, H_kv: int, D: int, dtype=np.float32) -> np.ndarray:
    """The WARM / FETCH RANGE form of stored records: [H_kv, N, D] in fp32 (each exact
    dequantised value rounded once to fp32), or fp16 (that fp32 value rounded to fp16)."""
    x32 = records_to_heads(rec, H_kv, D).astype(np.float32)
    return x32 if np.dtype(dtype) == np.float32 else x32.astype(np.float16)


# ----------------------------------------------------------------------------------
# Dense attention (two-pass softmax; not the online form the kernels use)
# ----------------------------------------------------------------------------------

def attend_rows(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, tau: float,
                allowed: np.ndarray | None = None):
    """softmax(tau * q k^T) v for each query row, with an optional [R, T] boolean key mask.

    Returns (O [R, D], LSE [R]) with LSE = log(sum_t exp(tau q.k_t)) in natural-log units.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    z = tau * (q_rows @ keys.T)                       # [R, T]
    if allowed is not None:
        z = np.where(allowed, z, -np.inf)
    m = z.max(axis=1, keepdims=True)                  # pass 1: max
    w = np.exp(z - m)                                 # pass 2: weights
    l = w.sum(axis=1, keepdims=True)
    O = (w @ values) / l
    LSE = (m + np.log(l))[:, 0]
    return O, LSE


def suffix_allowed(M: int, N: int, S: int, causal: bool, window: int = 0) -> np.ndarray:
    """[M, N + S] key mask of the fused forms: every row sees the N prefix keys; with causal, row
    i (0-based, of M) sees suffix keys j <= S - M + i (bottom-right alignment), else all S. With
    window = W > 0, row i sees only positions p_i - W + 1 .. p_i, p_i = N + S - M + i."""
    allowed = np.ones((M, N + S), dtype=bool)
    if S and causal:
        for i in range(M):
            jmax = S - M + i
            allowed[i, N + max(jmax + 1, 0):] = False
    if window > 0:
        for i in range(M):
            p_i = N + S - M + i
            allowed[i, :max(p_i - window + 1, 0)] = False
    return allowed


def prefix_query(Q, K, V, head_map=None, K_suf=None, V_suf=None, causal: bool = True, window: int = 0):
    """Attention of Q [H_q, M, D] over the prefix K/V [H_kv, N, D] (+ optional suffix [H_kv, S, D]).

    Query row i (0-based, of M) sees all N prefix keys and, when causal, suffix keys
    j <= S - M + i (bottom-right alignment); without causal it sees the whole suffix. A window
    W > 0 keeps only the W positions up to p_i = N + S - M + i (see suffix_allowed).
    Returns (O [H_q, M, D] float64, LSE [H_q, M] float64).
    """
    Q = np.asarray(Q, dtype=np.float64)
    H_q, M, D = Q.shape
    H_kv, N, _ = K.shape
    if head_map is None:
        head_map = np.arange(H_q) // (H_q // H_kv)
    tau = 1.0 / math.sqrt(D)
    S = 0 if K_suf is None else K_suf.shape[1]
    O = np.zeros((H_q, M, D))
    LSE = np.zeros((H_q, M))
    allowed = suffix_allowed(M, N, S, causal, window)
    for h in range(H_q):
        g = int(head_map[h])
        keys = np.asarray(K[g], dtype=np.float64)
        vals = np.asarray(V[g], dtype=np.float64)
        if S:
            keys = np.concatenate([keys, np.asarray(K_suf[g], dtype=np.float64)])
            vals = np.concatenate([vals, np.asarray(V_suf[g], dtype=np.float64)])
        O[h], LSE[h] = attend_rows(Q[h], keys, vals, tau, allowed)
    return O, LSE


def merge_partials(O1, L1, O2, L2):
    """Online-softmax merge of two attention partials over disjoint key sets.

    L = max + log(e^(L1-max) + e^(L2-max)); O = e^(L1-L) O1 + e^(L2-L) O2.
    """
    L1 = np.asarray(L1, dtype=np.float64)
    L2 = np.asarray(L2, dtype=np.float64)
    mx = np.maximum(L1, L2)
    L = mx + np.log(np.exp(L1 - mx) + np.exp(L2 - mx))
    O = np.exp(L1 - L)[..., None] * O1 + np.exp(L2 - L)[..., None] * O2
    return O, L


# ----------------------------------------------------------------------------------
# Block-mean top-K sparse attention
# ----------------------------------------------------------------------------------

def block_means(K, B: int) -> np.ndarray:
    """K_mean[g, b, :] = mean of K[g, t, :] over the tokens t of block b (last block may be partial)."""
    K = np.asarray(K, dtype=np.float64)
    H_kv, N, D = K.shape
    nb = (N + B - 1) // B
    out = np.zeros((H_kv, nb, D))
    for b in range(nb):
        out[:, b] = K[:, b * B:min(N, (b + 1) * B)].mean(axis=1)
    return out


def block_scores(Q, K_mean, head_map) -> np.ndarray:
    """score[h, b] = tau * q_h . K_mean[head_map[h], b] for M=1 queries Q [H_q, D]."""
    Q = np.asarray(Q, dtype=np.float64).reshape(np.shape(Q)[0], -1)
    tau = 1.0 / math.sqrt(Q.shape[1])
    return np.stack([tau * (K_mean[int(head_map[h])] @ Q[h]) for h in range(Q.shape[0])])


def select_top_blocks(scores: np.ndarray, K_top: int) -> np.ndarray:
    """Per row: the K_top largest scores (ties -> lower block index), returned sorted ascending."""
    H, nb = scores.shape
    k = min(K_top, nb)
    idx = np.zeros((H, k), dtype=np.int32)
    for h in range(H):
        order = sorted(range(nb), key=lambda b: (-scores[h, b], b))
        idx[h] = sorted(order[:k])
    return idx


def topk_margin(scores: np.ndarray, K_top: int) -> np.ndarray:
    """Per row, the gap between the K-th and (K+1)-th largest scores (inf when K_top >= n_blocks)."""
    H, nb = scores.shape
    if K_top >= nb:
        return np.full(H, np.inf)
    s = -np.sort(-scores, axis=1)
    return s[:, K_top - 1] - s[:, K_top]


def sparse_query(Q, K, V, head_map, B: int, K_top: int, K_suf=None, V_suf=None):
    """M=1 attention of each q head over the tokens of its selected blocks (+ the whole suffix).

    Q [H_q, D] (or [H_q, 1, D]). Returns (O [H_q, D], LSE [H_q], idx [H_q, k], scores [H_q, nb]).
    """
    Q = np.asarray(Q, dtype=np.float64).reshape(np.shape(Q)[0], -1)
    H_q, D = Q.shape
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    N = K.shape[1]
    tau = 1.0 / math.sqrt(D)
    scores = block_scores(Q, block_means(K, B), head_map)
    idx = select_top_blocks(scores, K_top)
    O = np.zeros((H_q, D))
    LSE = np.zeros(H_q)
    for h in range(H_q):
        g = int(head_map[h])
        toks = np.concatenate([np.arange(b * B, min(N, (b + 1) * B)) for b in idx[h]])
        keys, vals = K[g, toks], V[g, toks]
        if K_suf is not None and K_suf.shape[1]:
            keys = np.concatenate([keys, np.asarray(K_suf[g], dtype=np.float64)])
            vals = np.concatenate([vals, np.asarray(V_suf[g], dtype=np.float64)])
        o, l = attend_rows(Q[h:h + 1], keys, vals, tau)
        O[h], LSE[h] = o[0], l[0]
    return O, LSE, idx, scores


def sparse_query_indices(Q, K, V, indices, counts, head_map=None):
    """M=1 attention of each q head over the prefix tokens a caller chose for it.

    Q [H_q, D] (or [H_q, 1, D]); K, V [H_kv, N, D]; indices [H_q, K_sparse_max] token
    positions; counts [H_q]: head h attends to tokens indices[h, :counts[h]] of kv head
    head_map[h] (default h // (H_q / H_kv)). Returns (O [H_q, D], LSE [H_q]).
    """
    Q = np.asarray(Q, dtype=np.float64).reshape(np.shape(Q)[0], -1)
    H_q, D = Q.shape
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if head_map is None:
        head_map = np.arange(H_q) // (H_q // K.shape[0])
    tau = 1.0 / math.sqrt(D)
    O = np.zeros((H_q, D))
    LSE = np.zeros(H_q)
    for h in range(H_q):
        g = int(head_map[h])
        toks = np.asarray(indices[h][:int(counts[h])], dtype=np.int64)
        o, l = attend_rows(Q[h:h + 1], K[g, toks], V[g, toks], tau)
        O[h], LSE[h] = o[0], l[0]
    return O, LSE
