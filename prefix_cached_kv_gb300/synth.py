"""Seeded synthetic inputs shaped like the workloads of the shared-prefix KV pages.

This module only draws random inputs. It holds none of the attention, merge,
quantisation or selection arithmetic: the CPU oracle (test infrastructure) and
the CUDA path both receive the exact bytes produced here.

Every tensor comes from its own stream, keyed by (seed, stream id, extra ints),
so that a slice of one workload can be regenerated alone.

Recipe (see "Shared KV Cache Serving -- Pion as LLM Memory", section
"Stage 2: ATTEND.PREFIX.*", and "ATTEND.* and ATTEND.PREFIX.*", section
"Wire forms", for the shapes the pages use):

* K, V: fp16, entries N(0, 1). K column d of kv head g is multiplied by a
  factor f[g, d] ~ lognormal(0, 0.5) before rounding to fp16 (real keys have
  per-channel outliers). ``col_scale=False`` gives plain N(0, 1).
* Q: N(0, 1) in fp32 (or fp16 for the batched-Q workload).
* Suffix K/V: same recipe as the prefix, drawn from their own streams.
* Needles (sparse workload): a seeded set of distinct block indices; every
  token of a needle block gets ``3 * u_g`` added to its key, where u_g is the
  unit vector along the sum of the query rows that map to kv head g.
"""
from __future__ import annotations

import numpy as np

# Stream ids: one per tensor role.
S_K, S_V, S_KSCALE, S_Q, S_KSUF, S_VSUF, S_NEEDLE = 1, 2, 3, 4, 5, 6, 7


def rng(seed: int, stream: int, *extra: int) -> np.random.Generator:
    """Independent generator for (seed, stream, *extra)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream), *map(int, extra)])))


def default_head_map(H_q: int, H_kv: int) -> np.ndarray:
    """q head h -> kv head h // (H_q / H_kv): the grouped-query convention of the workloads."""
    assert H_q % H_kv == 0
    return (np.arange(H_q) // (H_q // H_kv)).astype(np.int32)


def gen_kv(seed: int, H_kv: int, N: int, D: int, col_scale: bool = True, layer: int = 0):
    """Prefix K, V as fp16 arrays of shape [H_kv, N, D]."""
    K = rng(seed, S_K, layer).standard_normal((H_kv, N, D), dtype=np.float32)
    V = rng(seed, S_V, layer).standard_normal((H_kv, N, D), dtype=np.float32)
    if col_scale:
        f = np.exp(0.5 * rng(seed, S_KSCALE, layer).standard_normal((H_kv, 1, D))).astype(np.float32)
        K = K * f
    return K.astype(np.float16), V.astype(np.float16)


def gen_q(seed: int, H_q: int, M: int, D: int, dtype=np.float32, layer: int = 0):
    """Query rows [H_q, M, D]."""
    return rng(seed, S_Q, layer).standard_normal((H_q, M, D), dtype=np.float32).astype(dtype)


def gen_suffix(seed: int, H_kv: int, S: int, D: int, layer: int = 0):
    """Dense suffix K_suf, V_suf as fp16 [H_kv, S, D]."""
    Ks = rng(seed, S_KSUF, layer).standard_normal((H_kv, S, D), dtype=np.float32)
    Vs = rng(seed, S_VSUF, layer).standard_normal((H_kv, S, D), dtype=np.float32)
    return Ks.astype(np.float16), Vs.astype(np.float16)


def needle_blocks(seed: int, n_blocks: int, n_needles: int) -> np.ndarray:
    """Distinct needle block indices, drawn without replacement, sorted ascending."""
    return np.sort(rng(seed, S_NEEDLE).choice(n_blocks, size=n_needles, replace=False)).astype(np.int32)


def plant_needles(K: np.ndarray, Q: np.ndarray, head_map: np.ndarray, blocks: np.ndarray, B: int,
                  shift: float = 3.0) -> np.ndarray:
    """Return a copy of fp16 K [H_kv, N, D] with needle blocks pulled toward the queries.

    Q is [H_q, D] (or [H_q, 1, D]). For kv head g, u_g = normalize(sum of Q rows with
    head_map == g); every token of each needle block gets ``shift * u_g`` added.
    """
    Q2 = Q.reshape(Q.shape[0], -1).astype(np.float64)
    K2 = K.astype(np.float32).copy()
    N = K.shape[1]
    for g in range(K.shape[0]):
        u = Q2[head_map == g].sum(axis=0)
        u = u / np.linalg.norm(u)
        for b in blocks:
            t0, t1 = int(b) * B, min(N, (int(b) + 1) * B)
            K2[g, t0:t1, :] += (shift * u).astype(np.float32)
    return K2.astype(np.float16)


STRESS_KINDS = ("q30", "q100", "monotone", "dominant_prefix", "dominant_suffix", "bias_scale")


def gen_stress(kind: str, seed: int, H_q: int, H_kv: int, N: int, D: int, M: int = 1, S: int = 0,
               rise: float = 0.75, q_dtype=np.float32):
    """Inputs that push the online softmax and the number formats to their edges.

    Returns (Q [H_q, M, D] q_dtype, K, V [H_kv, N, D] fp16, K_suf, V_suf [H_kv, S, D] fp16 or None).
    Scores are only shaped through the inputs; nothing here computes attention.

    * ``q30`` / ``q100``: the standard recipe with Q multiplied by 30 or 100, so scaled logits
      reach the hundreds.
    * ``monotone``: every q head is ``8 e + 0.25 n`` for one shared unit vector e, and key t
      (prefix, then the suffix continuing the sequence) is ``c t e + 0.25 n``; c is chosen so that
      tau * q.k grows by about ``rise`` log2 units per token, so the running maximum moves all
      along the sequence.
    * ``dominant_prefix`` / ``dominant_suffix``: the same e construction with flat keys, except one
      key (a seeded prefix token, or a seeded suffix token) that gets ``b e`` added, b chosen so
      that its score exceeds the others by about 60 natural-log units.
    * ``bias_scale``: the standard recipe, except that in every kv head the first 32 dimensions of
      K and V are ``+60 + 0.02 n`` and the next 32 (when D > 32) are ``-8 + 0.004 n``: groups with
      a large bias and a tiny fp16 scale once quantised.
    """
    if kind not in STRESS_KINDS:
        raise ValueError(kind)
    r = lambda k, shape: rng(seed, 100 + k).standard_normal(shape, dtype=np.float32)
    if kind in ("q30", "q100", "bias_scale"):
        K, V = gen_kv(seed, H_kv, N, D)
        Q = gen_q(seed, H_q, M, D).astype(np.float32)
        Ks = Vs = None
        if S:
            Ks, Vs = gen_suffix(seed, H_kv, S, D)
        if kind != "bias_scale":
            Q = Q * np.float32(30.0 if kind == "q30" else 100.0)
        else:
            def shift(X):
                X = X.astype(np.float32)
                X[..., :32] = 60.0 + 0.02 * r(1 + X.shape[1], X[..., :32].shape)
                if X.shape[2] > 32:
                    X[..., 32:64] = -8.0 + 0.004 * r(2 + X.shape[1], X[..., 32:64].shape)
                return X.astype(np.float16)
            K, V = shift(K), shift(V)
            if S:
                Ks, Vs = shift(Ks), shift(Vs)
        return Q.astype(q_dtype), K, V, Ks, Vs
    e = r(3, (D,))
    e = (e / np.linalg.norm(e)).astype(np.float32)
    tau = 1.0 / np.sqrt(D)
    qa = 8.0
    Q = (qa * e[None, None, :] + 0.25 * r(4, (H_q, M, D))).astype(np.float32)
    T = N + S
    Kall = 0.25 * r(5, (H_kv, T, D))
    Vall = r(6, (H_kv, T, D))
    if kind == "monotone":
        c = rise / np.log2(np.e) / (tau * qa)          # key growth per token along e
        Kall = Kall + (c * np.arange(T, dtype=np.float32))[None, :, None] * e[None, None, :]
    else:
        b = 60.0 / (tau * qa)
        pick = rng(seed, 107)
        t_star = int(pick.integers(0, N)) if kind == "dominant_prefix" else N + int(pick.integers(0, max(S, 1)))
        if kind == "dominant_suffix" and S == 0:
            raise ValueError("dominant_suffix needs S > 0")
        Kall[:, t_star, :] += b * e[None, :]
    Kall = Kall.astype(np.float16)
    Vall = Vall.astype(np.float16)
    K, V = np.ascontiguousarray(Kall[:, :N]), np.ascontiguousarray(Vall[:, :N])
    Ks = Vs = None
    if S:
        Ks, Vs = np.ascontiguousarray(Kall[:, N:]), np.ascontiguousarray(Vall[:, N:])
    return Q.astype(q_dtype), K, V, Ks, Vs


# Workload table: the five shapes the pages' measurements are quoted on.
WORKLOADS = {
    "prefix_m1_fp16": dict(H_q=8, H_kv=8, N=2048, D=128, M=1, layers=1, fmt="fp16", S_suf=0),
    "gqa_decode_mlx4g32": dict(H_q=32, H_kv=8, N=8192, D=64, M=1, layers=16, fmt="mlx4g32", S_suf=16),
    "batched_q_prefill": dict(H_q=24, H_kv=8, N=4096, D=128, M=512, layers=28, fmt="fp16", S_suf=512),
    "sparse_topk_64k": dict(H_q=8, H_kv=2, N=65536, D=256, M=1, layers=1, fmt="fp16", S_suf=32, B=64, K_top=8),
    "cartridge_mlx4g32": dict(H_q=32, H_kv=8, N=86580, D=128, M=1, layers=36, fmt="mlx4g32", S_suf=0,
                              sessions=64, window=8192),
}


def cartridge_window_start(s: int, N: int = 86580, window: int = 8192) -> int:
    """Token offset of session s's window in the cartridge workload."""
    return (s * window) % (N - window)


def torch_gen_kv_device(seed: int, H_kv: int, N: int, D: int, device, col_scale: bool = False, layer: int = 0):
    """Large K/V generated on the device with torch's seeded generator (for sizes the host
    cannot draw quickly). Same recipe as gen_kv; different random stream than gen_kv."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1000003 + int(layer) * 7919 + 17) & 0x7FFFFFFFFFFF)
    K = torch.randn((H_kv, N, D), generator=g, device=device, dtype=torch.float32)
    V = torch.randn((H_kv, N, D), generator=g, device=device, dtype=torch.float32)
    if col_scale:
        f = torch.exp(0.5 * torch.randn((H_kv, 1, D), generator=g, device=device, dtype=torch.float32))
        K = K * f
    return K.half(), V.half()


def torch_gen_rows_device(seed: int, rows: int, cols: int, device, stream: int = 0):
    """[rows, cols] fp16 N(0,1) on the device (token-major rows, e.g. a cartridge layer)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1000003 + int(stream) * 7919 + 29) & 0x7FFFFFFFFFFF)
    return torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).half()
