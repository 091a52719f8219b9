"""Thin ctypes binding of libpck (the C ABI in include/pck.h).

Argument marshalling only: torch tensors provide device memory and the current stream; every
step of the computation runs in the CUDA library. There is no fallback: if ``libpck.so`` is
missing this module raises at import of the library.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpck.so")

OK, MISS, COLDMISS = 0, 1, 3
EINVAL, EUNSUPPORTED, ENOMEM, ECUDA = -1, -2, -3, -4
FMT_FP16, FMT_MLX4G32 = 0, 1
DT_F32, DT_F16 = 0, 1
MAX_BATCH = 64

# Every symbol include/pck.h declares.
EXPORTS = (
    "pck_create", "pck_destroy", "pck_last_error", "pck_store", "pck_store_records", "pck_lookup",
    "pck_drop", "pck_build_block_means", "pck_query", "pck_query_fused", "pck_query_sparse_auto",
    "pck_query_sparse_auto_fused", "pck_query_batch", "pck_query_sparse_batch", "pck_quantize_mlx4g32", "pck_info", "pck_sync",
    "pck_attend_records_noalloc", "pck_noalloc_status", "pck_query_sparse", "pck_get_block_means",
    "pck_dequantize_mlx4g32", "pck_query_batch_host",
)


class PckError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"pck status {code}: {msg}")
        self.code = code


class InfoT(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("slots_used", "slots_max", "cold_entries", "bytes_resident",
                                              "queries_served", "stores", "evictions")]


class QueryDesc(ctypes.Structure):
    _fields_ = [("sid", ctypes.c_char_p), ("layer", ctypes.c_int), ("Q", ctypes.c_void_p), ("O", ctypes.c_void_p),
                ("LSE", ctypes.c_void_p), ("K_suf", ctypes.c_void_p), ("V_suf", ctypes.c_void_p)]


class SparseDesc(ctypes.Structure):
    _fields_ = [("sid", ctypes.c_char_p), ("layer", ctypes.c_int), ("Q", ctypes.c_void_p), ("O", ctypes.c_void_p),
                ("LSE", ctypes.c_void_p), ("K_suf", ctypes.c_void_p), ("V_suf", ctypes.c_void_p),
                ("idx_out", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpck.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i, i64, cp = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_char_p
    sig = {
        "pck_create": (i, [ctypes.POINTER(vp), i, i]),
        "pck_destroy": (None, [vp]),
        "pck_last_error": (cp, [vp]),
        "pck_store": (i, [vp, cp, i, i, i, i, i, vp, vp, i, vp]),
        "pck_store_records": (i, [vp, cp, i, i, i, i, vp, vp, vp]),
        "pck_lookup": (i, [vp, cp, i]),
        "pck_drop": (i, [vp, cp, i, vp]),
        "pck_build_block_means": (i, [vp, cp, i, i, vp]),
        "pck_query": (i, [vp, cp, i, i, i, i, i, vp, vp, i, i, vp, vp, vp]),
        "pck_query_fused": (i, [vp, cp, i, i, i, i, i, i, i, vp, vp, vp, vp, i, i, vp, vp, vp]),
        "pck_query_sparse_auto": (i, [vp, cp, i, i, i, i, i, i, i, vp, vp, i, vp, vp, vp, vp]),
        "pck_query_sparse_auto_fused": (i, [vp, cp, i, i, i, i, i, i, i, i, vp, vp, vp, vp, i, vp, vp, vp, vp]),
        "pck_query_batch": (i, [vp, i, ctypes.POINTER(QueryDesc), i, i, i, i, i, vp, vp]),
        "pck_query_batch_host": (i, [vp, i, ctypes.POINTER(QueryDesc), i, i, i, i, i, vp, vp]),
        "pck_query_sparse_batch": (i, [vp, i, ctypes.POINTER(SparseDesc), i, i, i, i, i, i, i, vp, vp]),
        "pck_quantize_mlx4g32": (i, [vp, i, i64, i, vp, vp]),
        "pck_info": (i, [vp, ctypes.POINTER(InfoT)]),
        "pck_sync": (i, [vp, vp]),
        "pck_attend_records_noalloc": (i, [i, i, i, vp, vp, i, i, vp, vp, i, vp, vp, vp, vp, vp]),
        "pck_noalloc_status": (i, [vp, ctypes.POINTER(ctypes.c_int)]),
        "pck_query_sparse": (i, [vp, cp, i, i, i, i, i, vp, vp, vp, vp, i, vp, vp, vp]),
        "pck_get_block_means": (i, [vp, cp, i, i, vp, vp]),
        "pck_dequantize_mlx4g32": (i, [vp, i64, i, i, i, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return DT_F16
    if t.dtype == torch.float32:
        return DT_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _hm(head_map):
    if head_map is None:
        return None
    arr = (ctypes.c_int32 * len(head_map))(*[int(x) for x in head_map])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def _spec(t, name, dtype=None, numel=None, at_least=None, nbytes=None):
    """What the library will read or write through t: its dtype (one or a tuple), an exact element
    count, a minimum element count, or a minimum size in bytes."""
    return (t, name, dtype, numel, at_least, nbytes)


def _check_all(*specs, host=False):
    """Check caller tensors before their pointers reach the library, which trusts the sizes the
    call implies: dtypes and sizes of every tensor first, then contiguity, then the device (or,
    for host-buffer calls, that every tensor is page-locked host memory)."""
    live = [sp for sp in specs if sp[0] is not None]
    for t, name, dtype, numel, at_least, nbytes in live:
        if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
            raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
        if numel is not None and t.numel() != numel:
            raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")
        if at_least is not None and t.numel() < at_least:
            raise ValueError(f"{name}: {t.numel()} elements, at least {at_least} needed")
        if nbytes is not None and t.numel() * t.element_size() < nbytes:
            raise ValueError(f"{name}: {t.numel() * t.element_size()} bytes, at least {nbytes} needed")
    for t, name, *_ in live:
        if not t.is_contiguous():
            raise ValueError(f"{name}: must be contiguous")
    for t, name, *_ in live:
        if host and (t.is_cuda or not t.is_pinned()):
            raise ValueError(f"{name}: must be a pinned host tensor")
        if not host and not t.is_cuda:
            raise ValueError(f"{name}: must be on the CUDA device")


_FP = (torch.float16, torch.float32)


def _check_suffix(K_suf, V_suf, D, H_kv=None):
    if K_suf is None and V_suf is None:
        return
    if K_suf is None or V_suf is None or K_suf.dim() != 3 or V_suf.shape != K_suf.shape:
        raise ValueError("K_suf and V_suf must both be given, [H_kv, S_suf, D] of one shape")
    if K_suf.shape[2] != D or (H_kv is not None and K_suf.shape[0] != H_kv):
        raise ValueError(f"suffix shape {tuple(K_suf.shape)} does not match H_kv={H_kv}, D={D}")


def _check_descs(descs, H_q, H_kv, D, S_suf, q_dtype, sparse=False, host=False):
    """Descriptor tensors of a batched call: Q [H_q, D] of q_dtype, O (fp32) and LSE (fp32) of at
    least H_q * D and H_q elements, the suffix [H_kv, S_suf, D] fp16, idx int32 (sparse)."""
    qt = {DT_F32: torch.float32, DT_F16: torch.float16}.get(q_dtype)
    if qt is None:
        raise ValueError(f"q_dtype={q_dtype}")
    specs = []
    for i, d in enumerate(descs):
        specs += [_spec(d["Q"], f"descs[{i}].Q", qt, numel=H_q * D),
                  _spec(d["O"], f"descs[{i}].O", torch.float32, at_least=H_q * D),
                  _spec(d.get("LSE"), f"descs[{i}].LSE", torch.float32, at_least=H_q)]
        if S_suf > 0:
            for k in ("K_suf", "V_suf"):
                specs.append(_spec(d.get(k), f"descs[{i}].{k}", torch.float16, numel=H_kv * S_suf * D))
        if sparse:
            specs.append(_spec(d.get("idx"), f"descs[{i}].idx", torch.int32, at_least=H_q))
    _check_all(*specs, host=host)


def quantize_mlx4g32(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """mlx4g32 records (uint8 [rows, kv_dim/2 + kv_dim/8]) of x ([rows, kv_dim], fp16/fp32)."""
    lib = load_library()
    if x.dim() != 2:
        raise ValueError("x must be [rows, kv_dim]")
    rows, kv_dim = x.shape
    if out is None:
        out = torch.empty((rows, kv_dim // 2 + kv_dim // 8), dtype=torch.uint8, device=x.device)
    _check_all(_spec(x, "x", _FP), _spec(out, "out", nbytes=rows * (kv_dim // 2 + kv_dim // 8)))
    rc = lib.pck_quantize_mlx4g32(_ptr(x), _dt(x), rows, kv_dim, _ptr(out), _stream(stream))
    if rc != OK:
        raise PckError(rc, "pck_quantize_mlx4g32 rejected its arguments")
    return out


def dequantize_mlx4g32(records: torch.Tensor, N: int, H_kv: int, D: int, dtype=torch.float32, out=None,
                       stream=None) -> torch.Tensor:
    """Token-major mlx4g32 records [N, rec] -> [H_kv, N, D] in fp32 or fp16 (WARM / FETCH RANGE form)."""
    lib = load_library()
    if out is None:
        out = torch.empty((H_kv, N, D), dtype=dtype, device=records.device)
    kv = H_kv * D
    _check_all(_spec(records, "records", nbytes=N * (kv // 2 + kv // 8)),
               _spec(out, "out", (torch.float32, torch.float16), numel=H_kv * N * D))
    rc = lib.pck_dequantize_mlx4g32(_ptr(records), N, H_kv, D, _dt(out), _ptr(out), _stream(stream))
    if rc != OK:
        raise PckError(rc, "pck_dequantize_mlx4g32 rejected its arguments")
    return out


class Context:
    """One libpck context (slot table + workspaces) on one device."""

    def __init__(self, device: int = 0, max_slots: int = 256):
        self.lib = load_library()
        h = ctypes.c_void_p()
        torch.cuda.init()
        rc = self.lib.pck_create(ctypes.byref(h), device, max_slots)
        if rc != OK:
            raise PckError(rc, "pck_create failed")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            self.lib.pck_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def last_error(self) -> str:
        return (self.lib.pck_last_error(self.h) or b"").decode()

    def _rc(self, rc: int, ok=(OK,)):
        if rc not in ok:
            raise PckError(rc, self.last_error())
        return rc

    # ---- store / lookup / drop
    def store(self, sid: str, layer: int, K: torch.Tensor, V: torch.Tensor, fmt: int = FMT_FP16, stream=None):
        if K.dim() != 3 or V.shape != K.shape or V.dtype != K.dtype:
            raise ValueError("K and V must be [H_kv, N, D] tensors of one shape and dtype")
        _check_all(_spec(K, "K", _FP), _spec(V, "V", _FP))
        H_kv, N, D = K.shape
        return self._rc(self.lib.pck_store(self.h, sid.encode(), layer, H_kv, N, D, fmt, _ptr(K), _ptr(V), _dt(K),
                                           _stream(stream)))

    def store_records(self, sid: str, layer: int, H_kv: int, N: int, D: int, K_rec, V_rec, stream=None):
        rec = N * (H_kv * D // 2 + H_kv * D // 8)
        _check_all(_spec(K_rec, "K_rec", nbytes=rec), _spec(V_rec, "V_rec", nbytes=rec))
        return self._rc(self.lib.pck_store_records(self.h, sid.encode(), layer, H_kv, N, D, _ptr(K_rec), _ptr(V_rec),
                                                   _stream(stream)))

    def lookup(self, sid: str, layer: int) -> int:
        return self.lib.pck_lookup(self.h, sid.encode(), layer)

    def drop(self, sid: str, layer: int = -1, stream=None) -> int:
        rc = self.lib.pck_drop(self.h, sid.encode(), layer, _stream(stream))
        if rc < 0:
            raise PckError(rc, self.last_error())
        return rc

    def build_block_means(self, sid: str, layer: int, B: int, stream=None):
        return self._rc(self.lib.pck_build_block_means(self.h, sid.encode(), layer, B, _stream(stream)))

    # ---- queries (O and LSE are allocated when not given)
    def query(self, sid, layer, Q, head_map=None, top_k=0, fa_window=0, O=None, LSE=None, want_lse=True, stream=None):
        if Q.dim() != 3:
            raise ValueError("Q must be [H_q, M, D]")
        H_q, M, D = Q.shape
        O = torch.empty((H_q, M, D), dtype=torch.float32, device=Q.device) if O is None else O
        if LSE is None and want_lse:
            LSE = torch.empty((H_q, M), dtype=torch.float32, device=Q.device)
        _check_all(_spec(Q, "Q", _FP), _spec(O, "O", torch.float32, at_least=H_q * M * D),
                   _spec(LSE, "LSE", torch.float32, at_least=H_q * M))
        hm = _hm(head_map)
        self._rc(self.lib.pck_query(self.h, sid.encode(), layer, H_q, D, M, _dt(Q), _ptr(Q), hm[0] if hm else None,
                                    top_k, fa_window, _ptr(O), _ptr(LSE), _stream(stream)))
        return O, LSE

    def query_fused(self, sid, layer, Q, K_suf, V_suf, head_map=None, causal=True, fa_window=0, O=None, LSE=None,
                    want_lse=True, stream=None):
        if Q.dim() != 3:
            raise ValueError("Q must be [H_q, M, D]")
        H_q, M, D = Q.shape
        if K_suf is None:
            raise ValueError("query_fused needs K_suf and V_suf")
        _check_suffix(K_suf, V_suf, D)
        H_kv, S_suf, _ = K_suf.shape
        O = torch.empty((H_q, M, D), dtype=torch.float32, device=Q.device) if O is None else O
        if LSE is None and want_lse:
            LSE = torch.empty((H_q, M), dtype=torch.float32, device=Q.device)
        _check_all(_spec(Q, "Q", _FP), _spec(K_suf, "K_suf", torch.float16), _spec(V_suf, "V_suf", torch.float16),
                   _spec(O, "O", torch.float32, at_least=H_q * M * D),
                   _spec(LSE, "LSE", torch.float32, at_least=H_q * M))
        hm = _hm(head_map)
        self._rc(self.lib.pck_query_fused(self.h, sid.encode(), layer, H_q, D, M, S_suf, H_kv, _dt(Q), _ptr(Q),
                                          _ptr(K_suf), _ptr(V_suf), hm[0] if hm else None, int(bool(causal)),
                                          fa_window, _ptr(O), _ptr(LSE), _stream(stream)))
        return O, LSE

    def query_sparse_auto(self, sid, layer, Q, B, K_top, H_kv, head_map=None, K_suf=None, V_suf=None, fa_window=0,
                          O=None, LSE=None, idx=None, stream=None):
        H_q, D = Q.shape[0], Q.shape[-1]
        _check_suffix(K_suf, V_suf, D, H_kv)
        O = torch.empty((H_q, D), dtype=torch.float32, device=Q.device) if O is None else O
        LSE = torch.empty((H_q,), dtype=torch.float32, device=Q.device) if LSE is None else LSE
        if idx is None:   # the library writes [H_q, min(K_top, n_blocks)] contiguously
            idx = torch.empty((H_q, K_top), dtype=torch.int32, device=Q.device)
        _check_all(_spec(Q, "Q", _FP, numel=H_q * D), _spec(K_suf, "K_suf", torch.float16),
                   _spec(V_suf, "V_suf", torch.float16), _spec(O, "O", torch.float32, at_least=H_q * D),
                   _spec(LSE, "LSE", torch.float32, at_least=H_q), _spec(idx, "idx", torch.int32, at_least=H_q))
        hm = _hm(head_map)
        if K_suf is None:
            rc = self.lib.pck_query_sparse_auto(self.h, sid.encode(), layer, H_q, D, B, K_top, H_kv, _dt(Q), _ptr(Q),
                                                hm[0] if hm else None, fa_window, _ptr(O), _ptr(LSE), _ptr(idx),
                                                _stream(stream))
        else:
            rc = self.lib.pck_query_sparse_auto_fused(self.h, sid.encode(), layer, H_q, D, B, K_top, H_kv,
                                                      K_suf.shape[1], _dt(Q), _ptr(Q), _ptr(K_suf), _ptr(V_suf),
                                                      hm[0] if hm else None, fa_window, _ptr(O), _ptr(LSE), _ptr(idx),
                                                      _stream(stream))
        self._rc(rc)
        return O, LSE, idx

    def query_sparse(self, sid, layer, Q, indices, counts, head_map=None, fa_window=0, O=None, LSE=None,
                     stream=None):
        """QUERY_SPARSE: Q [H_q, D] (device); indices [H_q, K_sparse_max] and counts [H_q], host
        integer arrays (positions in the prefix); returns (O [H_q, D], LSE [H_q])."""
        import numpy as np
        H_q, D = Q.shape[0], Q.shape[-1]
        idx = np.ascontiguousarray(indices, dtype=np.int32)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        if idx.ndim != 2 or idx.shape[0] != H_q or cnt.shape != (H_q,):
            raise ValueError("indices must be [H_q, K_sparse_max] and counts [H_q]")
        O = torch.empty((H_q, D), dtype=torch.float32, device=Q.device) if O is None else O
        LSE = torch.empty((H_q,), dtype=torch.float32, device=Q.device) if LSE is None else LSE
        _check_all(_spec(Q, "Q", _FP, numel=H_q * D), _spec(O, "O", torch.float32, at_least=H_q * D),
                   _spec(LSE, "LSE", torch.float32, at_least=H_q))
        hm = _hm(head_map)
        self._rc(self.lib.pck_query_sparse(self.h, sid.encode(), layer, H_q, D, idx.shape[1], _dt(Q), _ptr(Q),
                                           idx.ctypes.data_as(ctypes.c_void_p), cnt.ctypes.data_as(ctypes.c_void_p),
                                           hm[0] if hm else None, fa_window, _ptr(O), _ptr(LSE), _stream(stream)))
        return O, LSE

    def get_block_means(self, sid, layer, B, H_kv, N, D, stream=None):
        """The slot's block means, fp32 [H_kv, ceil(N/B), D] (device)."""
        out = torch.empty((H_kv, (N + B - 1) // B, D), dtype=torch.float32, device="cuda")
        self._rc(self.lib.pck_get_block_means(self.h, sid.encode(), layer, B, _ptr(out), _stream(stream)))
        return out

    def sparse_batch_caller(self, descs, H_q, H_kv, D, B, K_top, S_suf=0, q_dtype=DT_F32, head_map=None):
        """Prebuild a pck_query_sparse_batch call over descs (dicts with sid, layer, Q, O, and
        optionally LSE, K_suf, V_suf, idx); returns a no-argument callable issuing it on the
        current stream (cheap enough to capture in a CUDA graph)."""
        _check_descs(descs, H_q, H_kv, D, S_suf, q_dtype, sparse=True)
        n = len(descs)
        arr = (SparseDesc * n)()
        keep = []
        opt = lambda d, k: d[k].data_ptr() if d.get(k) is not None else None
        for i, d in enumerate(descs):
            sid = d["sid"].encode()
            keep.append(sid)
            arr[i] = SparseDesc(sid, d["layer"], d["Q"].data_ptr(), d["O"].data_ptr(), opt(d, "LSE"), opt(d, "K_suf"),
                                opt(d, "V_suf"), opt(d, "idx"))
        hm = _hm(head_map)
        fn, h = self.lib.pck_query_sparse_batch, self.h

        def call():
            rc = fn(h, n, arr, H_q, H_kv, D, B, K_top, S_suf, q_dtype, hm[0] if hm else None, _stream(None))
            if rc != OK:
                raise PckError(rc, self.last_error())
        call._keep = (arr, keep, hm)
        return call

    def query_sparse_batch(self, descs, H_q, H_kv, D, B, K_top, S_suf=0, q_dtype=DT_F32, head_map=None):
        """n sparse queries in one scoring, one selection and one gather-decode launch (plus its
        merge); see sparse_batch_caller."""
        self.sparse_batch_caller(descs, H_q, H_kv, D, B, K_top, S_suf, q_dtype, head_map)()

    def query_batch(self, descs, H_q, H_kv, D, S_suf=0, q_dtype=DT_F32, head_map=None, stream=None):
        """descs: list of dicts with sid, layer, Q, O, LSE (optional), K_suf/V_suf (optional)."""
        _check_descs(descs, H_q, H_kv, D, S_suf, q_dtype)
        n = len(descs)
        arr = (QueryDesc * n)()
        keep = []
        for i, d in enumerate(descs):
            sid = d["sid"].encode()
            keep.append(sid)
            arr[i] = QueryDesc(sid, d["layer"], d["Q"].data_ptr(), d["O"].data_ptr(),
                               d["LSE"].data_ptr() if d.get("LSE") is not None else None,
                               d["K_suf"].data_ptr() if d.get("K_suf") is not None else None,
                               d["V_suf"].data_ptr() if d.get("V_suf") is not None else None)
        hm = _hm(head_map)
        return self._rc(self.lib.pck_query_batch(self.h, n, arr, H_q, H_kv, D, S_suf, q_dtype, hm[0] if hm else None,
                                                 _stream(stream)))

    def batch_caller(self, descs, H_q, H_kv, D, S_suf=0, q_dtype=DT_F32, head_map=None, host=False):
        """Prebuild the descriptor array of a pck_query_batch call; returns a no-argument callable
        that issues the call on the current stream (cheap enough to capture in a CUDA graph).
        host=True: the descriptors' tensors are pinned host tensors and the call is
        pck_query_batch_host (the library moves the bytes)."""
        _check_descs(descs, H_q, H_kv, D, S_suf, q_dtype, host=host)
        n = len(descs)
        arr = (QueryDesc * n)()
        keep = []
        for i, d in enumerate(descs):
            sid = d["sid"].encode()
            keep.append(sid)
            arr[i] = QueryDesc(sid, d["layer"], d["Q"].data_ptr(), d["O"].data_ptr(),
                               d["LSE"].data_ptr() if d.get("LSE") is not None else None,
                               d["K_suf"].data_ptr() if d.get("K_suf") is not None else None,
                               d["V_suf"].data_ptr() if d.get("V_suf") is not None else None)
        hm = _hm(head_map)
        fn, h = self.lib.pck_query_batch_host if host else self.lib.pck_query_batch, self.h

        def call():
            rc = fn(h, n, arr, H_q, H_kv, D, S_suf, q_dtype, hm[0] if hm else None, _stream(None))
            if rc != OK:
                raise PckError(rc, self.last_error())
        call._keep = (arr, keep, hm)
        return call

    def info(self) -> dict:
        out = InfoT()
        self._rc(self.lib.pck_info(self.h, ctypes.byref(out)))
        return {n: getattr(out, n) for n, _ in InfoT._fields_}

    def sync(self, stream=None):
        return self._rc(self.lib.pck_sync(self.h, _stream(stream)))
