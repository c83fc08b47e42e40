"""fp64 CPU oracle for paged attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, one thread per output row);
this module only compiles it with gcc, loads it with ctypes and marshals numpy arrays.
See ``attn_oracle.c`` for the definitions it follows and their sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

__all__ = ["build", "lib_path", "decode", "prefill", "decode_split_partials", "partial_ranges", "combine",
           "kv_append", "masked", "load_variant"]


def _compile(src: str, out: str, extra: Sequence[str] = ()) -> None:
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", out, src, "-lm", "-lpthread", *extra]
    subprocess.run(cmd, check=True)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so next to it (skipped when up to date)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        _compile(_SRC, tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib_path() -> str:
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_D = ctypes.c_double


def _declare(lib):
    lib.oracle_decode_rows.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _L, _P, _D, _L, _P, _P, _P, _I]
    lib.oracle_prefill_rows.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _L, _P, _D, _L, _P, _P, _P, _I]
    lib.oracle_decode_split_partials.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _L, _P, _D, _I, _P, _P, _I]
    lib.oracle_combine.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P]
    lib.oracle_kv_append.argtypes = [_I, _I, _I, _P, _P, _P, _L, _P, _P, _P, _P]
    lib.oracle_masked_rows.argtypes = [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _L, _P, _D, _P, _I, _L, _L, _I, _L,
                                       _P, _P, _P, _I]
    lib.oracle_partial_ranges.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _L, _D, _L, _P, _P, _P, _P, _P, _P, _I]
    for f in ("oracle_decode_rows", "oracle_prefill_rows", "oracle_decode_split_partials", "oracle_combine",
              "oracle_partial_ranges", "oracle_kv_append", "oracle_masked_rows"):
        getattr(lib, f).restype = None
    return lib


def _get():
    global _lib
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def load_variant(path: str):
    """Load another compiled copy of the oracle (used by the mutation tests)."""
    return _declare(ctypes.CDLL(path))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _threads(n: Optional[int]) -> int:
    return int(n) if n else (os.cpu_count() or 1)


def decode(w, rows: Optional[np.ndarray] = None, nthreads: Optional[int] = None, lib=None) -> np.ndarray:
    """Decode attention of workload ``w``.

    ``rows`` is an int array [n, 2] of (b, h) pairs; default every pair, returned as [B, Hq, d].
    With ``rows`` given, returns [n, d] in the order listed.
    """
    lib = lib or _get()
    B, Hq, Hkv, D = w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim
    full = rows is None
    if full:
        bb, hh = np.meshgrid(np.arange(B, dtype=np.int32), np.arange(Hq, dtype=np.int32), indexing="ij")
        rows = np.stack([bb.ravel(), hh.ravel()], axis=1)
    rows = _c(rows, np.int32)
    ib, ih = _c(rows[:, 0], np.int32), _c(rows[:, 1], np.int32)
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    q, kp, vp = _c(w.q, np.uint16), _c(w.k_pool, np.uint16), _c(w.v_pool, np.uint16)
    r2t, sl = _c(w.req_to_token, np.int32), _c(w.seq_lens, np.int32)
    lib.oracle_decode_rows(B, Hq, Hkv, D, _ptr(q), _ptr(kp), _ptr(vp), _ptr(r2t), r2t.shape[1], _ptr(sl),
                           float(w.sm_scale), rows.shape[0], _ptr(ib), _ptr(ih), _ptr(out), _threads(nthreads))
    return out.reshape(B, Hq, D) if full else out


def prefill(w, rows: Optional[np.ndarray] = None, nthreads: Optional[int] = None, lib=None) -> np.ndarray:
    """Ragged prefill attention of workload ``w``.

    ``rows`` is an int array [n, 2] of (flat query row, h) pairs; default every pair,
    returned as [total_q, Hq, d].  With ``rows`` given, returns [n, d].
    """
    lib = lib or _get()
    B, Hq, Hkv, D = w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim
    TQ = int(w.q.shape[0])
    full = rows is None
    if full:
        rr, hh = np.meshgrid(np.arange(TQ, dtype=np.int32), np.arange(Hq, dtype=np.int32), indexing="ij")
        rows = np.stack([rr.ravel(), hh.ravel()], axis=1)
    rows = _c(rows, np.int32)
    ir, ih = _c(rows[:, 0], np.int32), _c(rows[:, 1], np.int32)
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    q, kp, vp = _c(w.q, np.uint16), _c(w.k_pool, np.uint16), _c(w.v_pool, np.uint16)
    qo, r2t, sl = _c(w.qo_indptr, np.int32), _c(w.req_to_token, np.int32), _c(w.seq_lens, np.int32)
    lib.oracle_prefill_rows(B, Hq, Hkv, D, _ptr(q), _ptr(qo), _ptr(kp), _ptr(vp), _ptr(r2t), r2t.shape[1],
                            _ptr(sl), float(w.sm_scale), rows.shape[0], _ptr(ir), _ptr(ih), _ptr(out),
                            _threads(nthreads))
    return out.reshape(TQ, Hq, D) if full else out


def decode_split_partials(w, S: int, nthreads: Optional[int] = None, lib=None):
    """Even S-way split-KV partials: (o_part [B,Hq,S,d], ml_part [B,Hq,S,2]) in fp64."""
    lib = lib or _get()
    B, Hq, Hkv, D = w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim
    o = np.zeros((B, Hq, S, D), dtype=np.float64)
    ml = np.zeros((B, Hq, S, 2), dtype=np.float64)
    q, kp, vp = _c(w.q, np.uint16), _c(w.k_pool, np.uint16), _c(w.v_pool, np.uint16)
    r2t, sl = _c(w.req_to_token, np.int32), _c(w.seq_lens, np.int32)
    lib.oracle_decode_split_partials(B, Hq, Hkv, D, _ptr(q), _ptr(kp), _ptr(vp), _ptr(r2t), r2t.shape[1],
                                     _ptr(sl), float(w.sm_scale), int(S), _ptr(o), _ptr(ml), _threads(nthreads))
    return o, ml


def partial_ranges(w, items, nthreads: Optional[int] = None, lib=None):
    """Split partials over explicit key ranges: ``items`` is an int array [n, 4] of
    (b, h, lo, hi) -- query head h of request b over its keys lo .. hi-1.

    Returns (o [n, d], ml [n, 2]) in fp64: o unnormalised, ml = (max logit, sum of exp);
    an empty range gives (0, -inf, 0).
    """
    lib = lib or _get()
    B, Hq, Hkv, D = w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim
    items = np.asarray(items, dtype=np.int64).reshape(-1, 4)
    ib, ih = _c(items[:, 0], np.int32), _c(items[:, 1], np.int32)
    lo, hi = _c(items[:, 2], np.int64), _c(items[:, 3], np.int64)
    n = items.shape[0]
    o = np.zeros((n, D), dtype=np.float64)
    ml = np.zeros((n, 2), dtype=np.float64)
    q, kp, vp = _c(w.q, np.uint16), _c(w.k_pool, np.uint16), _c(w.v_pool, np.uint16)
    r2t = _c(w.req_to_token, np.int32)
    lib.oracle_partial_ranges(B, Hq, Hkv, D, _ptr(q), _ptr(kp), _ptr(vp), _ptr(r2t), r2t.shape[1],
                              float(w.sm_scale), n, _ptr(ib), _ptr(ih), _ptr(lo), _ptr(hi), _ptr(o), _ptr(ml),
                              _threads(nthreads))
    return o, ml


def combine(o_part: np.ndarray, ml_part: np.ndarray, nsplit: Optional[np.ndarray] = None, lib=None) -> np.ndarray:
    """Log-sum-exp combine of split partials; ``nsplit[b]`` limits the splits read per request."""
    lib = lib or _get()
    o_part = _c(o_part, np.float64)
    ml_part = _c(ml_part, np.float64)
    B, Hq, S, D = o_part.shape
    ns = None if nsplit is None else _c(nsplit, np.int32)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lib.oracle_combine(B, Hq, S, D, _ptr(o_part), _ptr(ml_part), _ptr(ns), _ptr(out))
    return out


def kv_append(w, qo_indptr, k_new: np.ndarray, v_new: np.ndarray, lib=None):
    """KV append: the pools of ``w`` after writing new token i of request b into slot
    ``req_to_token[b, seq_len_b - q_len_b + i]``.  ``qo_indptr`` [B+1] gives the new rows of
    each request in ``k_new`` / ``v_new`` [total_q, Hkv, d] (bf16 bits).  Returns new arrays
    (k_pool, v_pool); ``w`` is not modified."""
    lib = lib or _get()
    B, Hkv, D = w.batch, w.num_kv_heads, w.head_dim
    kp, vp = np.array(w.k_pool, dtype=np.uint16, order="C"), np.array(w.v_pool, dtype=np.uint16, order="C")
    qo, sl, r2t = _c(qo_indptr, np.int32), _c(w.seq_lens, np.int32), _c(w.req_to_token, np.int32)
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    lib.oracle_kv_append(B, Hkv, D, _ptr(qo), _ptr(sl), _ptr(r2t), r2t.shape[1], _ptr(kn), _ptr(vn), _ptr(kp),
                         _ptr(vp))
    return kp, vp


def masked(w, mask: np.ndarray, causal: bool = True, rows: Optional[np.ndarray] = None,
           nthreads: Optional[int] = None, lib=None) -> np.ndarray:
    """Attention of workload ``w`` with an explicit mask: ``mask`` is uint8/bool, 2-D
    [B, kv_pitch] or 3-D [B, q_pitch, kv_pitch] (nonzero = visible).  Prefill workloads also
    take ``causal`` (False: every row sees all seq_len keys the mask leaves).  ``rows`` as
    for ``decode`` / ``prefill``; default every row, returned as [rows, Hq, d]."""
    lib = lib or _get()
    B, Hq, Hkv, D = w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim
    is_decode = w.kind == "decode"
    n_rows = B if is_decode else int(w.q.shape[0])
    full = rows is None
    if full:
        rr, hh = np.meshgrid(np.arange(n_rows, dtype=np.int32), np.arange(Hq, dtype=np.int32), indexing="ij")
        rows = np.stack([rr.ravel(), hh.ravel()], axis=1)
    rows = _c(rows, np.int32)
    ir, ih = _c(rows[:, 0], np.int32), _c(rows[:, 1], np.int32)
    m = _c(np.asarray(mask).astype(np.uint8), np.uint8)
    if m.ndim not in (2, 3) or m.shape[0] != B:
        raise ValueError("mask must be [B, kv_pitch] or [B, q_pitch, kv_pitch]")
    kv_pitch, q_pitch = m.shape[-1], (m.shape[1] if m.ndim == 3 else 0)
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    q, kp, vp = _c(w.q, np.uint16), _c(w.k_pool, np.uint16), _c(w.v_pool, np.uint16)
    r2t, sl = _c(w.req_to_token, np.int32), _c(w.seq_lens, np.int32)
    qo = None if is_decode else _c(w.qo_indptr, np.int32)
    lib.oracle_masked_rows(int(is_decode), B, Hq, Hkv, D, _ptr(q), _ptr(qo), _ptr(kp), _ptr(vp), _ptr(r2t),
                           r2t.shape[1], _ptr(sl), float(w.sm_scale), _ptr(m), int(m.ndim), kv_pitch, q_pitch,
                           int(bool(causal)), rows.shape[0], _ptr(ir), _ptr(ih), _ptr(out), _threads(nthreads))
    return out.reshape(n_rows, Hq, D) if full else out
