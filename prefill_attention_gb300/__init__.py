"""Python binding of libastr_attn.so: GB300 paged decode and ragged prefill attention.

This module only marshals arguments: it takes device tensors (PyTorch is used for device
memory and streams), passes their pointers and shapes to the C ABI declared in
``include/astr_attn.h`` and returns the status code.  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback.  If the library has
not been built, importing succeeds but every call raises ``RuntimeError``.

Function names mirror the C entry points.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

__all__ = [
    "Dims", "AstrAttnError", "load", "lib_path", "make_dims",
    "astr_attn_paged_decode", "astr_attn_decode_split", "astr_attn_decode_combine", "astr_attn_prefill_ragged",
    "astr_attn_paged_decode_noalloc", "astr_attn_kv_append", "astr_attn_paged_decode_masked",
    "astr_attn_prefill_ragged_masked", "Mask", "make_mask", "KvLayout", "make_kv_layout",
    "astr_attn_decode_contiguous", "astr_attn_prefill_contiguous", "QoLayout", "make_qo_layout",
    "astr_attn_decode_strided", "astr_attn_prefill_strided", "astr_attn_decode_num_splits", "astr_attn_decode_workspace_bytes", "astr_attn_status_string",
    "astr_attn_version", "alloc_decode_workspace",
    "ASTR_OK", "ASTR_ERR_INVALID_ARG", "ASTR_ERR_UNSUPPORTED", "ASTR_ERR_MISALIGNED",
    "ASTR_ERR_WORKSPACE_TOO_SMALL", "ASTR_ERR_LAUNCH_FAILED", "ASTR_ERR_DEVICE", "EXPORTED_SYMBOLS",
    "ASTR_KSTATUS_TIMEOUT", "ASTR_KSTATUS_BAD_INPUT", "ASTR_KSTATUS_SMEM", "ASTR_KSTATUS_RANGE",
    "ASTR_KSTATUS_PLAN", "astr_attn_prefill_plan", "make_prefill_plan", "attach_prefill_plan",
    "ASTR_DIMS_STABLE_INDICES",
]

ASTR_OK = 0
ASTR_ERR_INVALID_ARG = -1
ASTR_ERR_UNSUPPORTED = -2
ASTR_ERR_MISALIGNED = -3
ASTR_ERR_WORKSPACE_TOO_SMALL = -4
ASTR_ERR_LAUNCH_FAILED = -5
ASTR_ERR_DEVICE = -6

# bits of the status word (dims.status)
ASTR_KSTATUS_TIMEOUT = 1
ASTR_KSTATUS_BAD_INPUT = 2
ASTR_KSTATUS_SMEM = 4
ASTR_KSTATUS_RANGE = 8
ASTR_KSTATUS_PLAN = 16

# dims.flags
ASTR_DIMS_STABLE_INDICES = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libastr_attn.so")
_lib = None

EXPORTED_SYMBOLS = [
    "astr_attn_decode_num_splits", "astr_attn_decode_workspace_bytes", "astr_attn_paged_decode",
    "astr_attn_decode_combine", "astr_attn_prefill_ragged", "astr_attn_status_string", "astr_attn_version",
    "astr_attn_decode_split", "astr_attn_paged_decode_noalloc", "astr_attn_kv_append",
    "astr_attn_paged_decode_masked", "astr_attn_prefill_ragged_masked", "astr_attn_decode_contiguous",
    "astr_attn_prefill_contiguous", "astr_attn_decode_strided", "astr_attn_prefill_strided",
    "astr_attn_prefill_plan",
]


class AstrAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({astr_attn_status_string(status)})")
        self.status = status


class Dims(ctypes.Structure):
    """Mirror of ``astr_attn_dims`` (see include/astr_attn.h for the meaning of each field)."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("num_slots", ctypes.c_int64), ("r2t_stride", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32), ("total_q", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
        ("max_splits", ctypes.c_int32), ("num_splits", ctypes.c_int32),
        ("status", ctypes.c_void_p), ("wait_limit", ctypes.c_uint32),
        ("prefill_plan", ctypes.c_void_p), ("prefill_plan_words", ctypes.c_int64),
        ("flags", ctypes.c_uint32),
    ]


class Mask(ctypes.Structure):
    """Mirror of ``astr_attn_mask`` (see include/astr_attn.h)."""
    _fields_ = [("mask", ctypes.c_void_p), ("dims", ctypes.c_int32), ("kv_pitch", ctypes.c_int32),
                ("q_pitch", ctypes.c_int32), ("causal", ctypes.c_int32)]


def make_mask(mask=None, causal: bool = True) -> Mask:
    """Mask struct for a device uint8/bool tensor of shape [B, kv_pitch] or [B, q_pitch, kv_pitch]
    (or None: no explicit mask, only the causal flag)."""
    if mask is None:
        return Mask(None, 0, 0, 0, int(bool(causal)))
    shape = tuple(mask.shape)
    if len(shape) not in (2, 3):
        raise ValueError("mask must be [B, kv_pitch] or [B, q_pitch, kv_pitch]")
    return Mask(int(mask.data_ptr()), len(shape), int(shape[-1]), int(shape[1]) if len(shape) == 3 else 0,
                int(bool(causal)))


class KvLayout(ctypes.Structure):
    """Mirror of ``astr_attn_kv_layout`` (strides in elements; see include/astr_attn.h)."""
    _fields_ = [("batch_stride", ctypes.c_int64), ("token_stride", ctypes.c_int64), ("head_stride", ctypes.c_int64)]


def make_kv_layout(cache) -> KvLayout:
    """Layout of a contiguous K/V cache tensor given with its logical dims ordered
    [batch, position, kv_head, head_dim] (a "blhd" tensor as is, a "bhld" one as
    ``cache.transpose(1, 2)``): the strides are read from the tensor, no copy is made."""
    sb, sl, sh, se = (int(x) for x in cache.stride())
    if se != 1:
        raise ValueError("head_dim must be the contiguous dimension")
    return KvLayout(sb, sl, sh)


class QoLayout(ctypes.Structure):
    """Mirror of ``astr_attn_qo_layout`` (strides in elements; see include/astr_attn.h)."""
    _fields_ = [("q_batch_stride", ctypes.c_int64), ("q_token_stride", ctypes.c_int64),
                ("q_head_stride", ctypes.c_int64), ("o_batch_stride", ctypes.c_int64),
                ("o_token_stride", ctypes.c_int64), ("o_head_stride", ctypes.c_int64)]


def make_qo_layout(q, out, padded: bool) -> QoLayout:
    """Strides of query / output tensors given with logical dims [rows, Hq, d] (packed; padded
    = False) or [B, L, Hq, d] (padded per request; a "bhld" tensor as ``t.transpose(1, 2)``),
    read from the tensors themselves (no copy)."""
    def strides(t):
        st = [int(x) for x in t.stride()]
        if st[-1] != 1:
            raise ValueError("head_dim must be the contiguous dimension")
        return (st[0], st[1], st[2]) if padded else (0, st[0], st[1])
    return QoLayout(*strides(q), *strides(out))


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libastr_attn.so (built by ``prefill_attention_gb300.build``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is not built; run `python -m prefill_attention_gb300.build` "
                           "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I32, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    D = ctypes.POINTER(Dims)
    lib.astr_attn_decode_num_splits.argtypes = [D, I32, ctypes.POINTER(ctypes.c_int)]
    lib.astr_attn_decode_workspace_bytes.argtypes = [D, ctypes.POINTER(ctypes.c_size_t),
                                                     ctypes.POINTER(ctypes.c_size_t)]
    lib.astr_attn_paged_decode.argtypes = [P, P, P, P, P, P, P, P, P, D, F, P]
    lib.astr_attn_decode_split.argtypes = [P, P, P, P, P, P, P, P, D, F, P]
    lib.astr_attn_decode_combine.argtypes = [P, P, P, P, P, D, P]
    lib.astr_attn_paged_decode_noalloc.argtypes = [P, P, P, P, P, P, P, D, F, P]
    lib.astr_attn_prefill_ragged.argtypes = [P, P, P, P, P, P, P, P, D, F, P]
    lib.astr_attn_kv_append.argtypes = [P, P, P, P, P, P, P, D, P]
    M = ctypes.POINTER(Mask)
    lib.astr_attn_paged_decode_masked.argtypes = [P, P, P, P, P, P, M, P, P, P, D, F, P]
    lib.astr_attn_prefill_ragged_masked.argtypes = [P, P, P, P, P, P, P, M, P, D, F, P]
    LY = ctypes.POINTER(KvLayout)
    lib.astr_attn_decode_contiguous.argtypes = [P, P, P, LY, P, P, M, P, P, P, D, F, P]
    lib.astr_attn_prefill_contiguous.argtypes = [P, P, P, P, LY, P, P, M, P, D, F, P]
    QL = ctypes.POINTER(QoLayout)
    lib.astr_attn_decode_strided.argtypes = [P, P, P, P, LY, QL, P, P, M, P, P, P, D, F, P]
    lib.astr_attn_prefill_strided.argtypes = [P, P, P, P, P, LY, QL, P, P, M, P, D, F, P]
    SZ = ctypes.c_size_t
    lib.astr_attn_prefill_plan.argtypes = [P, P, D, I32, I32, I32, P, SZ, ctypes.POINTER(SZ)]
    lib.astr_attn_status_string.argtypes = [I32]
    lib.astr_attn_status_string.restype = ctypes.c_char_p
    lib.astr_attn_version.argtypes = []
    for f in ("astr_attn_decode_num_splits", "astr_attn_decode_workspace_bytes", "astr_attn_paged_decode",
              "astr_attn_decode_split", "astr_attn_decode_combine", "astr_attn_prefill_ragged", "astr_attn_version",
              "astr_attn_paged_decode_noalloc", "astr_attn_kv_append", "astr_attn_paged_decode_masked",
              "astr_attn_prefill_ragged_masked", "astr_attn_decode_contiguous", "astr_attn_prefill_contiguous",
              "astr_attn_decode_strided", "astr_attn_prefill_strided", "astr_attn_prefill_plan"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def make_dims(batch, num_qo_heads, num_kv_heads, head_dim, num_slots, r2t_stride, max_seq_len, total_q=0,
              max_q_len=0, max_splits=1, num_splits=0, status=None, wait_limit=0, flags=0) -> Dims:
    """``status``: optional device int32 tensor (or pointer) the kernels OR their ASTR_KSTATUS_*
    bits into; ``wait_limit``: polls per pipeline wait before a kernel gives up (0 = default);
    ``flags``: ASTR_DIMS_* bits (see include/astr_attn.h)."""
    d = Dims(int(batch), int(num_qo_heads), int(num_kv_heads), int(head_dim), int(num_slots), int(r2t_stride),
             int(max_seq_len), int(total_q), int(max_q_len), int(max_splits), int(num_splits), _ptr(status),
             int(wait_limit))
    d.flags = int(flags)
    return d


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int, where: str, check: bool) -> int:
    if check and status != ASTR_OK:
        raise AstrAttnError(status, where)
    return status


def astr_attn_status_string(status: int) -> str:
    return load().astr_attn_status_string(int(status)).decode()


def astr_attn_version() -> int:
    return int(load().astr_attn_version())


def astr_attn_decode_num_splits(dims: Dims, device: int = 0, check: bool = True) -> int:
    n = ctypes.c_int(0)
    st = load().astr_attn_decode_num_splits(ctypes.byref(dims), int(device), ctypes.byref(n))
    _check(st, "astr_attn_decode_num_splits", check)
    return n.value if st == ASTR_OK else st


def astr_attn_decode_workspace_bytes(dims: Dims, check: bool = True):
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = load().astr_attn_decode_workspace_bytes(ctypes.byref(dims), ctypes.byref(a), ctypes.byref(b))
    _check(st, "astr_attn_decode_workspace_bytes", check)
    return (a.value, b.value) if st == ASTR_OK else st


def astr_attn_paged_decode(q, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, o_part, ml_part, out,
                           dims: Dims, sm_scale: float, stream=None, check: bool = True) -> int:
    """Split-KV paged decode; arrays are device tensors (or raw device pointers as ints)."""
    st = load().astr_attn_paged_decode(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(req_to_token), _ptr(seq_lens),
                                       _ptr(kv_indptr), _ptr(o_part), _ptr(ml_part), _ptr(out), ctypes.byref(dims),
                                       float(sm_scale), _stream(stream))
    return _check(st, "astr_attn_paged_decode", check)


def astr_attn_decode_split(q, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, o_part, ml_part, dims: Dims,
                           sm_scale: float, stream=None, check: bool = True) -> int:
    """The split kernel alone (writes o_part / ml_part)."""
    st = load().astr_attn_decode_split(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(req_to_token), _ptr(seq_lens),
                                       _ptr(kv_indptr), _ptr(o_part), _ptr(ml_part), ctypes.byref(dims),
                                       float(sm_scale), _stream(stream))
    return _check(st, "astr_attn_decode_split", check)


def astr_attn_paged_decode_noalloc(q, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, out, dims: Dims,
                                   sm_scale: float, stream=None, check: bool = True) -> int:
    """Paged decode with the split partials in the library's own fixed device array.

    For callers that cannot pass a workspace (see include/astr_attn.h): no allocation
    happens anywhere in the call.  Calls that overlap on the GPU share the array and race.
    """
    st = load().astr_attn_paged_decode_noalloc(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(req_to_token),
                                               _ptr(seq_lens), _ptr(kv_indptr), _ptr(out), ctypes.byref(dims),
                                               float(sm_scale), _stream(stream))
    return _check(st, "astr_attn_paged_decode_noalloc", check)


def astr_attn_decode_combine(o_part, ml_part, seq_lens, kv_indptr, out, dims: Dims, stream=None,
                             check: bool = True) -> int:
    st = load().astr_attn_decode_combine(_ptr(o_part), _ptr(ml_part), _ptr(seq_lens), _ptr(kv_indptr), _ptr(out),
                                         ctypes.byref(dims), _stream(stream))
    return _check(st, "astr_attn_decode_combine", check)


def astr_attn_prefill_ragged(q, qo_indptr, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, out, dims: Dims,
                             sm_scale: float, stream=None, check: bool = True) -> int:
    st = load().astr_attn_prefill_ragged(_ptr(q), _ptr(qo_indptr), _ptr(k_pool), _ptr(v_pool), _ptr(req_to_token),
                                         _ptr(seq_lens), _ptr(kv_indptr), _ptr(out), ctypes.byref(dims),
                                         float(sm_scale), _stream(stream))
    return _check(st, "astr_attn_prefill_ragged", check)


def astr_attn_prefill_plan(qo_indptr_host, seq_lens_host, dims: Dims, causal: bool = True, num_ctas: int = 0,
                           device: int = 0, check: bool = True):
    """Host work plan for the prefill calls of one batch (``astr_attn_prefill_plan``): returns the
    plan as a numpy int32 array, or None when no plan applies (UNSUPPORTED).  ``qo_indptr_host``
    and ``seq_lens_host`` are host arrays (numpy, lists or CPU tensors) equal to the call's."""
    import numpy as np

    def host(a):
        if hasattr(a, "detach"):  # a torch tensor (on any device): its values on the host
            a = a.detach().cpu().numpy()
        return np.ascontiguousarray(np.asarray(a, dtype=np.int32))

    qo, sl = host(qo_indptr_host), host(seq_lens_host)
    if qo.shape != (dims.batch + 1,) or sl.shape != (dims.batch,):
        raise ValueError("qo_indptr_host must hold batch + 1 entries and seq_lens_host batch entries")
    lib = load()
    need = ctypes.c_size_t(0)
    args = (qo.ctypes.data, sl.ctypes.data, ctypes.byref(dims), int(bool(causal)), int(num_ctas), int(device))
    st = lib.astr_attn_prefill_plan(*args, None, 0, ctypes.byref(need))
    if st == ASTR_ERR_UNSUPPORTED:
        return None
    _check(st, "astr_attn_prefill_plan", check)
    if st != ASTR_OK:
        return None
    plan = np.zeros(max(int(need.value), 1), np.int32)
    st = lib.astr_attn_prefill_plan(*args, plan.ctypes.data, plan.size, ctypes.byref(need))
    _check(st, "astr_attn_prefill_plan", check)
    return plan if st == ASTR_OK else None


def make_prefill_plan(qo_indptr_host, seq_lens_host, dims: Dims, causal: bool = True, device=None):
    """The plan of ``astr_attn_prefill_plan`` copied to the current CUDA device (an int32 tensor),
    or None when no plan applies; ``attach_prefill_plan`` points a Dims at it."""
    import torch
    dev = torch.cuda.current_device() if device is None else int(device)
    plan = astr_attn_prefill_plan(qo_indptr_host, seq_lens_host, dims, causal=causal, device=dev)
    if plan is None:
        return None
    return torch.from_numpy(plan).to(torch.device("cuda", dev))


def attach_prefill_plan(dims: Dims, plan) -> Dims:
    """Point ``dims`` at a device plan tensor (or detach it with None); returns dims."""
    if plan is None:
        dims.prefill_plan, dims.prefill_plan_words = None, 0
        return dims
    import torch
    if not (isinstance(plan, torch.Tensor) and plan.is_cuda and plan.dtype == torch.int32 and plan.is_contiguous()):
        raise ValueError("a prefill plan is a contiguous int32 CUDA tensor (see make_prefill_plan)")
    dims.prefill_plan, dims.prefill_plan_words = int(plan.data_ptr()), int(plan.numel())
    return dims


def astr_attn_kv_append(k_new, v_new, qo_indptr, req_to_token, seq_lens, k_pool, v_pool, dims: Dims, stream=None,
                        check: bool = True) -> int:
    """Write the new tokens' K/V rows ([total_q, Hkv, d]) into their pool slots in place."""
    st = load().astr_attn_kv_append(_ptr(k_new), _ptr(v_new), _ptr(qo_indptr), _ptr(req_to_token), _ptr(seq_lens),
                                    _ptr(k_pool), _ptr(v_pool), ctypes.byref(dims), _stream(stream))
    return _check(st, "astr_attn_kv_append", check)


def astr_attn_paged_decode_masked(q, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, mask: Mask, o_part, ml_part,
                                  out, dims: Dims, sm_scale: float, stream=None, check: bool = True) -> int:
    """Paged decode with an explicit mask (``make_mask``)."""
    st = load().astr_attn_paged_decode_masked(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(req_to_token),
                                              _ptr(seq_lens), _ptr(kv_indptr),
                                              None if mask is None else ctypes.byref(mask), _ptr(o_part),
                                              _ptr(ml_part), _ptr(out), ctypes.byref(dims), float(sm_scale),
                                              _stream(stream))
    return _check(st, "astr_attn_paged_decode_masked", check)


def astr_attn_prefill_ragged_masked(q, qo_indptr, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, mask: Mask,
                                    out, dims: Dims, sm_scale: float, stream=None, check: bool = True) -> int:
    """Ragged prefill with an explicit mask and/or the causal offset off (``make_mask``)."""
    st = load().astr_attn_prefill_ragged_masked(_ptr(q), _ptr(qo_indptr), _ptr(k_pool), _ptr(v_pool),
                                                _ptr(req_to_token), _ptr(seq_lens), _ptr(kv_indptr),
                                                None if mask is None else ctypes.byref(mask), _ptr(out),
                                                ctypes.byref(dims), float(sm_scale), _stream(stream))
    return _check(st, "astr_attn_prefill_ragged_masked", check)


def astr_attn_decode_contiguous(q, k_cache, v_cache, layout: KvLayout, seq_lens, kv_indptr, o_part, ml_part, out,
                                dims: Dims, sm_scale: float, mask: Optional[Mask] = None, stream=None,
                                check: bool = True) -> int:
    """Split-KV decode over a contiguous K/V cache (``make_kv_layout``); optional explicit mask."""
    st = load().astr_attn_decode_contiguous(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                            None if layout is None else ctypes.byref(layout), _ptr(seq_lens),
                                            _ptr(kv_indptr), None if mask is None else ctypes.byref(mask),
                                            _ptr(o_part), _ptr(ml_part), _ptr(out), ctypes.byref(dims),
                                            float(sm_scale), _stream(stream))
    return _check(st, "astr_attn_decode_contiguous", check)


def astr_attn_prefill_contiguous(q, qo_indptr, k_cache, v_cache, layout: KvLayout, seq_lens, kv_indptr, out,
                                 dims: Dims, sm_scale: float, mask: Optional[Mask] = None, stream=None,
                                 check: bool = True) -> int:
    """Ragged prefill over a contiguous K/V cache; optional mask / causal switch (``make_mask``)."""
    st = load().astr_attn_prefill_contiguous(_ptr(q), _ptr(qo_indptr), _ptr(k_cache), _ptr(v_cache),
                                             None if layout is None else ctypes.byref(layout), _ptr(seq_lens),
                                             _ptr(kv_indptr), None if mask is None else ctypes.byref(mask),
                                             _ptr(out), ctypes.byref(dims), float(sm_scale), _stream(stream))
    return _check(st, "astr_attn_prefill_contiguous", check)


def _ref(x):
    return None if x is None else ctypes.byref(x)


def astr_attn_decode_strided(q, k, v, req_to_token, seq_lens, kv_indptr, o_part, ml_part, out, dims: Dims,
                             sm_scale: float, kv_layout: Optional[KvLayout] = None,
                             qo_layout: Optional[QoLayout] = None, mask: Optional[Mask] = None, stream=None,
                             check: bool = True) -> int:
    """Decode with K/V paged (kv_layout None) or contiguous, query / output by strides (qo_layout;
    None = packed), optional mask."""
    st = load().astr_attn_decode_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(req_to_token), _ref(kv_layout),
                                         _ref(qo_layout), _ptr(seq_lens), _ptr(kv_indptr), _ref(mask), _ptr(o_part),
                                         _ptr(ml_part), _ptr(out), ctypes.byref(dims), float(sm_scale),
                                         _stream(stream))
    return _check(st, "astr_attn_decode_strided", check)


def astr_attn_prefill_strided(q, qo_indptr, k, v, req_to_token, seq_lens, kv_indptr, out, dims: Dims,
                              sm_scale: float, kv_layout: Optional[KvLayout] = None,
                              qo_layout: Optional[QoLayout] = None, mask: Optional[Mask] = None, stream=None,
                              check: bool = True) -> int:
    """Ragged prefill with K/V paged or contiguous, query / output by strides, optional mask."""
    st = load().astr_attn_prefill_strided(_ptr(q), _ptr(qo_indptr), _ptr(k), _ptr(v), _ptr(req_to_token),
                                          _ref(kv_layout), _ref(qo_layout), _ptr(seq_lens), _ptr(kv_indptr),
                                          _ref(mask), _ptr(out), ctypes.byref(dims), float(sm_scale),
                                          _stream(stream))
    return _check(st, "astr_attn_prefill_strided", check)


def alloc_decode_workspace(dims: Dims, device="cuda"):
    """Allocate (once, outside the hot loop) o_part and ml_part for ``dims`` with PyTorch."""
    import torch
    ob, mb = astr_attn_decode_workspace_bytes(dims)
    o_part = torch.empty(ob // 4, dtype=torch.float32, device=device)
    ml_part = torch.empty(mb // 4, dtype=torch.float32, device=device)
    return o_part, ml_part
