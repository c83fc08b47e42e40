"""Seeded synthetic workloads for paged attention (shared by the oracle and the CUDA path).

This module draws inputs only: request lengths, the page_size=1 slot permutation,
and bf16 Q/K/V. It contains none of the attention arithmetic, so the oracle and the
CUDA kernels can both consume its arrays without sharing any method code.

Draw order for a seed (numpy PCG64 via ``default_rng``):
  decode : seq_lens, slot permutation, q, k, v
  prefill: q_lens, prefixes (seq_len = prefix + q_len), slot permutation, q, k, v
Every float is drawn as fp32 N(0,1) and rounded to bf16 with round-to-nearest-even.
Request b's token j lives in slot ``perm[kv_indptr[b] + j]``; table entries past
``seq_len_b`` hold slot 0 and are never read.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "CONFIGS", "config", "make_decode", "make_prefill",
    "fp32_to_bf16_bits", "bf16_bits_to_fp32", "make_from_lengths", "append_rows", "make_mask",
]


def fp32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round-to-nearest-even); returns uint16 bit patterns.

    Inputs are finite normals here, so the NaN case of the rounding rule is not needed;
    NaN inputs are mapped to the canonical quiet NaN to stay safe.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_fp32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Workload:
    """One batch of paged-attention inputs, all host numpy arrays.

    Layouts: q [rows, Hq, d] bf16 bits (rows = B for decode, total_q for prefill);
    k_pool, v_pool [num_slots, Hkv, d] bf16 bits; req_to_token [B, r2t_stride] int32;
    seq_lens [B] int32; kv_indptr [B+1] int32 (exclusive prefix sum of seq_lens);
    qo_indptr [B+1] int32 for prefill (None for decode).
    """
    name: str
    kind: str                 # "decode" | "prefill"
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    sm_scale: float
    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    req_to_token: np.ndarray
    seq_lens: np.ndarray
    kv_indptr: np.ndarray
    qo_indptr: Optional[np.ndarray] = None
    seed: int = 0

    @property
    def num_slots(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def r2t_stride(self) -> int:
        return int(self.req_to_token.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0]) if self.kind == "prefill" else self.batch

    @property
    def q_lens(self) -> np.ndarray:
        if self.qo_indptr is None:
            return np.ones(self.batch, dtype=np.int32)
        return np.diff(self.qo_indptr).astype(np.int32)

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.batch else 0

    def kv_bytes(self) -> int:
        """Bytes of K and V rows that one decode call must read (each attended token, each KV head)."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim * 2 * 2


# The five workloads: (kind, B, Hq, Hkv, d, length ranges, r2t_stride).
CONFIGS = {
    1: dict(name="decode-tiny B=4 Hq8/Hkv2 d64 seq16-128", kind="decode", B=4, Hq=8, Hkv=2, d=64,
            seq=(16, 128), stride=128),
    2: dict(name="decode B=32 Hq32/Hkv8 d128 seq200-2000", kind="decode", B=32, Hq=32, Hkv=8, d=128,
            seq=(200, 2000), stride=2000),
    3: dict(name="decode-long B=8 Hq32/Hkv8 d128 seq16384-32768", kind="decode", B=8, Hq=32, Hkv=8, d=128,
            seq=(16384, 32768), stride=32768),
    4: dict(name="decode-large B=256 Hq32/Hkv8 d128 seq512-4096", kind="decode", B=256, Hq=32, Hkv=8,
            d=128, seq=(512, 4096), stride=4096),
    5: dict(name="prefill-ragged 16 req q1-512 prefix0-2048 Hq32/Hkv8 d128", kind="prefill", B=16, Hq=32,
            Hkv=8, d=128, qlen=(1, 512), prefix=(0, 2048), stride=2560),
}


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return fp32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def make_from_lengths(rng: np.random.Generator, *, kind: str, name: str, seq_lens, q_lens, Hq: int, Hkv: int,
                      d: int, stride: Optional[int] = None, sm_scale: Optional[float] = None,
                      extra_slots: int = 0, seed: int = 0) -> Workload:
    """Build a workload from given lengths: draws the slot permutation, then q, k, v.

    ``extra_slots`` appends pool rows that no request references (used by poison tests).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    B = int(seq_lens.shape[0])
    kv_indptr = np.zeros(B + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum(seq_lens)
    T = int(kv_indptr[-1])
    if stride is None:
        stride = max(1, int(seq_lens.max()) if B else 1)
    perm = rng.permutation(T).astype(np.int64)
    r2t = np.zeros((B, stride), dtype=np.int32)
    for b in range(B):
        n = int(seq_lens[b])
        r2t[b, :n] = perm[kv_indptr[b]:kv_indptr[b] + n]
    if kind == "decode":
        qo_indptr = None
        q = _normal_bf16(rng, (B, Hq, d))
    else:
        q_lens = np.asarray(q_lens, dtype=np.int64)
        qo_indptr = np.zeros(B + 1, dtype=np.int64)
        qo_indptr[1:] = np.cumsum(q_lens)
        q = _normal_bf16(rng, (int(qo_indptr[-1]), Hq, d))
        qo_indptr = qo_indptr.astype(np.int32)
    num_slots = T + extra_slots
    k_pool = _normal_bf16(rng, (num_slots, Hkv, d))
    v_pool = _normal_bf16(rng, (num_slots, Hkv, d))
    return Workload(name=name, kind=kind, batch=B, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                    sm_scale=float(sm_scale if sm_scale is not None else 1.0 / math.sqrt(d)),
                    q=q, k_pool=k_pool, v_pool=v_pool, req_to_token=r2t,
                    seq_lens=seq_lens.astype(np.int32), kv_indptr=kv_indptr.astype(np.int32),
                    qo_indptr=qo_indptr, seed=seed)


def make_decode(B: int, Hq: int, Hkv: int, d: int, seq: tuple, seed: int, stride: Optional[int] = None,
                name: str = "decode", extra_slots: int = 0) -> Workload:
    rng = np.random.default_rng(seed)
    seq_lens = rng.integers(seq[0], seq[1] + 1, size=B)
    return make_from_lengths(rng, kind="decode", name=name, seq_lens=seq_lens, q_lens=None, Hq=Hq, Hkv=Hkv, d=d,
                             stride=stride if stride is not None else seq[1], extra_slots=extra_slots, seed=seed)


def make_prefill(B: int, Hq: int, Hkv: int, d: int, qlen: tuple, prefix: tuple, seed: int,
                 stride: Optional[int] = None, name: str = "prefill", extra_slots: int = 0) -> Workload:
    rng = np.random.default_rng(seed)
    q_lens = rng.integers(qlen[0], qlen[1] + 1, size=B)
    prefixes = rng.integers(prefix[0], prefix[1] + 1, size=B)
    seq_lens = prefixes + q_lens
    return make_from_lengths(rng, kind="prefill", name=name, seq_lens=seq_lens, q_lens=q_lens, Hq=Hq, Hkv=Hkv,
                             d=d, stride=stride if stride is not None else qlen[1] + prefix[1],
                             extra_slots=extra_slots, seed=seed)


def append_rows(w: Workload, seed: int):
    """New K/V rows for the KV-append step over workload ``w``: (qo_indptr, k_new, v_new).

    A prefill workload appends its q_len_b new tokens per request (its own qo_indptr); a
    decode workload appends one token per request that has at least one key (the current
    token, the last key of the request).  k_new and v_new are [total_new, Hkv, d] bf16 bits,
    drawn K then V from ``default_rng(seed)`` as fp32 N(0,1) rounded to bf16.
    """
    rng = np.random.default_rng(seed)
    if w.qo_indptr is not None:
        qo = np.asarray(w.qo_indptr, dtype=np.int32)
    else:
        qo = np.zeros(w.batch + 1, dtype=np.int32)
        qo[1:] = np.cumsum(np.minimum(w.seq_lens, 1))
    n = int(qo[-1])
    k_new = _normal_bf16(rng, (n, w.num_kv_heads, w.head_dim))
    v_new = _normal_bf16(rng, (n, w.num_kv_heads, w.head_dim))
    return qo, k_new, v_new


def make_mask(w: Workload, dims: int, seed: int, keep: float = 0.75) -> np.ndarray:
    """An explicit attention mask for workload ``w``: uint8 (1 = visible, 0 = masked), each
    byte 1 with probability ``keep`` (``default_rng(seed)``, one uniform per byte).

    dims = 2: [B, kv_pitch]; dims = 3: [B, q_pitch, kv_pitch] with q_pitch = max_q_len (1 for
    decode).  kv_pitch = max_seq_len rounded up to 16 bytes; bytes past a request's keys or
    rows are drawn too and are never read.
    """
    rng = np.random.default_rng(seed)
    kv_pitch = max(16, -(-w.max_seq_len // 16) * 16)
    shape = (w.batch, kv_pitch) if dims == 2 else (w.batch, max(1, w.max_q_len), kv_pitch)
    return (rng.random(shape) < keep).astype(np.uint8)


def config(idx: int, seed: Optional[int] = None) -> Workload:
    """Workload ``idx`` (1..5) with seed 20260 + idx unless overridden."""
    c = CONFIGS[idx]
    s = 20260 + idx if seed is None else seed
    if c["kind"] == "decode":
        return make_decode(c["B"], c["Hq"], c["Hkv"], c["d"], c["seq"], s, stride=c["stride"], name=c["name"])
    return make_prefill(c["B"], c["Hq"], c["Hkv"], c["d"], c["qlen"], c["prefix"], s, stride=c["stride"],
                        name=c["name"])
