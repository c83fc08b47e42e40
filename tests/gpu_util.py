"""Helpers for the GPU parity tests: upload a workload, call the C ABI, read results back."""
import numpy as np

import prefill_attention_gb300 as pa
import split_schedule
from split_schedule import SLOT_KEYS  # noqa: F401

TOL = 1e-2  # max abs error of bf16 outputs against the fp64 oracle


def _torch():
    import torch
    return torch


def bf16_dev(a, device="cuda"):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def i32_dev(a, device="cuda"):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def to_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def upload(w, device="cuda"):
    d = dict(q=bf16_dev(w.q, device), k=bf16_dev(w.k_pool, device), v=bf16_dev(w.v_pool, device),
             r2t=i32_dev(w.req_to_token, device), seq=i32_dev(w.seq_lens, device), kvi=i32_dev(w.kv_indptr, device))
    if w.qo_indptr is not None:
        d["qo"] = i32_dev(w.qo_indptr, device)
    return d


def decode_dims(w, max_splits=32, num_splits=0):
    return pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride,
                        w.max_seq_len, max_splits=max_splits, num_splits=num_splits)


def prefill_dims(w):
    return pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride,
                        w.max_seq_len, total_q=w.total_q, max_q_len=w.max_q_len)


def decode_chunk_slots(w, n_chunks, max_splits):
    """Chunk length in 32-key slots of the decode split schedule, as documented for
    astr_attn_paged_decode."""
    return split_schedule.chunk_slots(w.seq_lens, w.max_seq_len, n_chunks, max_splits)


def run_decode(w, t=None, max_splits=32, num_splits=0, stream=None, return_parts=False):
    torch = _torch()
    t = t or upload(w)
    dims = decode_dims(w, max_splits, num_splits)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.empty_like(t["q"])
    pa.astr_attn_paged_decode(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, out, dims,
                              w.sm_scale, stream=stream)
    torch.cuda.synchronize()
    if return_parts:
        n_chunks = pa.astr_attn_decode_num_splits(dims, torch.cuda.current_device())
        B, Hq, D = w.batch, w.num_qo_heads, w.head_dim
        o = o_part.view(B, Hq, max_splits, D).cpu().numpy().astype(np.float64)
        ml = ml_part.view(B, Hq, max_splits, 2).cpu().numpy().astype(np.float64)
        return out, o, ml, n_chunks
    return out


def run_prefill(w, t=None, stream=None):
    torch = _torch()
    t = t or upload(w)
    dims = prefill_dims(w)
    out = torch.empty_like(t["q"])
    pa.astr_attn_prefill_ragged(t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], out, dims,
                                w.sm_scale, stream=stream)
    torch.cuda.synchronize()
    return out
