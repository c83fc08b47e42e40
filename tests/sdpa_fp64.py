"""Independent fp64 formulation of paged attention through torch's SDPA library routine.

Used only to pin the oracle.  It follows the batched torch-native path described on the
AstrAI commit page "astrai/extension/backend/attention.py @c9ceca1" (batched-SDPA commit):
gather each request's K/V through its req_to_token row into padded [B, max_kv] tensors,
expand KV heads to query heads (consecutive groups, as in the fallback-GQA bullet of page
"astrai/extension @6f67ba8"), build one boolean mask [B, 1, max_q, max_kv] that folds the
per-request causal offset seq_len - q_len and the KV padding, make one SDPA call, and
unpack the valid query rows back to flat qo_indptr order.
"""
import numpy as np
import torch
import torch.nn.functional as F

from workload import bf16_bits_to_fp32


def _f64(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bf16_bits_to_fp32(bits).astype(np.float64))


def sdpa_paged(w, extra_mask=None, causal: bool = True) -> np.ndarray:
    """Returns [rows, Hq, d] float64, rows = B (decode) or total_q (prefill).

    ``extra_mask`` (2-D [B, kv] or 3-D [B, q, kv], nonzero = visible) is AND-ed into the
    boolean mask; ``causal=False`` drops the causal term (the prefill-mask commit of page
    "astrai/extension @6f67ba8": causal and mask coexist, causal may be off).  Rows with no
    visible key come back as NaN from SDPA; callers compare them separately."""
    B, Hq, Hkv, D = w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim
    G = Hq // Hkv
    seq = w.seq_lens.astype(np.int64)
    qlen = w.q_lens.astype(np.int64)
    qo = np.zeros(B + 1, dtype=np.int64)
    qo[1:] = np.cumsum(qlen)
    max_kv = int(seq.max())
    max_q = int(qlen.max())
    k_pool, v_pool, q_all = _f64(w.k_pool), _f64(w.v_pool), _f64(w.q)
    # gather K/V: [B, max_kv] slot ids; padding points at slot 0 and is masked out
    pos = np.arange(max_kv)[None, :]
    kv_valid = pos < seq[:, None]
    slots = np.where(kv_valid, w.req_to_token[:, :max_kv].astype(np.int64), 0)
    slots_t = torch.from_numpy(slots)
    K = k_pool[slots_t]            # [B, max_kv, Hkv, D]
    V = v_pool[slots_t]
    K = K.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)   # [B, Hq, max_kv, D]
    V = V.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    # pad queries: padded rows gather row 0 and are dropped afterwards
    qi = np.arange(max_q)[None, :]
    q_valid = qi < qlen[:, None]
    qrows = np.where(q_valid, qo[:-1, None] + qi, 0)
    Q = q_all[torch.from_numpy(qrows)].permute(0, 2, 1, 3)  # [B, Hq, max_q, D]
    # bottom-right causal: key j visible to local row i iff j <= (seq - qlen) + i, and j < seq
    offset = (seq - qlen)[:, None, None]
    mask = kv_valid[:, None, :] & np.ones((B, max_q, 1), dtype=bool)
    if causal:
        mask = mask & (pos[:, None, :] <= offset + qi[:, :, None])
    if extra_mask is not None:
        em = np.asarray(extra_mask) != 0
        if em.ndim == 2:
            em = em[:, None, :max_kv]
        else:
            em = em[:, :max_q, :max_kv]
            if em.shape[1] < max_q:  # rows past the mask's q extent are padding, dropped below
                em = np.concatenate([em, np.zeros((B, max_q - em.shape[1], max_kv), dtype=bool)], axis=1)
        mask = mask & em
    # fully masked padded rows would give NaN; they are dropped, so let them see key 0
    mask = mask | (~q_valid[:, :, None] & (pos[:, None, :] == 0))
    mask_t = torch.from_numpy(mask)[:, None, :, :]
    O = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask_t, scale=float(w.sm_scale))
    O = O.permute(0, 2, 1, 3)  # [B, max_q, Hq, D]
    return O[torch.from_numpy(q_valid)].numpy()
