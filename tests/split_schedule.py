"""The decode split schedule documented for astr_attn_paged_decode, as key ranges.

Test helper (CPU only, no GPU or library import).  The schedule is how the library chooses
its split boundaries; it is not part of what attention computes, so it lives here rather
than in the oracle.  The oracle only supplies the partial of one split over an explicit key
range (``oracle.partial_ranges``); this module turns the documented schedule into those
ranges:

  * request b's keys are cut into slots of W keys from its first key (the last possibly
    short); the batch's slots lie end to end in request order, request b starting at slot
    SP_b = sum over b' < b of ceil(seq_len_b' / W);
  * the slot sequence is cut into chunks of C slots, C = max(ceil(S / n_chunks), F) with
    F = max(1, ceil(ceil(max_seq_len / W) / (max_splits - 1))) (C = S for max_splits = 1);
  * the piece of request b in chunk c is partial slot c - SP_b // C of (b, h).
"""
import numpy as np

import oracle

SLOT_KEYS = 32  # W: keys per slot of the library's schedule


def _slots(n, W):
    return -(-int(n) // W) if int(n) > 0 else 0


def chunk_slots(seq_lens, max_seq_len, n_chunks, max_splits, W=SLOT_KEYS):
    """Chunk length C in slots for ``n_chunks`` chunks per KV head and a partial capacity of
    ``max_splits`` slots per (request, head)."""
    total = sum(_slots(n, W) for n in seq_lens)
    if max_splits <= 1:
        return max(total, 1)
    c = -(-total // n_chunks)
    floor = max(1, -(-(-(-int(max_seq_len) // W)) // (max_splits - 1)))
    return max(c, floor)


def pieces(seq_lens, C, W=SLOT_KEYS):
    """The (request b, partial slot s, first key lo, end key hi) of every request piece, by
    overlapping each request's slot interval with the chunk grid."""
    out, sp = [], 0
    for b, n in enumerate(seq_lens):
        n = max(int(n), 0)
        ns = _slots(n, W)
        c = sp // C
        while ns > 0 and c * C < sp + ns:
            g0, g1 = max(c * C, sp), min((c + 1) * C, sp + ns)
            out.append((b, c - sp // C, (g0 - sp) * W, min((g1 - sp) * W, n)))
            c += 1
        sp += ns
    return out


def split_counts(seq_lens, C, W=SLOT_KEYS):
    """Number of chunks that overlap each request (the partial slots it uses)."""
    ns = np.zeros(len(seq_lens), dtype=np.int32)
    for b, s, _, _ in pieces(seq_lens, C, W):
        ns[b] = max(ns[b], s + 1)
    return ns


def chunk_partials(w, C, pitch, W=SLOT_KEYS, lib=None):
    """Oracle partials laid out as the library's split step writes them: (o [B,Hq,pitch,d],
    ml [B,Hq,pitch,2], nsplit [B]); slots no piece maps to hold NaN."""
    B, Hq, D = w.batch, w.num_qo_heads, w.head_dim
    ps = pieces(w.seq_lens, C, W)
    items = np.array([(b, h, lo, hi) for (b, s, lo, hi) in ps for h in range(Hq)], dtype=np.int64).reshape(-1, 4)
    o = np.full((B, Hq, pitch, D), np.nan)
    ml = np.full((B, Hq, pitch, 2), np.nan)
    if len(items):
        po, pml = oracle.partial_ranges(w, items, lib=lib)
        k = 0
        for (b, s, _, _) in ps:
            for h in range(Hq):
                if s < pitch:
                    o[b, h, s], ml[b, h, s] = po[k], pml[k]
                k += 1
    return o, ml, split_counts(w.seq_lens, C, W)
