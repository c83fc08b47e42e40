"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Each ``pin_*`` takes a loaded oracle library (the real one, or a planted mutant in the
mutation tests) and raises AssertionError when the oracle disagrees with:
  * torch's fp64 SDPA library routine on the padded/masked formulation (special case
    reducing to a library routine),
  * closed forms (q = 0 gives the mean of the visible V rows; one key gives that V row;
    constant V gives the constant; hand-worked examples in tests/golden),
  * invariances (slot permutation, key shift, per-request markers),
  * the split-KV identity (partials + log-sum-exp combine equals unsplit softmax),
  * the KV-append step: attention over the pool after the append equals SDPA over each
    request's cached keys followed by its new rows, laid out contiguously,
  * explicit masks: SDPA with the mask AND-ed in (causal on or off), rows with no visible key
    exactly zero (empty-sum reading); an all-ones mask, a 3-D causal pattern with causal off,
    a 2-D mask repeated over rows and a decode mask turned into a shorter slot table all
    reproduce the corresponding unmasked or 2-D results bit for bit.
"""
import dataclasses
import json
import math
import os

import numpy as np

import oracle
import workload
from workload import bf16_bits_to_fp32, fp32_to_bf16_bits, make_from_lengths

import split_schedule
from sdpa_fp64 import sdpa_paged

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")


def _small_decode(seed=7, B=3, Hq=8, Hkv=2, d=16, lo=1, hi=40):
    rng = np.random.default_rng(seed)
    seq = rng.integers(lo, hi + 1, size=B)
    return make_from_lengths(rng, kind="decode", name="small", seq_lens=seq, q_lens=None, Hq=Hq, Hkv=Hkv, d=d)


def _small_prefill(seed=11, B=4, Hq=8, Hkv=2, d=16, qmax=9, pmax=12):
    rng = np.random.default_rng(seed)
    ql = rng.integers(1, qmax + 1, size=B)
    pre = rng.integers(0, pmax + 1, size=B)
    return make_from_lengths(rng, kind="prefill", name="small", seq_lens=pre + ql, q_lens=ql, Hq=Hq, Hkv=Hkv,
                             d=d)


def _set_rows(pool_bits, slots, kvh, values_f32):
    pool_bits[slots, kvh, :] = fp32_to_bf16_bits(values_f32)


# ------------------------------------------------------------------ library routine


def pin_sdpa_decode(lib, w=None, tol=1e-12):
    w = w or workload.config(1)
    ref = sdpa_paged(w)
    got = oracle.decode(w, lib=lib)
    err = np.abs(got - ref).max()
    assert err <= tol, f"decode vs fp64 SDPA: max abs err {err}"


def pin_sdpa_prefill(lib, w=None, tol=1e-12):
    w = w or workload.make_prefill(16, 32, 8, 128, (1, 64), (0, 256), seed=20265, name="prefill-small")
    ref = sdpa_paged(w)
    got = oracle.prefill(w, lib=lib)
    err = np.abs(got - ref).max()
    assert err <= tol, f"prefill vs fp64 SDPA: max abs err {err}"


def pin_prefix0_is_textbook_causal(lib):
    """With no cached prefix, bottom-right and top-left causal coincide: SDPA is_causal=True."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(3)
    ql = np.array([5, 1, 9])
    w = make_from_lengths(rng, kind="prefill", name="p0", seq_lens=ql, q_lens=ql, Hq=4, Hkv=2, d=8)
    got = oracle.prefill(w, lib=lib)
    q = bf16_bits_to_fp32(w.q).astype(np.float64)
    k = bf16_bits_to_fp32(w.k_pool).astype(np.float64)
    v = bf16_bits_to_fp32(w.v_pool).astype(np.float64)
    for b in range(w.batch):
        rows = slice(int(w.qo_indptr[b]), int(w.qo_indptr[b + 1]))
        slots = w.req_to_token[b, :ql[b]]
        Q = torch.from_numpy(q[rows]).permute(1, 0, 2)                       # [Hq, L, d]
        K = torch.from_numpy(k[slots]).permute(1, 0, 2).repeat_interleave(2, 0)
        V = torch.from_numpy(v[slots]).permute(1, 0, 2).repeat_interleave(2, 0)
        ref = F.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=w.sm_scale).permute(1, 0, 2)
        err = np.abs(got[rows] - ref.numpy()).max()
        assert err <= 1e-12, f"prefix-0 prefill vs is_causal SDPA (request {b}): {err}"


# ------------------------------------------------------------------ closed forms


def pin_golden(lib):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    env = {"e": math.e, "exp": math.exp, "sinh": math.sinh, "cosh": math.cosh, "__builtins__": {}}
    for c in cases:
        d = c["head_dim"]
        exp_vals = [eval(s, env) for s in c["expected_formula"]]  # noqa: S307 (fixed fixture)
        assert np.allclose(exp_vals, c["expected"], rtol=0, atol=1e-15), f"fixture formula mismatch: {c['name']}"
        kp = fp32_to_bf16_bits(np.array(c["k_pool"], np.float32).reshape(-1, 1, d))
        vp = fp32_to_bf16_bits(np.array(c["v_pool"], np.float32).reshape(-1, 1, d))
        assert np.array_equal(bf16_bits_to_fp32(kp).ravel(), np.array(c["k_pool"], np.float32).ravel())
        r2t = np.array([c["req_to_token"]], np.int32)
        seq = np.array([c["seq_len"]], np.int32)
        if c.get("prefill"):
            ql = c["q_len"]
            q = fp32_to_bf16_bits(np.array(c["q"], np.float32).reshape(ql, 1, d))
            w = workload.Workload(name=c["name"], kind="prefill", batch=1, num_qo_heads=1, num_kv_heads=1,
                                  head_dim=d, sm_scale=c["sm_scale"], q=q, k_pool=kp, v_pool=vp,
                                  req_to_token=r2t, seq_lens=seq, kv_indptr=np.array([0, seq[0]], np.int32),
                                  qo_indptr=np.array([0, ql], np.int32))
            got = oracle.prefill(w, lib=lib)[:, 0, 0]
        else:
            q = fp32_to_bf16_bits(np.array(c["q"], np.float32).reshape(1, 1, d))
            w = workload.Workload(name=c["name"], kind="decode", batch=1, num_qo_heads=1, num_kv_heads=1,
                                  head_dim=d, sm_scale=c["sm_scale"], q=q, k_pool=kp, v_pool=vp,
                                  req_to_token=r2t, seq_lens=seq, kv_indptr=np.array([0, seq[0]], np.int32))
            got = oracle.decode(w, lib=lib)[0, 0]
        err = np.abs(got - np.array(c["expected"])).max()
        assert err <= 1e-14, f"golden '{c['name']}': got {got}, expected {c['expected']}"


def pin_q_zero_is_mean_of_visible_v(lib):
    """q = 0 makes all logits equal, so the output is the plain mean of the visible V rows."""
    for w in (_small_decode(seed=21), _small_prefill(seed=22)):
        w.q[:] = 0
        v = bf16_bits_to_fp32(w.v_pool).astype(np.float64)
        G = w.num_qo_heads // w.num_kv_heads
        if w.kind == "decode":
            got = oracle.decode(w, lib=lib)
            for b in range(w.batch):
                sl = w.req_to_token[b, :w.seq_lens[b]]
                for h in range(w.num_qo_heads):
                    ref = v[sl, h // G].mean(axis=0)
                    assert np.abs(got[b, h] - ref).max() <= 1e-13, f"q=0 decode b={b} h={h}"
        else:
            got = oracle.prefill(w, lib=lib)
            for b in range(w.batch):
                c = int(w.seq_lens[b]) - int(w.q_lens[b])
                for i in range(int(w.q_lens[b])):
                    sl = w.req_to_token[b, :c + i + 1]
                    for h in range(w.num_qo_heads):
                        ref = v[sl, h // G].mean(axis=0)
                        r = int(w.qo_indptr[b]) + i
                        assert np.abs(got[r, h] - ref).max() <= 1e-13, f"q=0 prefill b={b} i={i} h={h}"


def pin_single_key_returns_v(lib):
    rng = np.random.default_rng(5)
    w = make_from_lengths(rng, kind="decode", name="one", seq_lens=[1, 1, 1], q_lens=None, Hq=8, Hkv=4, d=32)
    got = oracle.decode(w, lib=lib)
    v = bf16_bits_to_fp32(w.v_pool).astype(np.float64)
    for b in range(3):
        for h in range(8):
            assert np.array_equal(got[b, h], v[w.req_to_token[b, 0], h // 2]), f"seq_len=1 b={b} h={h}"


def pin_per_request_marker(lib):
    """Every V row of request b set to b+1 (all heads): each output row of request b equals b+1.

    Catches any mixing of requests (wrong req_to_token row, qo_indptr or seq_len routing).
    """
    for w in (_small_decode(seed=31, B=5), _small_prefill(seed=32, B=5)):
        for b in range(w.batch):
            sl = w.req_to_token[b, :w.seq_lens[b]]
            w.v_pool[sl] = fp32_to_bf16_bits(np.full((len(sl), w.num_kv_heads, w.head_dim), b + 1, np.float32))
        got = oracle.decode(w, lib=lib) if w.kind == "decode" else oracle.prefill(w, lib=lib)
        if w.kind == "decode":
            ref = np.broadcast_to((np.arange(w.batch) + 1.0)[:, None, None], got.shape)
        else:
            owner = np.repeat(np.arange(w.batch), w.q_lens)
            ref = np.broadcast_to((owner + 1.0)[:, None, None], got.shape)
        assert np.abs(got - ref).max() <= 1e-13, "per-request marker mismatch"


def pin_dominant_key(lib):
    """One key aligned with q and scaled far above the rest takes (numerically) all the weight."""
    rng = np.random.default_rng(9)
    w = make_from_lengths(rng, kind="decode", name="dom", seq_lens=[12], q_lens=None, Hq=1, Hkv=1, d=8,
                          sm_scale=1.0)
    w.q[0, 0] = fp32_to_bf16_bits(np.array([1, 0, 0, 0, 0, 0, 0, 0], np.float32))
    kf = bf16_bits_to_fp32(w.k_pool).copy()
    kf[:, 0, 0] = np.clip(kf[:, 0, 0], -2, 2)
    j = 7
    kf[w.req_to_token[0, j], 0, 0] = 64.0
    w.k_pool[:] = fp32_to_bf16_bits(kf)
    got = oracle.decode(w, lib=lib)[0, 0]
    ref = bf16_bits_to_fp32(w.v_pool[w.req_to_token[0, j], 0]).astype(np.float64)
    assert np.abs(got - ref).max() <= 1e-15, "dominant key"


# ------------------------------------------------------------------ invariances


def pin_slot_permutation(lib):
    """Paged == contiguous: the same logical K/V behind a different slot table gives the same bits."""
    w = _small_decode(seed=41, B=4)
    out1 = oracle.decode(w, lib=lib)
    T = w.num_slots
    rng = np.random.default_rng(42)
    perm = rng.permutation(T)          # new slot of old slot s is perm[s]
    k2 = np.empty_like(w.k_pool); v2 = np.empty_like(w.v_pool)
    k2[perm] = w.k_pool; v2[perm] = w.v_pool
    r2t2 = w.req_to_token.copy()
    for b in range(w.batch):
        n = w.seq_lens[b]
        r2t2[b, :n] = perm[w.req_to_token[b, :n]]
    w.k_pool, w.v_pool, w.req_to_token = k2, v2, r2t2
    out2 = oracle.decode(w, lib=lib)
    assert np.array_equal(out1, out2), "slot permutation changed the output"


def pin_key_shift(lib):
    """Adding one vector u to every key shifts all logits of a row equally: output unchanged."""
    rng = np.random.default_rng(51)
    w = make_from_lengths(rng, kind="decode", name="shift", seq_lens=[17, 5], q_lens=None, Hq=4, Hkv=2, d=8,
                          sm_scale=0.25)
    # small integers keep K + u exact in bf16
    kq = rng.integers(-4, 5, size=w.k_pool.shape).astype(np.float32)
    w.k_pool[:] = fp32_to_bf16_bits(kq)
    w.q[:] = fp32_to_bf16_bits(rng.integers(-3, 4, size=w.q.shape).astype(np.float32))
    out1 = oracle.decode(w, lib=lib)
    u = rng.integers(-8, 9, size=(1, w.num_kv_heads, w.head_dim)).astype(np.float32)
    w.k_pool[:] = fp32_to_bf16_bits(kq + u)
    out2 = oracle.decode(w, lib=lib)
    assert np.abs(out1 - out2).max() <= 1e-12, "key shift changed the output"


def pin_unreferenced_slots_unread(lib):
    """Masked/padded lanes contribute exactly zero: NaN in every slot the visible keys do not name,
    and table entries past seq_len pointing at those NaN slots, leave the output unchanged."""
    for kind in ("decode", "prefill"):
        rng = np.random.default_rng(61)
        ql = np.array([3, 1, 6, 2]) if kind == "prefill" else None
        seq = np.array([9, 4, 13, 2])
        w = make_from_lengths(rng, kind=kind, name="poison", seq_lens=seq, q_lens=ql, Hq=4, Hkv=2, d=8,
                              extra_slots=7, stride=20)
        T = int(seq.sum())
        base = oracle.decode(w, lib=lib) if kind == "decode" else oracle.prefill(w, lib=lib)
        w.k_pool[T:] = 0x7FC0
        w.v_pool[T:] = 0x7FC0
        for b in range(w.batch):
            w.req_to_token[b, seq[b]:] = T + (b % 7)
        got = oracle.decode(w, lib=lib) if kind == "decode" else oracle.prefill(w, lib=lib)
        assert np.isfinite(got).all() and np.array_equal(base, got), f"{kind}: poisoned slots leaked"


# ------------------------------------------------------------------ split-KV


def pin_split_combine(lib):
    """Even S-way partials + log-sum-exp combine == unsplit attention, for S up to past seq_len
    (so empty splits occur and must be neutral: m = -inf, l = 0, o = 0)."""
    w = _small_decode(seed=71, B=4, lo=1, hi=30)
    ref = oracle.decode(w, lib=lib)
    for S in (1, 2, 3, 7, 40):
        o, ml = oracle.decode_split_partials(w, S, lib=lib)
        got = oracle.combine(o, ml, lib=lib)
        err = np.abs(got - ref).max()
        assert err <= 1e-12, f"split combine S={S}: {err}"
        for b in range(w.batch):
            chunk = -(-int(w.seq_lens[b]) // S)
            for s in range(S):
                if s * chunk >= w.seq_lens[b]:
                    assert np.all(np.isneginf(ml[b, :, s, 0])) and np.all(ml[b, :, s, 1] == 0)
                    assert np.all(o[b, :, s] == 0)
                else:
                    assert np.all(np.isfinite(ml[b, :, s]))


def pin_chunk_partials_combine(lib):
    """Partials over key ranges that straddle the batch's request boundaries anywhere (the
    library's slot/chunk schedule, with several chunk lengths and slot widths; W = 1: chunks
    of the flat key space) + combine == unsplit attention."""
    w = _small_decode(seed=73, B=6, lo=0, hi=45)
    w.seq_lens[2] = 0   # an empty request owns no chunk
    w.kv_indptr[1:] = np.cumsum(w.seq_lens)
    ref = oracle.decode(w, lib=lib)
    T = int(w.kv_indptr[-1])
    for W in (1, 5, 32):
        n_slots = int(sum(-(-int(n) // W) for n in w.seq_lens))
        for C in (1, 2, 7, 16, 33, n_slots, n_slots + 5, T):
            ns = split_schedule.split_counts(w.seq_lens, C, W)
            pitch = max(1, int(ns.max()))
            o, ml, _ = split_schedule.chunk_partials(w, C, pitch, W, lib=lib)
            got = oracle.combine(np.nan_to_num(o), np.where(np.isnan(ml), -np.inf, ml), nsplit=ns, lib=lib)
            err = np.abs(got - ref).max()
            assert err <= 1e-12, f"chunk combine W={W} C={C}: {err}"
            # every written slot is a proper partial: finite m, positive l
            for b in range(w.batch):
                assert np.all(np.isfinite(ml[b, :, :ns[b], 0])) and np.all(ml[b, :, :ns[b], 1] > 0)


def pin_partial_ranges_match_even_split(lib):
    """A partial over an explicit key range equals the even-split partial over the same keys
    (two entry points of the oracle, the same definition)."""
    w = _small_decode(seed=75, B=3, lo=5, hi=30)
    S = 3
    o, ml = oracle.decode_split_partials(w, S, lib=lib)
    items = []
    for b in range(w.batch):
        n = int(w.seq_lens[b]); c = -(-n // S)
        for s in range(S):
            for h in range(w.num_qo_heads):
                items.append((b, h, min(s * c, n), min((s + 1) * c, n)))
    po, pml = oracle.partial_ranges(w, np.array(items), lib=lib)
    k = 0
    for b in range(w.batch):
        for s in range(S):
            for h in range(w.num_qo_heads):
                assert np.array_equal(po[k], o[b, h, s]) and np.array_equal(pml[k], ml[b, h, s])
                k += 1


def pin_partial_is_softmax_piece(lib):
    """One split's (m, l, o): m is the max logit, l*exp(m) the sum of exp(logit), o/l the
    softmax attention over that split's keys alone (checked against fp64 SDPA of that piece)."""
    import torch
    import torch.nn.functional as F
    w = _small_decode(seed=81, B=2, Hq=2, Hkv=1, d=8, lo=10, hi=12)
    S = 3
    o, ml = oracle.decode_split_partials(w, S, lib=lib)
    q = bf16_bits_to_fp32(w.q).astype(np.float64)
    k = bf16_bits_to_fp32(w.k_pool).astype(np.float64)
    v = bf16_bits_to_fp32(w.v_pool).astype(np.float64)
    for b in range(w.batch):
        n = int(w.seq_lens[b]); c = -(-n // S)
        for s in range(S):
            sl = w.req_to_token[b, s * c:min(n, (s + 1) * c)]
            for h in range(2):
                logits = (k[sl, 0] @ q[b, h]) * w.sm_scale
                assert abs(ml[b, h, s, 0] - logits.max()) <= 1e-13
                assert abs(ml[b, h, s, 1] - np.exp(logits - logits.max()).sum()) <= 1e-12
                ref = F.scaled_dot_product_attention(torch.from_numpy(q[b, h][None, None]),
                                                     torch.from_numpy(k[sl, 0][None]),
                                                     torch.from_numpy(v[sl, 0][None]),
                                                     scale=w.sm_scale).numpy()[0, 0]
                assert np.abs(o[b, h, s] / ml[b, h, s, 1] - ref).max() <= 1e-12


def pin_prefill_row_is_decode(lib):
    """Prefill row i of request b equals a decode over the first c_b + i + 1 keys."""
    w = _small_prefill(seed=91)
    got = oracle.prefill(w, lib=lib)
    for b in range(w.batch):
        c = int(w.seq_lens[b]) - int(w.q_lens[b])
        for i in range(int(w.q_lens[b])):
            r = int(w.qo_indptr[b]) + i
            wd = workload.Workload(name="d", kind="decode", batch=1, num_qo_heads=w.num_qo_heads,
                                   num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, sm_scale=w.sm_scale,
                                   q=w.q[r:r + 1].copy(), k_pool=w.k_pool, v_pool=w.v_pool,
                                   req_to_token=w.req_to_token[b:b + 1].copy(),
                                   seq_lens=np.array([c + i + 1], np.int32),
                                   kv_indptr=np.array([0, c + i + 1], np.int32))
            dec = oracle.decode(wd, lib=lib)[0]
            assert np.array_equal(dec, got[r]), f"prefill row b={b} i={i} != decode"


def _contiguous_after_append(w, qo, k_new, v_new):
    """The workload whose request b holds keys (its first c_b cached keys, then its new rows)
    in consecutive slots -- built by hand, without the append step."""
    seq = w.seq_lens.astype(np.int64)
    q_len = np.diff(qo.astype(np.int64))
    base = np.concatenate([[0], np.cumsum(seq)])
    T = int(base[-1])
    kp = np.zeros((max(T, 1), w.num_kv_heads, w.head_dim), np.uint16)
    vp = np.zeros_like(kp)
    r2t = np.zeros((w.batch, max(int(seq.max()), 1)), np.int32)
    for b in range(w.batch):
        c = int(seq[b] - q_len[b])
        cached = w.req_to_token[b, :c].astype(np.int64)
        kp[base[b]:base[b] + c] = w.k_pool[cached]
        vp[base[b]:base[b] + c] = w.v_pool[cached]
        kp[base[b] + c:base[b + 1]] = k_new[qo[b]:qo[b + 1]]
        vp[base[b] + c:base[b + 1]] = v_new[qo[b]:qo[b + 1]]
        r2t[b, :seq[b]] = np.arange(base[b], base[b + 1], dtype=np.int32)
    return dataclasses.replace(w, k_pool=kp, v_pool=vp, req_to_token=r2t)


def pin_append_then_attend_is_sdpa_over_concatenation(lib):
    """After the append, attention over the pool sees each request's cached keys followed by
    its new rows (prefill: q_len_b new tokens at the causal offset; decode: the current token
    as the last key), checked against fp64 SDPA on a hand-built contiguous layout."""
    for w in (_small_prefill(seed=101, pmax=6), _small_decode(seed=103)):
        w = dataclasses.replace(w, req_to_token=np.pad(w.req_to_token, ((0, 0), (0, 3))))
        qo, kn, vn = workload.append_rows(w, seed=105)
        kp, vp = oracle.kv_append(w, qo, kn, vn, lib=lib)
        after = dataclasses.replace(w, k_pool=kp, v_pool=vp)
        got = oracle.prefill(after, lib=lib) if w.kind == "prefill" else oracle.decode(after, lib=lib)
        ref = sdpa_paged(_contiguous_after_append(w, qo, kn, vn))
        err = np.abs(got - ref).max()
        assert err <= 1e-12, f"{w.kind}: attention after append vs SDPA over concatenation: {err}"


def pin_append_touches_only_new_slots(lib):
    """Slots that hold no new token keep their bytes; each new token's slot holds exactly its
    K and V rows (checked through the inverse of the slot table)."""
    w = _small_prefill(seed=107, pmax=6)
    w = dataclasses.replace(w, req_to_token=np.pad(w.req_to_token, ((0, 0), (0, 3))))
    qo, kn, vn = workload.append_rows(w, seed=109)
    kp, vp = oracle.kv_append(w, qo, kn, vn, lib=lib)
    owner = {}  # slot -> flat new row
    for b in range(w.batch):
        for i in range(int(qo[b + 1] - qo[b])):
            pos = int(w.seq_lens[b]) - int(qo[b + 1] - qo[b]) + i
            owner[int(w.req_to_token[b, pos])] = int(qo[b]) + i
    for slot in range(w.num_slots):
        if slot in owner:
            r = owner[slot]
            assert np.array_equal(kp[slot], kn[r]) and np.array_equal(vp[slot], vn[r]), f"slot {slot}"
        else:
            assert np.array_equal(kp[slot], w.k_pool[slot]) and np.array_equal(vp[slot], w.v_pool[slot]), \
                f"slot {slot} changed"


def _masked_cases():
    wp = _small_prefill(seed=121, qmax=9, pmax=12)
    wd = _small_decode(seed=123)
    out = []
    for w in (wp, wd):
        for dims in (2, 3):
            m = workload.make_mask(w, dims, seed=125 + dims, keep=0.6)
            if dims == 3:
                m[0, 0, :] = 0  # a row with no visible key
            else:
                m[-1, :] = 0    # a request with no visible key
            out.append((w, m))
    return out


def pin_masked_matches_sdpa(lib):
    """Masked attention (2-D and 3-D, causal on and off) against fp64 SDPA with the mask
    AND-ed into its boolean mask; rows that see no key are zero."""
    for w, m in _masked_cases():
        # the rows _masked_cases planted with no visible key (first row of request 0 for 3-D
        # masks, every row of the last request for 2-D masks)
        if w.kind == "decode":
            planted = [0] if m.ndim == 3 else [w.batch - 1]
        else:
            b = 0 if m.ndim == 3 else w.batch - 1
            planted = [0] if m.ndim == 3 else list(range(int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])))
        for causal in ((True, False) if w.kind == "prefill" else (True,)):
            got = oracle.masked(w, m, causal=causal, lib=lib)
            assert not got[planted].any(), "a row with no visible key is not zero"
            with np.errstate(invalid="ignore"):
                ref = sdpa_paged(w, extra_mask=m, causal=causal)
            empty = np.isnan(ref).all(axis=(1, 2))  # SDPA gives NaN or 0 there, by version
            ref[empty] = 0.0
            err = np.abs(got - ref).max()
            assert err <= 1e-12, f"{w.kind} dims={m.ndim} causal={causal}: masked vs SDPA {err}"


def pin_mask_identities(lib):
    """All-ones mask = no mask; 3-D lower-triangular causal pattern with causal off = causal;
    2-D mask = the same mask repeated over every row as 3-D (all bit-exact)."""
    wp = _small_prefill(seed=131)
    kv = -(-wp.max_seq_len // 16) * 16
    ones = np.ones((wp.batch, kv), np.uint8)
    assert np.array_equal(oracle.masked(wp, ones, lib=lib), oracle.prefill(wp, lib=lib))
    tri = np.zeros((wp.batch, wp.max_q_len, kv), np.uint8)
    for b in range(wp.batch):
        c = int(wp.seq_lens[b]) - int(wp.q_lens[b])
        for i in range(int(wp.q_lens[b])):
            tri[b, i, :c + i + 1] = 1
    assert np.array_equal(oracle.masked(wp, tri, causal=False, lib=lib), oracle.prefill(wp, lib=lib))
    m2 = workload.make_mask(wp, 2, seed=133, keep=0.5)
    m3 = np.repeat(m2[:, None, :], wp.max_q_len, axis=1)
    for causal in (True, False):
        assert np.array_equal(oracle.masked(wp, m2, causal=causal, lib=lib),
                              oracle.masked(wp, m3, causal=causal, lib=lib))


def pin_decode_mask_is_shorter_table(lib):
    """A decode mask equals decoding over a slot table that lists only the visible keys."""
    w = _small_decode(seed=137)
    m = workload.make_mask(w, 2, seed=139, keep=0.5)
    r2t = np.zeros_like(w.req_to_token)
    seq = np.zeros_like(w.seq_lens)
    for b in range(w.batch):
        keep = [int(w.req_to_token[b, j]) for j in range(int(w.seq_lens[b])) if m[b, j]]
        r2t[b, :len(keep)] = keep
        seq[b] = len(keep)
    kvi = np.concatenate([[0], np.cumsum(seq)]).astype(np.int32)
    short = dataclasses.replace(w, req_to_token=r2t, seq_lens=seq, kv_indptr=kvi)
    assert np.array_equal(oracle.masked(w, m, lib=lib), oracle.decode(short, lib=lib))


def pin_sdpa_head_dim_32(lib):
    """Head dim 32 (the size the pages' dispatch-switch commit adds) against fp64 SDPA, decode
    and prefill."""
    pin_sdpa_decode(lib, w=_small_decode(seed=141, Hq=8, Hkv=2, d=32))
    pin_sdpa_prefill(lib, w=_small_prefill(seed=143, Hq=8, Hkv=4, d=32))


ALL_PINS = [
    pin_sdpa_decode, pin_sdpa_prefill, pin_prefix0_is_textbook_causal, pin_golden,
    pin_q_zero_is_mean_of_visible_v, pin_single_key_returns_v, pin_per_request_marker, pin_dominant_key,
    pin_slot_permutation, pin_key_shift, pin_unreferenced_slots_unread, pin_split_combine, pin_chunk_partials_combine,
    pin_partial_ranges_match_even_split,
    pin_partial_is_softmax_piece, pin_prefill_row_is_decode,
    pin_append_then_attend_is_sdpa_over_concatenation, pin_append_touches_only_new_slots,
    pin_masked_matches_sdpa, pin_mask_identities, pin_decode_mask_is_shorter_table, pin_sdpa_head_dim_32,
]
