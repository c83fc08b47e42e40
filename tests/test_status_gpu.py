"""The status word (dims.status): errors that only the GPU can see reach the caller.

* A pipeline wait that runs out (forced here with a tiny dims.wait_limit on ordinary inputs)
  makes the kernels give up, report ASTR_KSTATUS_TIMEOUT and return; the stream
  synchronises (nothing is left waiting) and the next ordinary call on the same context is
  correct.
* A slot id outside the pool, or a key position past the table row, reads as a zero row (the
  KV append skips that token), touches no memory outside the buffers and is reported as
  ASTR_KSTATUS_BAD_INPUT; the other requests' outputs are unaffected.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import workload
from workload import make_from_lengths

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import prefill_attention_gb300 as pa  # noqa: E402
from gpu_util import TOL, bf16_dev, i32_dev, to_f64, upload  # noqa: E402


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _decode(w, t, status, wait_limit=0, max_splits=32, max_seq_len=None, r2t=None):
    dims = pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride,
                        w.max_seq_len if max_seq_len is None else max_seq_len, max_splits=max_splits,
                        status=status, wait_limit=wait_limit)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.zeros_like(t["q"])
    st = pa.astr_attn_paged_decode(t["q"], t["k"], t["v"], t["r2t"] if r2t is None else r2t, t["seq"], t["kvi"],
                                   o_part, ml_part, out, dims, w.sm_scale)
    assert st == pa.ASTR_OK
    torch.cuda.synchronize()
    return out


def _prefill(w, t, status, wait_limit=0, max_seq_len=None, r2t=None):
    dims = pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride,
                        w.max_seq_len if max_seq_len is None else max_seq_len, total_q=w.total_q,
                        max_q_len=w.max_q_len, status=status, wait_limit=wait_limit)
    out = torch.zeros_like(t["q"])
    st = pa.astr_attn_prefill_ragged(t["q"], t["qo"], t["k"], t["v"], t["r2t"] if r2t is None else r2t, t["seq"],
                                     t["kvi"], out, dims, w.sm_scale)
    assert st == pa.ASTR_OK
    torch.cuda.synchronize()
    return out


# wait_limit = 1: every wait is a single non-blocking test, and each kernel's first wait comes
# before the data it waits for can have arrived (that takes dependent global-memory round trips
# issued at about the same time), so it runs out
def test_decode_wait_that_runs_out_is_reported_and_the_context_survives():
    w = workload.config(2)
    t = upload(w)
    for _ in range(2):
        status = _status()
        out = _decode(w, t, status, wait_limit=1)  # returns: no kernel is left waiting
        assert int(status.item()) & pa.ASTR_KSTATUS_TIMEOUT
        assert torch.isnan(out.float()).any(), "the rows of the pairs that gave up are poisoned"
    status.zero_()
    got = to_f64(_decode(w, t, status))
    assert int(status.item()) == 0
    assert np.abs(got - oracle.decode(w)).max() <= TOL


def test_prefill_wait_that_runs_out_is_reported_and_the_context_survives():
    w = workload.make_prefill(6, 32, 8, 128, (1, 300), (0, 500), seed=71, name="timeout")
    t = upload(w)
    for _ in range(2):
        status = _status()
        _prefill(w, t, status, wait_limit=1)
        assert int(status.item()) & pa.ASTR_KSTATUS_TIMEOUT
    status.zero_()
    got = to_f64(_prefill(w, t, status))
    assert int(status.item()) == 0
    assert np.abs(got - oracle.prefill(w)).max() <= TOL


def _with_zero_slot(w):
    """w with one more pool row, all zeros (what the kernels read for a bad key)."""
    z = np.zeros((1, w.num_kv_heads, w.head_dim), np.uint16)
    return dataclasses.replace(w, k_pool=np.concatenate([w.k_pool, z]), v_pool=np.concatenate([w.v_pool, z]))


def test_decode_slot_id_outside_the_pool_is_reported():
    rng = np.random.default_rng(801)
    w = make_from_lengths(rng, kind="decode", name="bad-id", seq_lens=[40, 100, 7, 300], q_lens=None, Hq=8, Hkv=2,
                          d=64)
    bad = w.req_to_token.copy()
    bad[1, 50] = w.num_slots + 1000
    bad[3, 0] = -5
    t = upload(w)
    status = _status()
    got = to_f64(_decode(w, t, status, r2t=i32_dev(bad)))
    assert int(status.item()) == pa.ASTR_KSTATUS_BAD_INPUT
    # reference: the bad keys as zero rows
    wz = _with_zero_slot(w)
    r2t = bad.copy()
    r2t[1, 50] = r2t[3, 0] = w.num_slots
    ref = oracle.decode(dataclasses.replace(wz, req_to_token=r2t))
    assert np.abs(got - ref).max() <= TOL


def test_decode_key_position_past_the_table_row_is_not_read():
    """seq_lens of the last request beyond r2t_stride (a broken precondition): positions past
    the row are not read (the table is followed by a guard row, so even a stray read would stay
    inside the allocation) and are reported."""
    rng = np.random.default_rng(803)
    seq = np.array([30, 64, 50, 64])
    w = make_from_lengths(rng, kind="decode", name="past-row", seq_lens=seq, q_lens=None, Hq=8, Hkv=2, d=64,
                          stride=64)
    t = upload(w)
    long_seq = seq.copy()
    long_seq[3] = 80
    kvi = np.concatenate([[0], np.cumsum(long_seq)]).astype(np.int32)
    table = np.concatenate([w.req_to_token, np.zeros((1, 64), np.int32)])  # guard row
    r2t = i32_dev(table)
    t["seq"], t["kvi"] = i32_dev(long_seq), i32_dev(kvi)
    status = _status()
    got = to_f64(_decode(w, t, status, r2t=r2t, max_seq_len=64))
    assert int(status.item()) == pa.ASTR_KSTATUS_BAD_INPUT
    wz = _with_zero_slot(w)
    r2t_ref = np.full((4, 80), w.num_slots, np.int32)
    r2t_ref[:, :64] = w.req_to_token
    ref = oracle.decode(dataclasses.replace(wz, req_to_token=r2t_ref, seq_lens=long_seq.astype(np.int32),
                                            kv_indptr=kvi))
    assert np.abs(got - ref).max() <= TOL


def test_prefill_bad_slot_id_and_position_past_the_row_are_reported():
    rng = np.random.default_rng(805)
    ql = np.array([5, 64, 1, 30])
    seq = np.array([40, 64, 100, 64])
    w = make_from_lengths(rng, kind="prefill", name="bad-pf", seq_lens=seq, q_lens=ql, Hq=8, Hkv=2, d=128,
                          stride=100)
    bad = w.req_to_token.copy()
    bad[2, 10] = w.num_slots + 7
    t = upload(w)
    status = _status()
    got = to_f64(_prefill(w, t, status, r2t=i32_dev(bad)))
    assert int(status.item()) == pa.ASTR_KSTATUS_BAD_INPUT
    wz = _with_zero_slot(w)
    r2t = bad.copy()
    r2t[2, 10] = w.num_slots
    assert np.abs(got - oracle.prefill(dataclasses.replace(wz, req_to_token=r2t))).max() <= TOL
    # request 2's 100 keys past a table pitch of 64 (a guard row keeps any stray read inside)
    table = np.zeros((w.batch + 1, 64), np.int32)
    table[:w.batch] = w.req_to_token[:, :64]
    status.zero_()
    dims = pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, 64, 64,
                        total_q=w.total_q, max_q_len=w.max_q_len, status=status)
    out = torch.zeros_like(t["q"])
    st = pa.astr_attn_prefill_ragged(t["q"], t["qo"], t["k"], t["v"], i32_dev(table), t["seq"], t["kvi"], out, dims,
                                     w.sm_scale)
    assert st == pa.ASTR_OK
    torch.cuda.synchronize()
    assert int(status.item()) == pa.ASTR_KSTATUS_BAD_INPUT
    # the requests that stay inside the row are unaffected
    rows = np.concatenate([np.arange(w.qo_indptr[b], w.qo_indptr[b + 1]) for b in (0, 1, 3)])
    assert np.abs(to_f64(out)[rows] - oracle.prefill(w)[rows]).max() <= TOL


def test_append_slot_outside_the_pool_is_skipped_and_reported():
    w = workload.make_prefill(4, 8, 2, 64, (1, 20), (0, 30), seed=807, name="bad-append")
    qo, k_new, v_new = workload.append_rows(w, seed=808)
    bad = w.req_to_token.copy()
    c0 = int(w.seq_lens[0]) - int(w.q_lens[0])
    bad[0, c0] = w.num_slots + 3   # request 0's first new token
    t = upload(w)
    status = _status()
    dims = pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride,
                        w.max_seq_len, total_q=w.total_q, max_q_len=w.max_q_len, status=status)
    pa.astr_attn_kv_append(bf16_dev(k_new), bf16_dev(v_new), i32_dev(qo), i32_dev(bad), t["seq"], t["k"], t["v"],
                           dims)
    torch.cuda.synchronize()
    assert int(status.item()) == pa.ASTR_KSTATUS_BAD_INPUT
    kp, vp = oracle.kv_append(w, qo, k_new, v_new)
    skipped = int(w.req_to_token[0, c0])   # the slot the token would have gone to keeps its bytes
    kp[skipped], vp[skipped] = w.k_pool[skipped], w.v_pool[skipped]
    assert np.array_equal(t["k"].view(torch.int16).cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(t["v"].view(torch.int16).cpu().numpy().view(np.uint16), vp)


def test_clean_inputs_leave_the_status_word_zero():
    for w in (workload.config(1), workload.config(5)):
        t = upload(w)
        status = _status()
        if w.kind == "decode":
            _decode(w, t, status)
        else:
            _prefill(w, t, status)
        assert int(status.item()) == 0


def test_prefill_v_outside_the_fp16_range_is_reported():
    """P V runs in fp16: a V element beyond 65504 is reported (ASTR_KSTATUS_RANGE); requests
    that do not read it are unaffected."""
    w = workload.make_prefill(4, 8, 2, 128, (1, 40), (0, 60), seed=809, name="range")
    slot = int(w.req_to_token[1, 0])
    w.v_pool[slot, 0, 5] = workload.fp32_to_bf16_bits(np.array([1.0e5], np.float32))[0]
    t = upload(w)
    status = _status()
    got = to_f64(_prefill(w, t, status))
    assert int(status.item()) == pa.ASTR_KSTATUS_RANGE
    rows = np.concatenate([np.arange(w.qo_indptr[b], w.qo_indptr[b + 1]) for b in (0, 2, 3)])
    assert np.abs(got[rows] - oracle.prefill(w)[rows]).max() <= TOL
    # at the limit itself (65280 = the largest bf16 that fits fp16) nothing is reported and the
    # result is right
    w.v_pool[slot, 0, 5] = workload.fp32_to_bf16_bits(np.array([65280.0], np.float32))[0]
    t = upload(w)
    status.zero_()
    got = to_f64(_prefill(w, t, status))
    assert int(status.item()) == 0
    ref = oracle.prefill(w)
    # the large column carries the bf16 output's relative rounding (2^-8), the rest 1e-2
    assert np.all(np.abs(got - ref) <= TOL + 2.0 ** -7 * np.abs(ref))
