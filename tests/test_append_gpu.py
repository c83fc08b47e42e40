"""GPU parity of the KV-append step (C ABI) against the oracle: bit-exact pool bytes."""
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
from gpu_util import bf16_dev, decode_dims, i32_dev, prefill_dims, to_f64, upload  # noqa: E402


def _bits(t) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _append_dims(w, total_new):
    return pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride,
                        w.max_seq_len, total_q=total_new)


def run_append(w, qo, k_new, v_new, r2t=None):
    """Upload the pools of ``w``, append on the GPU, return the pools' bits."""
    kp, vp = bf16_dev(w.k_pool), bf16_dev(w.v_pool)
    table = w.req_to_token if r2t is None else r2t
    pa.astr_attn_kv_append(bf16_dev(k_new), bf16_dev(v_new), i32_dev(qo), i32_dev(table), i32_dev(w.seq_lens),
                           kp, vp, _append_dims(w, int(qo[-1])))
    torch.cuda.synchronize()
    return _bits(kp), _bits(vp)


def _check(w, qo, kn, vn):
    got_k, got_v = run_append(w, qo, kn, vn)
    ref_k, ref_v = oracle.kv_append(w, qo, kn, vn)
    assert np.array_equal(got_k, ref_k), "k_pool differs from the oracle"
    assert np.array_equal(got_v, ref_v), "v_pool differs from the oracle"


def test_append_extend_workload_full():
    """The 16-request extend workload: every new token of every request."""
    w = workload.config(5)
    qo, kn, vn = workload.append_rows(w, seed=501)
    _check(w, qo, kn, vn)


@pytest.mark.parametrize("cfg", [2, 4])
def test_append_decode_one_token_per_request(cfg):
    w = workload.config(cfg)
    qo, kn, vn = workload.append_rows(w, seed=502 + cfg)
    assert int(qo[-1]) == w.batch
    _check(w, qo, kn, vn)


@pytest.mark.parametrize("d,Hkv", [(64, 1), (64, 2), (128, 1), (128, 8), (128, 16), (64, 32)])
def test_append_ragged_with_empty_requests(d, Hkv):
    """q_len 0 requests, prefix 0, single-token requests; rows of 128 B to 8 KB (the last two
    take more than one round of loads per lane)."""
    rng = np.random.default_rng(d * 3 + Hkv)
    ql = np.array([0, 1, 7, 0, 33, 128, 1, 0, 250])
    pre = np.array([5, 0, 0, 0, 64, 3, 999, 2, 17])
    w = make_from_lengths(rng, kind="prefill", name="append-ragged", seq_lens=pre + ql, q_lens=ql, Hq=Hkv,
                          Hkv=Hkv, d=d, stride=1100)
    qo, kn, vn = workload.append_rows(w, seed=7)
    _check(w, qo, kn, vn)


@pytest.mark.parametrize("B", [1, 31, 32, 33, 1025, 3000])
def test_append_request_search_sizes(B):
    """Request lookup over one to three search rounds (32-way per round)."""
    rng = np.random.default_rng(B)
    ql = rng.integers(0, 4, size=B)
    ql[rng.integers(0, B)] = 1  # at least one new token
    pre = rng.integers(0, 20, size=B)
    w = make_from_lengths(rng, kind="prefill", name="append-search", seq_lens=pre + ql, q_lens=ql, Hq=8, Hkv=2,
                          d=64, stride=32)
    qo, kn, vn = workload.append_rows(w, seed=B + 1)
    _check(w, qo, kn, vn)


def test_append_skips_slot_ids_outside_the_pool():
    """A new token whose slot id is outside [0, num_slots) writes nothing; the others land."""
    rng = np.random.default_rng(17)
    ql = np.array([3, 4, 2])
    pre = np.array([2, 0, 5])
    w = make_from_lengths(rng, kind="prefill", name="append-bad-slot", seq_lens=pre + ql, q_lens=ql, Hq=4, Hkv=2,
                          d=128, stride=16)
    qo, kn, vn = workload.append_rows(w, seed=3)
    ref_k, ref_v = oracle.kv_append(w, qo, kn, vn)
    table = w.req_to_token.copy()
    for b, i, bad in ((0, 1, w.num_slots), (1, 3, -1), (2, 0, 1 << 30)):
        pos = int(w.seq_lens[b]) - int(ql[b]) + i
        slot = int(table[b, pos])
        ref_k[slot], ref_v[slot] = w.k_pool[slot], w.v_pool[slot]  # that token's slot keeps its bytes
        table[b, pos] = bad
    got_k, got_v = run_append(w, qo, kn, vn, r2t=table)
    assert np.array_equal(got_k, ref_k) and np.array_equal(got_v, ref_v)


def test_append_nothing_to_do():
    w = workload.config(1)
    kp, vp = bf16_dev(w.k_pool), bf16_dev(w.v_pool)
    qo = i32_dev(np.zeros(w.batch + 1, np.int32))
    empty = bf16_dev(np.zeros((1, w.num_kv_heads, w.head_dim), np.uint16))
    st = pa.astr_attn_kv_append(empty, empty, qo, i32_dev(w.req_to_token), i32_dev(w.seq_lens), kp, vp,
                                _append_dims(w, 0))
    torch.cuda.synchronize()
    assert st == pa.ASTR_OK
    assert np.array_equal(_bits(kp), w.k_pool) and np.array_equal(_bits(vp), w.v_pool)


def _cleared(w, qo):
    """The pools of ``w`` with the new tokens' slots zeroed, and those tokens' rows."""
    slots = []
    for b in range(w.batch):
        n = int(qo[b + 1] - qo[b])
        c = int(w.seq_lens[b]) - n
        slots.extend(int(s) for s in w.req_to_token[b, c:c + n])
    slots = np.array(slots, np.int64)
    kn, vn = w.k_pool[slots].copy(), w.v_pool[slots].copy()
    kp, vp = w.k_pool.copy(), w.v_pool.copy()
    kp[slots] = 0
    vp[slots] = 0
    return dataclasses.replace(w, k_pool=kp, v_pool=vp), kn, vn


def test_append_then_prefill_matches_oracle():
    """Write-then-gather: the extend workload's new K/V appended into a pool that lacks them,
    then the prefill over that pool, against the oracle's prefill of the complete pool."""
    w = workload.config(5)
    qo = np.asarray(w.qo_indptr, np.int32)
    wc, kn, vn = _cleared(w, qo)
    d = upload(wc)
    st = pa.astr_attn_kv_append(bf16_dev(kn), bf16_dev(vn), d["qo"], d["r2t"], d["seq"], d["k"], d["v"],
                                _append_dims(w, w.total_q))
    assert st == pa.ASTR_OK
    out = torch.empty_like(d["q"])
    pa.astr_attn_prefill_ragged(d["q"], d["qo"], d["k"], d["v"], d["r2t"], d["seq"], d["kvi"], out, prefill_dims(w),
                                w.sm_scale)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(d["k"]), w.k_pool) and np.array_equal(_bits(d["v"]), w.v_pool)
    rng = np.random.default_rng(5)
    rows = np.stack([rng.integers(0, w.total_q, 512), rng.integers(0, w.num_qo_heads, 512)], axis=1)
    ref = oracle.prefill(w, rows=rows)
    got = to_f64(out)[rows[:, 0], rows[:, 1]]
    assert float(np.abs(got - ref).max()) <= 1e-2


def test_append_then_decode_in_one_graph():
    """Decode step order (append the current token, then attend), captured once in a CUDA
    graph and replayed: outputs equal the oracle's decode of the complete pool."""
    w = workload.config(2)
    qo = np.arange(w.batch + 1, dtype=np.int32)
    wc, kn, vn = _cleared(w, qo)
    d = upload(wc)
    dk, dv, dqo = bf16_dev(kn), bf16_dev(vn), i32_dev(qo)
    dims = decode_dims(w)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.empty_like(d["q"])
    adims = _append_dims(w, w.batch)
    s = torch.cuda.Stream()

    def step():
        pa.astr_attn_kv_append(dk, dv, dqo, d["r2t"], d["seq"], d["k"], d["v"], adims, stream=s)
        pa.astr_attn_paged_decode(d["q"], d["k"], d["v"], d["r2t"], d["seq"], d["kvi"], o_part, ml_part, out, dims,
                                  w.sm_scale, stream=s)

    with torch.cuda.stream(s):
        step()  # eager run first (sets the decode kernel's attributes outside the capture)
    torch.cuda.synchronize()
    eager = out.clone()
    d["k"].copy_(bf16_dev(wc.k_pool))
    d["v"].copy_(bf16_dev(wc.v_pool))
    out.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(_bits(d["k"]), w.k_pool) and np.array_equal(_bits(d["v"]), w.v_pool)
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert float(np.abs(to_f64(out) - oracle.decode(w)).max()) <= 1e-2
