"""GPU parity of the split-KV paged decode (C ABI) against the fp64 oracle.

Tolerance: max abs error <= 1e-2 on bf16 outputs; slot-table routing bit-exact.
"""
import numpy as np
import pytest

import oracle
import workload
from workload import bf16_bits_to_fp32, fp32_to_bf16_bits, make_from_lengths

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import prefill_attention_gb300 as pa  # noqa: E402
import split_schedule  # noqa: E402
from gpu_util import SLOT_KEYS, TOL, decode_chunk_slots, decode_dims, run_decode, to_f64, upload  # noqa: E402


def _err(got, ref):
    return float(np.abs(got - ref).max())


@pytest.mark.parametrize("cfg", [1, 2])
def test_decode_config_full(cfg):
    w = workload.config(cfg)
    got = to_f64(run_decode(w))
    assert _err(got, oracle.decode(w)) <= TOL


@pytest.mark.parametrize("cfg", [3, 4])
def test_decode_config_full_long_and_large(cfg):
    """The long-context (B=8, seq 16K-32K) and large-batch (B=256, seq 512-4096) workloads, every
    (request, head) row against the fp64 oracle."""
    w = workload.config(cfg)
    got = to_f64(run_decode(w))
    assert np.isfinite(got).all()
    assert _err(got, oracle.decode(w)) <= TOL


@pytest.mark.parametrize("n_chunks", [1, 2, 3, 5, 16, 32, 200])
def test_forced_chunk_counts(n_chunks):
    w = workload.config(1)
    got = to_f64(run_decode(w, max_splits=32, num_splits=n_chunks))
    assert _err(got, oracle.decode(w)) <= TOL


@pytest.mark.parametrize("max_splits", [1, 2, 3, 64])
def test_workspace_capacity_floor(max_splits):
    """A small partial capacity raises the chunk floor; results stay correct."""
    w = workload.config(2)
    got = to_f64(run_decode(w, max_splits=max_splits))
    assert _err(got, oracle.decode(w)) <= TOL


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (128, 8, 8), (128, 16, 8), (128, 64, 8), (128, 128, 8),
                                      (64, 8, 2), (64, 4, 4), (64, 8, 4), (64, 16, 2), (64, 32, 2)])
def test_head_shapes_and_ragged_tails(d, Hq, Hkv):
    rng = np.random.default_rng(d * 1000 + Hq * 10 + Hkv)
    seq = [1, 7, 8, 9, 31, 33, 64, 65, 127, 128, 129, 200, 257, 0, 600]
    w = make_from_lengths(rng, kind="decode", name="shapes", seq_lens=seq, q_lens=None, Hq=Hq, Hkv=Hkv, d=d)
    for n in (0, 1, 4, 37):
        got = to_f64(run_decode(w, num_splits=n))
        assert _err(got, oracle.decode(w)) <= TOL, f"n_chunks={n}"


def test_partials_match_oracle_chunks():
    w = workload.config(1)
    max_splits, n = 8, 5
    out, o, ml, n_used = run_decode(w, max_splits=max_splits, num_splits=n, return_parts=True)
    assert n_used == n
    C = decode_chunk_slots(w, n, max_splits)
    o_ref, ml_ref, ns = split_schedule.chunk_partials(w, C, max_splits, SLOT_KEYS)
    assert ns.max() <= max_splits
    assert (ns >= 2).any()
    for b in range(w.batch):
        k = int(ns[b])
        if k < 2:   # single-chunk requests are written to `out` directly, without partials
            continue
        m, l = ml[b, :, :k, 0], ml[b, :, :k, 1]
        assert np.abs(m - ml_ref[b, :, :k, 0]).max() <= 1e-3
        assert np.abs(l / ml_ref[b, :, :k, 1] - 1).max() <= 1e-3
        norm = o[b, :, :k] / l[..., None]
        norm_ref = o_ref[b, :, :k] / ml_ref[b, :, :k, 1][..., None]
        assert np.abs(norm - norm_ref).max() <= TOL
    assert _err(to_f64(out), oracle.decode(w)) <= TOL


def test_combine_alone_on_oracle_chunk_partials():
    w = workload.config(1)
    max_splits, n = 8, 7
    dims = decode_dims(w, max_splits=max_splits, num_splits=n)
    C = decode_chunk_slots(w, n, max_splits)
    o_ref, ml_ref, ns = split_schedule.chunk_partials(w, C, max_splits, SLOT_KEYS)
    o_part = torch.from_numpy(np.nan_to_num(o_ref).astype(np.float32)).cuda().contiguous()
    ml_part = torch.from_numpy(np.nan_to_num(ml_ref).astype(np.float32)).cuda().contiguous()
    out = torch.empty((w.batch, w.num_qo_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    kvi = torch.from_numpy(w.kv_indptr).cuda()
    pa.astr_attn_decode_combine(o_part, ml_part, None, kvi, out, dims)
    torch.cuda.synchronize()
    assert _err(to_f64(out), oracle.decode(w)) <= TOL


def test_combine_alone_explicit_layout():
    """kv_indptr = NULL: every (b, h) row holds num_splits partials (here an even split)."""
    w = workload.config(1)
    S = 4
    o_ref, ml_ref = oracle.decode_split_partials(w, S)
    dims = decode_dims(w, max_splits=S, num_splits=S)
    o_part = torch.from_numpy(o_ref.astype(np.float32)).cuda().contiguous()
    ml_part = torch.from_numpy(ml_ref.astype(np.float32)).cuda().contiguous()
    out = torch.empty((w.batch, w.num_qo_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    pa.astr_attn_decode_combine(o_part, ml_part, None, None, out, dims)
    torch.cuda.synchronize()
    assert _err(to_f64(out), oracle.combine(o_ref, ml_ref)) <= TOL


def test_deterministic_bits():
    w = workload.config(2)
    t = upload(w)
    a = run_decode(w, t).view(torch.int16).cpu().numpy()
    b = run_decode(w, t).view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b)


def test_slot_permutation_bit_exact():
    """Paged == contiguous: identity slot table vs a permuted one, same S, same bits."""
    rng = np.random.default_rng(5)
    w = make_from_lengths(rng, kind="decode", name="perm", seq_lens=[100, 37, 512, 1], q_lens=None, Hq=32, Hkv=8,
                          d=128)
    T = w.num_slots
    # contiguous: token j of request b in slot kv_indptr[b] + j
    k_c = np.empty_like(w.k_pool); v_c = np.empty_like(w.v_pool)
    r2t_c = np.zeros_like(w.req_to_token)
    for b in range(w.batch):
        n = w.seq_lens[b]
        src = w.req_to_token[b, :n]
        dst = np.arange(w.kv_indptr[b], w.kv_indptr[b] + n)
        k_c[dst] = w.k_pool[src]; v_c[dst] = w.v_pool[src]
        r2t_c[b, :n] = dst
    wc = workload.Workload(**{**w.__dict__, "k_pool": k_c, "v_pool": v_c, "req_to_token": r2t_c})
    a = run_decode(w, num_splits=3).view(torch.int16).cpu().numpy()
    b = run_decode(wc, num_splits=3).view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b)
    assert T == int(w.seq_lens.sum())


def test_per_request_marker_exact():
    rng = np.random.default_rng(6)
    seq = [5, 300, 64, 1000, 2, 129]
    w = make_from_lengths(rng, kind="decode", name="marker", seq_lens=seq, q_lens=None, Hq=32, Hkv=8, d=128)
    for b in range(w.batch):
        sl = w.req_to_token[b, :seq[b]]
        w.v_pool[sl] = fp32_to_bf16_bits(np.full((len(sl), 8, 128), b + 1, np.float32))
    got = to_f64(run_decode(w))
    ref = np.broadcast_to((np.arange(w.batch) + 1.0)[:, None, None], got.shape)
    assert np.array_equal(got, ref)


def test_single_key_returns_v_exactly():
    rng = np.random.default_rng(8)
    w = make_from_lengths(rng, kind="decode", name="one", seq_lens=[1] * 5, q_lens=None, Hq=32, Hkv=8, d=128)
    got = to_f64(run_decode(w))
    v = bf16_bits_to_fp32(w.v_pool).astype(np.float64)
    for b in range(5):
        for h in range(32):
            assert np.array_equal(got[b, h], v[w.req_to_token[b, 0], h // 4])


def test_poisoned_unreferenced_slots_are_never_read():
    rng = np.random.default_rng(9)
    seq = np.array([50, 3, 700, 129])
    w = make_from_lengths(rng, kind="decode", name="poison", seq_lens=seq, q_lens=None, Hq=32, Hkv=8, d=128,
                          extra_slots=64, stride=1024)
    base = to_f64(run_decode(w, num_splits=5))
    T = int(seq.sum())
    w.k_pool[T:] = 0x7FC0
    w.v_pool[T:] = 0x7FC0
    for b in range(w.batch):
        w.req_to_token[b, seq[b]:] = T + (b * 7) % 64
    got = to_f64(run_decode(w, num_splits=5))
    assert np.isfinite(got).all()
    assert np.array_equal(base, got)


def test_zero_length_request_gives_zeros():
    rng = np.random.default_rng(10)
    w = make_from_lengths(rng, kind="decode", name="empty", seq_lens=[0, 40, 0, 3], q_lens=None, Hq=8, Hkv=2, d=64,
                          stride=64)
    got = to_f64(run_decode(w, num_splits=4))
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert _err(got, oracle.decode(w)) <= TOL


def test_q_zero_is_mean_of_v():
    rng = np.random.default_rng(11)
    w = make_from_lengths(rng, kind="decode", name="q0", seq_lens=[10, 999, 64], q_lens=None, Hq=32, Hkv=8, d=128)
    w.q[:] = 0
    got = to_f64(run_decode(w))
    v = bf16_bits_to_fp32(w.v_pool).astype(np.float64)
    for b in range(w.batch):
        ref = v[w.req_to_token[b, :w.seq_lens[b]]].mean(axis=0)  # [Hkv, d]
        assert np.abs(got[b] - np.repeat(ref, 4, axis=0)).max() <= TOL


def test_runs_on_callers_stream():
    w = workload.config(1)
    t = upload(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = run_decode(w, t, stream=s)
    assert _err(to_f64(out), oracle.decode(w)) <= TOL


def test_cuda_graph_replay_bit_exact():
    w = workload.config(2)
    t = upload(w)
    dims = decode_dims(w, max_splits=32)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.empty_like(t["q"])
    args = (t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, out, dims, w.sm_scale)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pa.astr_attn_paged_decode(*args, stream=s)   # eager run (also sets kernel attributes)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.astr_attn_paged_decode(*args, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_guard_bands_untouched():
    w = workload.config(1)
    t = upload(w)
    dims = decode_dims(w, max_splits=8)
    ob, mb = pa.astr_attn_decode_workspace_bytes(dims)
    pad = 256
    o_buf = torch.full((ob // 4 + 2 * pad,), 12345.0, device="cuda")
    m_buf = torch.full((mb // 4 + 2 * pad,), 12345.0, device="cuda")
    n_out = w.batch * w.num_qo_heads * w.head_dim
    out_buf = torch.full((n_out + 2 * pad,), 7.0, device="cuda", dtype=torch.bfloat16)
    pa.astr_attn_paged_decode(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_buf[pad:pad + ob // 4],
                              m_buf[pad:pad + mb // 4], out_buf[pad:pad + n_out], dims, w.sm_scale)
    torch.cuda.synchronize()
    for buf, n, val in ((o_buf, ob // 4, 12345.0), (m_buf, mb // 4, 12345.0), (out_buf, n_out, 7.0)):
        assert torch.all(buf[:pad] == val) and torch.all(buf[pad + n:] == val)
    got = to_f64(out_buf[pad:pad + n_out].view(w.batch, w.num_qo_heads, w.head_dim))
    assert _err(got, oracle.decode(w)) <= TOL


def test_split_then_combine_entry_points():
    """astr_attn_decode_split + astr_attn_decode_combine == astr_attn_paged_decode (bit-exact)."""
    w = workload.config(2)
    t = upload(w)
    dims = decode_dims(w, max_splits=16)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.empty_like(t["q"])
    pa.astr_attn_decode_split(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, dims,
                              w.sm_scale)
    pa.astr_attn_decode_combine(o_part, ml_part, t["seq"], t["kvi"], out, dims)
    torch.cuda.synchronize()
    got = to_f64(out)
    assert _err(got, oracle.decode(w)) <= TOL
    ref = run_decode(w, t, max_splits=16)
    assert np.abs(got - to_f64(ref)).max() <= TOL


@pytest.mark.parametrize("scale", [-0.125, 0.0, 0.3])
def test_scale_sign_and_zero(scale):
    rng = np.random.default_rng(44)
    seq = [1, 33, 200, 517, 0, 64]
    w = make_from_lengths(rng, kind="decode", name="scale", seq_lens=seq, q_lens=None, Hq=8, Hkv=2, d=64,
                          sm_scale=scale)
    for n in (0, 3):
        got = to_f64(run_decode(w, num_splits=n))
        assert _err(got, oracle.decode(w)) <= TOL, f"n_chunks={n}"


@pytest.mark.parametrize("B", [33, 64, 257, 300])
def test_batch_sizes_around_warmup_rounds(B):
    """Batches that take the one-round (B <= 32), partly filled multi-round (33-256) and
    skipped (B > 256) L2 warm-up before the dependency wait; results must not depend on it."""
    rng = np.random.default_rng(500 + B)
    seq = rng.integers(0, 97, B)
    seq[::17] = 0   # some empty requests
    w = make_from_lengths(rng, kind="decode", name="warm", seq_lens=seq, q_lens=None, Hq=8, Hkv=2, d=64)
    for n in (0, 37):
        got = to_f64(run_decode(w, num_splits=n))
        assert _err(got, oracle.decode(w)) <= TOL, f"n_chunks={n}"


def test_request_longer_than_max_seq_len_stays_in_bounds():
    """max_seq_len understated for one request: its pieces past max_splits partial slots are
    not written (its row is then wrong), every other row is right and no byte outside the
    workspace changes."""
    rng = np.random.default_rng(611)
    seq = np.array([20, 33, 200, 7, 40, 1])
    w = make_from_lengths(rng, kind="decode", name="overlong", seq_lens=seq, q_lens=None, Hq=8, Hkv=2, d=64)
    t = upload(w)
    max_splits = 3
    dims = pa.make_dims(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.num_slots, w.r2t_stride, 40,
                        max_splits=max_splits, num_splits=64)
    ob, mb = pa.astr_attn_decode_workspace_bytes(dims)
    pad = 256
    o_buf = torch.full((ob // 4 + 2 * pad,), 12345.0, device="cuda")
    m_buf = torch.full((mb // 4 + 2 * pad,), 12345.0, device="cuda")
    n_out = w.batch * w.num_qo_heads * w.head_dim
    out_buf = torch.full((n_out + 2 * pad,), 7.0, device="cuda", dtype=torch.bfloat16)
    pa.astr_attn_paged_decode(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_buf[pad:pad + ob // 4],
                              m_buf[pad:pad + mb // 4], out_buf[pad:pad + n_out], dims, w.sm_scale)
    torch.cuda.synchronize()
    for buf, n, val in ((o_buf, ob // 4, 12345.0), (m_buf, mb // 4, 12345.0), (out_buf, n_out, 7.0)):
        assert torch.all(buf[:pad] == val) and torch.all(buf[pad + n:] == val)
    got = to_f64(out_buf[pad:pad + n_out].view(w.batch, w.num_qo_heads, w.head_dim))
    ref = oracle.decode(w)
    ok_rows = [b for b in range(w.batch) if seq[b] <= 40]
    assert _err(got[ok_rows], ref[ok_rows]) <= TOL
