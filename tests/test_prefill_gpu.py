"""GPU parity of the tensor-core ragged prefill/extend (C ABI) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import workload
from workload import fp32_to_bf16_bits, make_from_lengths

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import prefill_attention_gb300 as pa  # noqa: E402
from gpu_util import TOL, prefill_dims, run_decode, run_prefill, to_f64, upload  # noqa: E402


def _err(got, ref):
    return float(np.abs(got - ref).max())


def test_prefill_config5_full():
    w = workload.config(5)
    got = to_f64(run_prefill(w))
    assert _err(got, oracle.prefill(w)) <= TOL


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (128, 8, 8), (128, 16, 8), (128, 64, 8), (128, 32, 2),
                                      (64, 8, 2), (64, 4, 4), (64, 16, 4), (64, 32, 2)])
def test_head_shapes(d, Hq, Hkv):
    rng = np.random.default_rng(d + Hq * 7 + Hkv)
    ql = np.array([1, 5, 31, 32, 33, 64, 100, 129])
    pre = np.array([0, 3, 0, 64, 17, 190, 1, 300])
    w = make_from_lengths(rng, kind="prefill", name="shapes", seq_lens=pre + ql, q_lens=ql, Hq=Hq, Hkv=Hkv, d=d)
    assert _err(to_f64(run_prefill(w)), oracle.prefill(w)) <= TOL


def test_prefix_zero_full_causal():
    rng = np.random.default_rng(3)
    ql = np.array([512, 7, 200])
    w = make_from_lengths(rng, kind="prefill", name="p0", seq_lens=ql, q_lens=ql, Hq=32, Hkv=8, d=128)
    assert _err(to_f64(run_prefill(w)), oracle.prefill(w)) <= TOL


def test_single_query_rows_equal_decode():
    """q_len = 1 for every request: prefill computes exactly the decode quantity."""
    rng = np.random.default_rng(4)
    seq = np.array([1, 65, 300, 2047])
    w = make_from_lengths(rng, kind="prefill", name="q1", seq_lens=seq, q_lens=np.ones(4, int), Hq=32, Hkv=8,
                          d=128)
    pf = to_f64(run_prefill(w))
    wd = workload.Workload(**{**w.__dict__, "kind": "decode", "qo_indptr": None})
    dc = to_f64(run_decode(wd))
    assert _err(pf, oracle.prefill(w)) <= TOL
    assert _err(pf, dc) <= 2 * TOL


def test_empty_requests_write_nothing():
    rng = np.random.default_rng(5)
    ql = np.array([3, 0, 40, 0])
    pre = np.array([10, 5, 0, 9])
    w = make_from_lengths(rng, kind="prefill", name="empty", seq_lens=pre + ql, q_lens=ql, Hq=8, Hkv=2, d=128)
    t = upload(w)
    out = torch.full_like(t["q"], 3.0)
    pa.astr_attn_prefill_ragged(t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], out,
                                prefill_dims(w), w.sm_scale)
    torch.cuda.synchronize()
    assert _err(to_f64(out), oracle.prefill(w)) <= TOL


def test_per_request_marker_exact():
    rng = np.random.default_rng(6)
    ql = np.array([1, 40, 130, 7])
    pre = np.array([0, 100, 33, 600])
    w = make_from_lengths(rng, kind="prefill", name="marker", seq_lens=pre + ql, q_lens=ql, Hq=32, Hkv=8, d=128)
    for b in range(w.batch):
        sl = w.req_to_token[b, :w.seq_lens[b]]
        w.v_pool[sl] = fp32_to_bf16_bits(np.full((len(sl), 8, 128), b + 1, np.float32))
    got = to_f64(run_prefill(w))
    owner = np.repeat(np.arange(w.batch), ql)
    assert np.array_equal(got, np.broadcast_to((owner + 1.0)[:, None, None], got.shape))


def test_poisoned_future_and_unreferenced_slots():
    """Keys past each row's causal limit, past seq_len, and unreferenced slots are NaN: output unchanged."""
    rng = np.random.default_rng(7)
    ql = np.array([9, 70, 1, 33])
    pre = np.array([5, 0, 64, 100])
    seq = pre + ql
    w = make_from_lengths(rng, kind="prefill", name="poison", seq_lens=seq, q_lens=ql, Hq=32, Hkv=8, d=128,
                          extra_slots=32, stride=256)
    base = to_f64(run_prefill(w))
    T = int(seq.sum())
    w.k_pool[T:] = 0x7FC0
    w.v_pool[T:] = 0x7FC0
    for b in range(w.batch):
        w.req_to_token[b, seq[b]:] = T + b
    got = to_f64(run_prefill(w))
    assert np.isfinite(got).all()
    assert np.array_equal(base, got)


def test_deterministic_bits():
    w = workload.config(5)
    t = upload(w)
    a = run_prefill(w, t).view(torch.int16).cpu().numpy()
    b = run_prefill(w, t).view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b)


def test_cuda_graph_replay_bit_exact():
    w = workload.config(5)
    t = upload(w)
    dims = prefill_dims(w)
    out = torch.empty_like(t["q"])
    args = (t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], out, dims, w.sm_scale)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pa.astr_attn_prefill_ragged(*args, stream=s)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.astr_attn_prefill_ragged(*args, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("scale", [-0.125, 0.0, 0.3])
def test_scale_sign_and_zero(scale):
    """The row max turns into a min for a negative scale; a zero scale gives the mean of the
    visible V rows (every logit 0)."""
    rng = np.random.default_rng(41)
    ql = np.array([1, 17, 64, 130])
    pre = np.array([0, 40, 3, 200])
    w = make_from_lengths(rng, kind="prefill", name="scale", seq_lens=pre + ql, q_lens=ql, Hq=8, Hkv=2, d=64,
                          sm_scale=scale)
    assert _err(to_f64(run_prefill(w)), oracle.prefill(w)) <= TOL


def test_many_requests_natural_order():
    """More requests than the kernel's shared-memory work-order table holds: the items are then
    dealt out in their natural order (the path every large batch takes)."""
    rng = np.random.default_rng(42)
    B = 1100
    ql = rng.integers(1, 5, B)
    pre = rng.integers(0, 21, B)
    w = make_from_lengths(rng, kind="prefill", name="many-req", seq_lens=pre + ql, q_lens=ql, Hq=8, Hkv=2, d=64)
    assert _err(to_f64(run_prefill(w)), oracle.prefill(w)) <= TOL


def test_many_items_sorted_order():
    """Many work items (KV head x query-tile pair), about 64 per CTA: still within the per-CTA
    list of the sorted order."""
    rng = np.random.default_rng(43)
    B = 600                          # 600 requests x 2 pairs x 8 KV heads = 9600 items
    ql = rng.integers(257, 281, B)   # G = 1: two 128-row tiles per pair, two pairs per request
    pre = rng.integers(0, 21, B)
    w = make_from_lengths(rng, kind="prefill", name="many-items", seq_lens=pre + ql, q_lens=ql, Hq=8, Hkv=8, d=64)
    assert _err(to_f64(run_prefill(w)), oracle.prefill(w)) <= TOL


def test_many_items_natural_order():
    """More work items than the per-CTA list of the sorted order holds (128 per CTA, i.e.
    19456 on 152 SMs): the items are then dealt out in their natural order."""
    rng = np.random.default_rng(44)
    B = 400                          # 400 requests x 2 pairs x 32 KV heads = 25600 items
    ql = rng.integers(257, 281, B)
    pre = rng.integers(0, 21, B)
    w = make_from_lengths(rng, kind="prefill", name="many-items-natural", seq_lens=pre + ql, q_lens=ql,
                          Hq=32, Hkv=32, d=64)
    assert _err(to_f64(run_prefill(w)), oracle.prefill(w)) <= TOL
