"""GPU parity of the explicit-mask entry points (2-D / 3-D masks, causal on or off) against
the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import workload
from workload import make_from_lengths, make_mask

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import prefill_attention_gb300 as pa  # noqa: E402
from gpu_util import TOL, decode_dims, prefill_dims, to_f64, upload  # noqa: E402


def _dev_mask(m):
    return torch.from_numpy(np.ascontiguousarray(m, dtype=np.uint8)).cuda()


def run_prefill_masked(w, m, causal=True):
    t = upload(w)
    out = torch.full_like(t["q"], float("nan"))
    dm = None if m is None else _dev_mask(m)
    pa.astr_attn_prefill_ragged_masked(t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"],
                                       pa.make_mask(dm, causal), out, prefill_dims(w), w.sm_scale)
    torch.cuda.synchronize()
    return out


def run_decode_masked(w, m, max_splits=32, num_splits=0):
    t = upload(w)
    dims = decode_dims(w, max_splits=max_splits, num_splits=num_splits)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.full_like(t["q"], float("nan"))
    pa.astr_attn_paged_decode_masked(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], pa.make_mask(_dev_mask(m)),
                                     o_part, ml_part, out, dims, w.sm_scale)
    torch.cuda.synchronize()
    return out


def _err(got, ref):
    return float(np.abs(got - ref).max())


@pytest.mark.parametrize("dims,causal", [(3, True), (2, False), (3, False), (2, True)])
def test_prefill_extend_workload_masked(dims, causal):
    w = workload.config(5)
    m = make_mask(w, dims, seed=40 + dims, keep=0.75)
    got = to_f64(run_prefill_masked(w, m, causal))
    assert _err(got, oracle.masked(w, m, causal=causal)) <= TOL


def test_prefill_causal_off_without_mask():
    rng = np.random.default_rng(61)
    ql = np.array([1, 5, 64, 100, 129, 300])
    pre = np.array([0, 3, 0, 190, 17, 40])
    w = make_from_lengths(rng, kind="prefill", name="noncausal", seq_lens=pre + ql, q_lens=ql, Hq=32, Hkv=8, d=128)
    ones = np.ones((w.batch, -(-w.max_seq_len // 16) * 16), np.uint8)
    got = to_f64(run_prefill_masked(w, None, causal=False))
    assert _err(got, oracle.masked(w, ones, causal=False)) <= TOL


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (128, 8, 8), (128, 16, 8), (128, 64, 4), (128, 32, 16),
                                      (64, 8, 2), (64, 4, 4), (64, 16, 4), (64, 32, 2), (64, 32, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_masked_head_shapes_and_ragged_rows(d, Hq, Hkv, causal):
    """3-D masks over ragged lengths, with a fully masked row, a fully masked request and a row
    whose only visible key is the last one."""
    rng = np.random.default_rng(d + Hq * 7 + Hkv + int(causal))
    ql = np.array([1, 5, 31, 33, 64, 100, 129, 2])
    pre = np.array([0, 3, 0, 64, 17, 190, 1, 40])
    w = make_from_lengths(rng, kind="prefill", name="mask-shapes", seq_lens=pre + ql, q_lens=ql, Hq=Hq, Hkv=Hkv, d=d)
    m = make_mask(w, 3, seed=7, keep=0.6)
    m[1, 2, :] = 0          # one row sees nothing
    m[7, :, :] = 0          # one request sees nothing
    m[5, 0, :] = 0
    m[5, 0, int(w.seq_lens[5]) - int(ql[5])] = 1  # row 0 of request 5: only its causal-edge key
    got = to_f64(run_prefill_masked(w, m, causal))
    ref = oracle.masked(w, m, causal=causal)
    assert _err(got, ref) <= TOL
    r = int(w.qo_indptr[1]) + 2
    assert not got[r].any() and not got[int(w.qo_indptr[7]):].any()


def test_prefill_all_ones_mask_equals_unmasked_bitwise():
    w = workload.config(5)
    ones = np.ones((w.batch, w.max_q_len, -(-w.max_seq_len // 16) * 16), np.uint8)
    t = upload(w)
    plain = torch.empty_like(t["q"])
    pa.astr_attn_prefill_ragged(t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], plain, prefill_dims(w),
                                w.sm_scale)
    masked = run_prefill_masked(w, ones, causal=True)
    assert torch.equal(plain.view(torch.int16), masked.view(torch.int16))


def test_prefill_causal_pattern_as_mask_equals_causal():
    """A 3-D mask holding the causal pattern, causal off, against the causal call (tolerance:
    the two kernels differ only in which predicate hides the same keys)."""
    rng = np.random.default_rng(71)
    ql = np.array([7, 64, 65, 200])
    pre = np.array([0, 30, 1, 100])
    w = make_from_lengths(rng, kind="prefill", name="mask-causal", seq_lens=pre + ql, q_lens=ql, Hq=32, Hkv=8, d=128)
    kv = -(-w.max_seq_len // 16) * 16
    tri = np.zeros((w.batch, w.max_q_len, kv), np.uint8)
    for b in range(w.batch):
        for i in range(int(ql[b])):
            tri[b, i, :int(pre[b]) + i + 1] = 1
    got = to_f64(run_prefill_masked(w, tri, causal=False))
    assert _err(got, oracle.prefill(w)) <= TOL


@pytest.mark.parametrize("dims", [2, 3])
def test_decode_masked_config2(dims):
    w = workload.config(2)
    m = make_mask(w, dims, seed=80 + dims, keep=0.7)
    got = to_f64(run_decode_masked(w, m))
    assert _err(got, oracle.masked(w, m)) <= TOL


@pytest.mark.parametrize("num_splits", [1, 7, 64, 200])
def test_decode_masked_whole_chunks_and_requests_hidden(num_splits):
    """Masks that hide whole requests, whole 32-key slots and whole chunks (partials with no
    visible key), over forced chunk counts."""
    rng = np.random.default_rng(90 + num_splits)
    seq = np.array([1, 31, 32, 33, 40, 100, 257, 700, 1000, 5])
    w = make_from_lengths(rng, kind="decode", name="mask-decode", seq_lens=seq, q_lens=None, Hq=32, Hkv=8, d=128)
    m = make_mask(w, 2, seed=3, keep=0.5)
    m[2, :] = 0                  # a request with no visible key
    m[7, :600] = 0               # most of a long request (whole slots and chunks)
    m[8, 1:] = 0                 # only the first key of another
    m[4, :39] = 0                # only the last key (position 39: second 16-byte chunk of slot 1)
    got = to_f64(run_decode_masked(w, m, max_splits=64, num_splits=num_splits))
    assert _err(got, oracle.masked(w, m)) <= TOL
    assert not got[2].any()


@pytest.mark.parametrize("d,Hq,Hkv", [(64, 8, 2), (64, 16, 16), (128, 128, 8), (128, 16, 8)])
def test_decode_masked_head_shapes(d, Hq, Hkv):
    rng = np.random.default_rng(d + Hq + Hkv)
    seq = rng.integers(0, 300, size=12)
    w = make_from_lengths(rng, kind="decode", name="mask-decode-shapes", seq_lens=seq, q_lens=None, Hq=Hq, Hkv=Hkv,
                          d=d, stride=320)
    m = make_mask(w, 3, seed=5, keep=0.6)
    got = to_f64(run_decode_masked(w, m))
    assert _err(got, oracle.masked(w, m)) <= TOL


def test_decode_all_ones_mask_equals_unmasked_bitwise():
    w = workload.config(2)
    t = upload(w)
    dims = decode_dims(w)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    plain = torch.empty_like(t["q"])
    pa.astr_attn_paged_decode(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, plain, dims,
                              w.sm_scale)
    ones = np.ones((w.batch, -(-w.max_seq_len // 16) * 16), np.uint8)
    masked = run_decode_masked(w, ones)
    assert torch.equal(plain.view(torch.int16), masked.view(torch.int16))
