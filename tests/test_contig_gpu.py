"""GPU parity of decode and prefill over a contiguous (stride-addressed) K/V cache: "blhd" and
"bhld" layouts, padded strides, with and without explicit masks, through the C ABI."""
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
from gpu_util import TOL, bf16_dev, decode_dims, i32_dev, prefill_dims, to_f64, upload  # noqa: E402

NAN_BF16 = np.uint16(0x7FC0)


def contiguous_cache(w, layout, pad_token=0, pad_batch=0):
    """The workload's K/V rows laid out contiguously by request position (positions past a
    request's keys hold NaN, so a read of them would show).  Returns device tensors K, V with
    logical dims [B, L, Hkv, d] (a view for "bhld") and L."""
    B, Hkv, d = w.batch, w.num_kv_heads, w.head_dim
    L = w.max_seq_len
    k = np.full((B, L, Hkv, d), NAN_BF16, np.uint16)
    v = np.full((B, L, Hkv, d), NAN_BF16, np.uint16)
    for b in range(B):
        n = int(w.seq_lens[b])
        slots = w.req_to_token[b, :n].astype(np.int64)
        k[b, :n] = w.k_pool[slots]
        v[b, :n] = w.v_pool[slots]
    out = []
    for a in (k, v):
        if layout == "blhd":
            buf = np.full((B, L + pad_batch, Hkv, d + pad_token), NAN_BF16, np.uint16)
            buf[:, :L, :, :d] = a
            t = bf16_dev(buf)[:, :L, :, :d]
        else:  # bhld
            buf = np.full((B, Hkv, L + pad_batch, d + pad_token), NAN_BF16, np.uint16)
            buf[:, :, :L, :d] = a.transpose(0, 2, 1, 3)
            t = bf16_dev(buf)[:, :, :L, :d].transpose(1, 2)
        out.append(t)
    return out[0], out[1], L


def run_decode_contig(w, layout, mask=None, pad_token=0, pad_batch=0, num_splits=0):
    t = upload(w)
    kc, vc, L = contiguous_cache(w, layout, pad_token, pad_batch)
    dims = decode_dims(w, max_splits=32, num_splits=num_splits)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.full_like(t["q"], float("nan"))
    dm = None if mask is None else torch.from_numpy(mask).cuda()
    pa.astr_attn_decode_contiguous(t["q"], kc, vc, pa.make_kv_layout(kc), t["seq"], t["kvi"], o_part, ml_part, out,
                                   dims, w.sm_scale, mask=None if dm is None else pa.make_mask(dm))
    torch.cuda.synchronize()
    return out


def run_prefill_contig(w, layout, mask=None, causal=True, pad_token=0, pad_batch=0):
    t = upload(w)
    kc, vc, L = contiguous_cache(w, layout, pad_token, pad_batch)
    out = torch.full_like(t["q"], float("nan"))
    dm = None if mask is None else torch.from_numpy(mask).cuda()
    m = None if (dm is None and causal) else pa.make_mask(dm, causal)
    pa.astr_attn_prefill_contiguous(t["q"], t["qo"], kc, vc, pa.make_kv_layout(kc), t["seq"], t["kvi"], out,
                                    prefill_dims(w), w.sm_scale, mask=m)
    torch.cuda.synchronize()
    return out


def _err(got, ref):
    return float(np.abs(got - ref).max())


@pytest.mark.parametrize("layout,pad_token,pad_batch", [("blhd", 0, 0), ("bhld", 0, 0), ("blhd", 8, 3),
                                                        ("bhld", 16, 5)])
def test_decode_contiguous_equals_paged_bitwise(layout, pad_token, pad_batch):
    """Same keys in the same order: the contiguous kernel's output is bit-identical to the
    paged kernel's, and within tolerance of the oracle."""
    w = workload.config(2)
    got = run_decode_contig(w, layout, pad_token=pad_token, pad_batch=pad_batch)
    t = upload(w)
    dims = decode_dims(w)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    paged = torch.empty_like(t["q"])
    pa.astr_attn_paged_decode(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, paged, dims,
                              w.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), paged.view(torch.int16))
    assert _err(to_f64(got), oracle.decode(w)) <= TOL


@pytest.mark.parametrize("d,Hq,Hkv", [(64, 8, 2), (64, 16, 16), (128, 128, 8), (128, 16, 8)])
@pytest.mark.parametrize("layout", ["blhd", "bhld"])
def test_decode_contiguous_shapes_and_ragged(d, Hq, Hkv, layout):
    rng = np.random.default_rng(d + Hq + Hkv)
    seq = np.array([0, 1, 31, 32, 33, 100, 257, 300])
    w = make_from_lengths(rng, kind="decode", name="contig-decode", seq_lens=seq, q_lens=None, Hq=Hq, Hkv=Hkv, d=d)
    got = to_f64(run_decode_contig(w, layout, num_splits=20))
    assert _err(got, oracle.decode(w)) <= TOL
    assert not got[0].any()


@pytest.mark.parametrize("dims", [2, 3])
def test_decode_contiguous_masked(dims):
    w = workload.config(2)
    m = make_mask(w, dims, seed=11 + dims, keep=0.6)
    m[3] = 0
    got = to_f64(run_decode_contig(w, "bhld", mask=m))
    assert _err(got, oracle.masked(w, m)) <= TOL


@pytest.mark.parametrize("layout,pad_token,pad_batch", [("blhd", 0, 0), ("bhld", 0, 0), ("bhld", 8, 7)])
def test_prefill_contiguous_extend_workload(layout, pad_token, pad_batch):
    w = workload.config(5)
    got = to_f64(run_prefill_contig(w, layout, pad_token=pad_token, pad_batch=pad_batch))
    assert _err(got, oracle.prefill(w)) <= TOL


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (128, 16, 16), (64, 32, 2), (64, 64, 4)])
@pytest.mark.parametrize("layout", ["blhd", "bhld"])
def test_prefill_contiguous_shapes_and_ragged(d, Hq, Hkv, layout):
    rng = np.random.default_rng(d * 5 + Hq + Hkv)
    ql = np.array([1, 5, 31, 33, 64, 100, 129, 0])
    pre = np.array([0, 3, 0, 64, 17, 190, 1, 9])
    w = make_from_lengths(rng, kind="prefill", name="contig-prefill", seq_lens=pre + ql, q_lens=ql, Hq=Hq, Hkv=Hkv,
                          d=d)
    got = to_f64(run_prefill_contig(w, layout))
    assert _err(got, oracle.prefill(w)) <= TOL


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_contiguous_masked_and_noncausal(causal):
    rng = np.random.default_rng(31)
    ql = np.array([7, 64, 65, 200, 1])
    pre = np.array([0, 30, 1, 100, 40])
    w = make_from_lengths(rng, kind="prefill", name="contig-mask", seq_lens=pre + ql, q_lens=ql, Hq=32, Hkv=8, d=128)
    m = make_mask(w, 3, seed=2, keep=0.7)
    got = to_f64(run_prefill_contig(w, "bhld", mask=m, causal=causal))
    assert _err(got, oracle.masked(w, m, causal=causal)) <= TOL
    got = to_f64(run_prefill_contig(w, "blhd", mask=None, causal=causal))
    ones = np.ones((w.batch, -(-w.max_seq_len // 16) * 16), np.uint8)
    assert _err(got, oracle.masked(w, ones, causal=causal)) <= TOL
