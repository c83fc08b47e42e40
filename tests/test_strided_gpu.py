"""Query and output tensors addressed by strides (astr_attn_decode_strided /
astr_attn_prefill_strided): packed rows with padded strides, and tensors padded per request in
"bhld" and "blhd" order, over the paged pool and over contiguous K/V caches, with masks.
Outputs are compared with the fp64 oracle (max abs error <= 1e-2); every element outside the
rows written is checked to be untouched."""
import numpy as np
import pytest

import oracle
from workload import make_from_lengths, make_mask

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import prefill_attention_gb300 as pa  # noqa: E402
from gpu_util import TOL, bf16_dev, decode_dims, prefill_dims, to_f64, upload  # noqa: E402
from test_contig_gpu import contiguous_cache  # noqa: E402

NAN = float("nan")


def _err(got, ref):
    return float(np.abs(got - ref).max())


def _rows_tensor(kind, B, L, H, d, pad):
    """A NaN-filled device tensor and its logical view: "packed" [B*L, H, d] rows whose head and
    row strides carry `pad` extra elements, "blhd" [B, L, H, d] or "bhld" [B, H, L, d] shown as
    [B, L, H, d]."""
    if kind == "packed":
        buf = torch.full((B * L, H, d + pad), NAN, dtype=torch.bfloat16, device="cuda")
        return buf, buf[:, :, :d]
    if kind == "blhd":
        buf = torch.full((B, L + 1, H, d + pad), NAN, dtype=torch.bfloat16, device="cuda")
        return buf, buf[:, :L, :, :d]
    buf = torch.full((B, H, L + 2, d + pad), NAN, dtype=torch.bfloat16, device="cuda")
    return buf, buf[:, :, :L, :d].transpose(1, 2)


def _fill_decode_q(view, q_bits, kind):
    q = bf16_dev(q_bits)                                    # [B, Hq, d]
    if kind == "packed":
        view.copy_(q)
    else:
        view[:, 0].copy_(q)


@pytest.mark.parametrize("q_kind,o_kind", [("packed", "packed"), ("bhld", "blhd"), ("blhd", "bhld"),
                                           ("packed", "bhld")])
@pytest.mark.parametrize("n_chunks", [0, 7])
def test_decode_strided_paged(q_kind, o_kind, n_chunks):
    rng = np.random.default_rng(900 + n_chunks)
    w = make_from_lengths(rng, kind="decode", name="strided", seq_lens=[1, 33, 700, 0, 129, 64], q_lens=None, Hq=16,
                          Hkv=4, d=128)
    t = upload(w)
    B, H, d = w.batch, w.num_qo_heads, w.head_dim
    qbuf, qv = _rows_tensor(q_kind, B, 1, H, d, 8)
    obuf, ov = _rows_tensor(o_kind, B, 1, H, d, 16)
    _fill_decode_q(qv, w.q, q_kind)
    dims = decode_dims(w, max_splits=32, num_splits=n_chunks)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    lay = pa.make_qo_layout(qv, ov, padded=q_kind != "packed")
    if (q_kind == "packed") != (o_kind == "packed"):  # mixed: build the layout from both halves
        ql = pa.make_qo_layout(qv, qv, padded=q_kind != "packed")
        ol = pa.make_qo_layout(ov, ov, padded=o_kind != "packed")
        lay = pa.QoLayout(ql.q_batch_stride, ql.q_token_stride, ql.q_head_stride, ol.o_batch_stride,
                          ol.o_token_stride, ol.o_head_stride)
    pa.astr_attn_decode_strided(qv, t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, ov, dims,
                                w.sm_scale, qo_layout=lay)
    torch.cuda.synchronize()
    got = to_f64(ov if o_kind == "packed" else ov[:, 0])
    assert _err(got, oracle.decode(w)) <= TOL
    written = torch.zeros_like(obuf, dtype=torch.bool)
    (written[:, :, :d] if o_kind == "packed" else
     (written[:, :1, :, :d] if o_kind == "blhd" else written[:, :, :1, :d]))[...] = True
    assert torch.isnan(obuf.float()[~written]).all(), "an element outside the outputs was written"


def test_decode_strided_contiguous_cache_and_mask():
    rng = np.random.default_rng(911)
    w = make_from_lengths(rng, kind="decode", name="strided-contig", seq_lens=[40, 300, 1, 129], q_lens=None, Hq=32,
                          Hkv=8, d=64)
    t = upload(w)
    kc, vc, _ = contiguous_cache(w, "bhld")
    m = make_mask(w, 2, seed=912, keep=0.6)
    B, H, d = w.batch, w.num_qo_heads, w.head_dim
    qbuf, qv = _rows_tensor("bhld", B, 1, H, d, 8)
    obuf, ov = _rows_tensor("blhd", B, 1, H, d, 8)
    _fill_decode_q(qv, w.q, "bhld")
    dims = decode_dims(w, max_splits=32, num_splits=5)
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    pa.astr_attn_decode_strided(qv, kc, vc, None, t["seq"], t["kvi"], o_part, ml_part, ov, dims, w.sm_scale,
                                kv_layout=pa.make_kv_layout(kc), qo_layout=pa.make_qo_layout(qv, ov, padded=True),
                                mask=pa.make_mask(torch.from_numpy(m).cuda()))
    torch.cuda.synchronize()
    assert _err(to_f64(ov[:, 0]), oracle.masked(w, m)) <= TOL


def _prefill_case(seed, Hq, Hkv, d):
    rng = np.random.default_rng(seed)
    ql = np.array([1, 5, 33, 64, 0, 129, 7])
    pre = np.array([0, 40, 3, 100, 9, 300, 0])
    return make_from_lengths(rng, kind="prefill", name="strided-pf", seq_lens=pre + ql, q_lens=ql, Hq=Hq, Hkv=Hkv,
                             d=d)


def _padded_rows(w, view):
    """Copy the packed query rows of w into a padded [B, L, Hq, d] view."""
    q = bf16_dev(w.q)
    for b in range(w.batch):
        q0, q1 = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        if q1 > q0:
            view[b, :q1 - q0].copy_(q[q0:q1])


def _gather_padded(w, view):
    rows = []
    for b in range(w.batch):
        n = int(w.q_lens[b])
        if n:
            rows.append(view[b, :n])
    return torch.cat(rows)


@pytest.mark.parametrize("q_kind,o_kind", [("packed", "packed"), ("bhld", "bhld"), ("blhd", "blhd"),
                                           ("bhld", "packed"), ("packed", "blhd")])
@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (64, 8, 2), (32, 16, 4)])
def test_prefill_strided_paged(q_kind, o_kind, d, Hq, Hkv):
    w = _prefill_case(920 + d + Hq, Hq, Hkv, d)
    t = upload(w)
    B, H, L = w.batch, w.num_qo_heads, w.max_q_len
    TQ = w.total_q
    if q_kind == "packed":
        qbuf, qv = _rows_tensor("packed", 1, TQ, H, d, 8)
        qv.copy_(bf16_dev(w.q))
    else:
        qbuf, qv = _rows_tensor(q_kind, B, L, H, d, 8)
        _padded_rows(w, qv)
    if o_kind == "packed":
        obuf, ov = _rows_tensor("packed", 1, TQ, H, d, 16)
    else:
        obuf, ov = _rows_tensor(o_kind, B, L, H, d, 16)
    ql = pa.make_qo_layout(qv, qv, padded=q_kind != "packed")
    ol = pa.make_qo_layout(ov, ov, padded=o_kind != "packed")
    lay = pa.QoLayout(ql.q_batch_stride, ql.q_token_stride, ql.q_head_stride, ol.o_batch_stride, ol.o_token_stride,
                      ol.o_head_stride)
    pa.astr_attn_prefill_strided(qv, t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], ov, prefill_dims(w),
                                 w.sm_scale, qo_layout=lay)
    torch.cuda.synchronize()
    got = to_f64(ov if o_kind == "packed" else _gather_padded(w, ov))
    assert _err(got, oracle.prefill(w)) <= TOL
    # rows past each request's q_len (padded outputs) and the padding columns are untouched
    n_written = TQ * H * d
    assert int((~torch.isnan(obuf.float())).sum()) == n_written


def test_prefill_strided_contiguous_cache_mask_and_causal_off():
    w = _prefill_case(931, 32, 8, 128)
    t = upload(w)
    kc, vc, _ = contiguous_cache(w, "blhd")
    m = make_mask(w, 3, seed=932, keep=0.7)
    B, H, d, L = w.batch, w.num_qo_heads, w.head_dim, w.max_q_len
    qbuf, qv = _rows_tensor("bhld", B, L, H, d, 8)
    _padded_rows(w, qv)
    obuf, ov = _rows_tensor("bhld", B, L, H, d, 8)
    dm = torch.from_numpy(m).cuda()
    for causal in (True, False):
        pa.astr_attn_prefill_strided(qv, t["qo"], kc, vc, None, t["seq"], t["kvi"], ov, prefill_dims(w), w.sm_scale,
                                     kv_layout=pa.make_kv_layout(kc), qo_layout=pa.make_qo_layout(qv, ov, True),
                                     mask=pa.make_mask(dm, causal))
        torch.cuda.synchronize()
        assert _err(to_f64(_gather_padded(w, ov)), oracle.masked(w, m, causal=causal)) <= TOL, f"causal={causal}"
