"""Prefill calls with a host work plan (dims.prefill_plan): the same items run, only their order
and CTA change, so every output bit equals the call without a plan; a plan that does not match
the call is ignored (ASTR_KSTATUS_PLAN) and the results stay right; a damaged row is reported."""
import numpy as np
import pytest

import oracle
import workload
from workload import make_mask

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import prefill_attention_gb300 as pa  # noqa: E402
from gpu_util import TOL, prefill_dims, to_f64, upload  # noqa: E402
from test_contig_gpu import contiguous_cache  # noqa: E402


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _run(w, t, dims, status=None, mask=None):
    dims.status = None if status is None else int(status.data_ptr())
    out = torch.full_like(t["q"], float("nan"))
    if mask is None:
        pa.astr_attn_prefill_ragged(t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], out, dims,
                                    w.sm_scale)
    else:
        pa.astr_attn_prefill_ragged_masked(t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], mask, out,
                                           dims, w.sm_scale)
    torch.cuda.synchronize()
    return out


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("cfg", ["extend", "g1", "g16-d64", "d32"])
def test_planned_call_is_bit_identical(cfg):
    w = {"extend": lambda: workload.config(5),
         "g1": lambda: workload.make_prefill(6, 8, 8, 128, (100, 700), (0, 2000), seed=61, name="g1"),
         "g16-d64": lambda: workload.make_prefill(9, 32, 2, 64, (1, 300), (0, 900), seed=62, name="g16"),
         "d32": lambda: workload.make_prefill(12, 16, 4, 32, (1, 200), (0, 400), seed=63, name="d32")}[cfg]()
    t = upload(w)
    ref = _run(w, t, prefill_dims(w))
    dims = prefill_dims(w)
    plan = pa.make_prefill_plan(w.qo_indptr, w.seq_lens, dims)
    assert plan is not None
    st = _status()
    got = _run(w, t, pa.attach_prefill_plan(dims, plan), st)
    assert int(st.item()) == 0
    assert np.array_equal(_bits(got), _bits(ref))
    assert np.abs(to_f64(got) - oracle.prefill(w)).max() <= TOL


def test_planned_masked_and_causal_off():
    w = workload.make_prefill(7, 32, 8, 128, (1, 150), (0, 300), seed=64, name="plan-mask")
    t = upload(w)
    m = torch.from_numpy(make_mask(w, 3, seed=65, keep=0.7)).cuda()
    for causal in (True, False):
        mask = pa.make_mask(m, causal)
        ref = _run(w, t, prefill_dims(w), mask=mask)
        dims = prefill_dims(w)
        plan = pa.make_prefill_plan(w.qo_indptr, w.seq_lens, dims, causal=causal)
        st = _status()
        got = _run(w, t, pa.attach_prefill_plan(dims, plan), st, mask=mask)
        assert int(st.item()) == 0, f"causal={causal}"
        assert np.array_equal(_bits(got), _bits(ref)), f"causal={causal}"


def test_planned_contiguous_cache():
    w = workload.make_prefill(5, 32, 8, 128, (1, 200), (0, 500), seed=66, name="plan-contig")
    t = upload(w)
    kc, vc, _ = contiguous_cache(w, "blhd")
    lay = pa.make_kv_layout(kc)

    def run(dims, st=None):
        dims.status = None if st is None else int(st.data_ptr())
        out = torch.full_like(t["q"], float("nan"))
        pa.astr_attn_prefill_contiguous(t["q"], t["qo"], kc, vc, lay, t["seq"], t["kvi"], out, dims, w.sm_scale)
        torch.cuda.synchronize()
        return out

    ref = run(prefill_dims(w))
    dims = prefill_dims(w)
    st = _status()
    got = run(pa.attach_prefill_plan(dims, pa.make_prefill_plan(w.qo_indptr, w.seq_lens, dims)), st)
    assert int(st.item()) == 0
    assert np.array_equal(_bits(got), _bits(ref))


def test_plan_for_other_inputs_is_ignored_and_reported():
    w = workload.config(5)
    t = upload(w)
    ref = _run(w, t, prefill_dims(w))
    # made for other key counts (a stale plan of another batch)
    other = w.seq_lens.copy()
    other[0] += 1
    dims = prefill_dims(w)
    stale = pa.make_prefill_plan(w.qo_indptr, other, dims)
    # made for another grid, another causal flag
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    few = torch.from_numpy(pa.astr_attn_prefill_plan(w.qo_indptr, w.seq_lens, dims, num_ctas=sms - 8)).cuda()
    acausal = pa.make_prefill_plan(w.qo_indptr, w.seq_lens, dims, causal=False)
    for name, plan in (("stale", stale), ("grid", few), ("causal", acausal)):
        st = _status()
        got = _run(w, t, pa.attach_prefill_plan(prefill_dims(w), plan), st)
        assert int(st.item()) == pa.ASTR_KSTATUS_PLAN, name
        assert np.array_equal(_bits(got), _bits(ref)), name
    # a plan buffer shorter than the launch's rows is not read at all
    good = pa.make_prefill_plan(w.qo_indptr, w.seq_lens, dims)
    d2 = pa.attach_prefill_plan(prefill_dims(w), good)
    d2.prefill_plan_words = good.numel() - 1
    st = _status()
    got = _run(w, t, d2, st)
    assert int(st.item()) == pa.ASTR_KSTATUS_PLAN
    assert np.array_equal(_bits(got), _bits(ref))


def test_damaged_plan_row_is_reported():
    """A row entry that names no item of the call (the header and checksum still match) is
    dropped and reported; nothing outside the buffers is touched."""
    w = workload.config(5)
    t = upload(w)
    dims = prefill_dims(w)
    plan = pa.astr_attn_prefill_plan(w.qo_indptr, w.seq_lens, dims)
    row0 = 8
    assert plan[row0] >= 1
    plan[row0 + 1] = w.batch + 5  # request index past the batch
    st = _status()
    _run(w, t, pa.attach_prefill_plan(dims, torch.from_numpy(plan).cuda()), st)
    assert int(st.item()) == pa.ASTR_KSTATUS_BAD_INPUT


def test_planned_strided_padded_query_and_output():
    """A plan serves the strided entry point too: padded "bhld" query and "blhd" output."""
    w = workload.make_prefill(6, 32, 8, 128, (1, 130), (0, 400), seed=67, name="plan-strided")
    t = upload(w)
    B, H, d, L = w.batch, w.num_qo_heads, w.head_dim, w.max_q_len
    q = torch.zeros(B, H, L, d, dtype=torch.bfloat16, device="cuda")
    qv = q.transpose(1, 2)
    for b in range(B):
        q0, q1 = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        qv[b, :q1 - q0].copy_(t["q"][q0:q1])
    def run(dims):
        o = torch.full((B, L, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        pa.astr_attn_prefill_strided(qv, t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o, dims, w.sm_scale,
                                     qo_layout=pa.make_qo_layout(qv, o, padded=True))
        torch.cuda.synchronize()
        return o

    ref = run(prefill_dims(w))
    dims = prefill_dims(w)
    st = _status()
    dims.status = int(st.data_ptr())
    got = run(pa.attach_prefill_plan(dims, pa.make_prefill_plan(w.qo_indptr, w.seq_lens, dims)))
    assert int(st.item()) == 0
    assert np.array_equal(_bits(got), _bits(ref))


def test_planned_call_in_a_cuda_graph():
    """The plan and every argument stay fixed for a batch, so planned calls capture and replay."""
    w = workload.config(5)
    t = upload(w)
    dims = prefill_dims(w)
    plan = pa.make_prefill_plan(w.qo_indptr, w.seq_lens, dims)
    pa.attach_prefill_plan(dims, plan)
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
