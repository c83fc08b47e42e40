"""dims.flags = ASTR_DIMS_STABLE_INDICES: the decode split step plans its chunks from the index
arrays before its dependency wait.  The same chunks come out, so every output bit equals the
call without the flag -- for the paged, masked, contiguous-cache and strided entry points, the
two-launch form and a CUDA-graph replay -- and the results match the fp64 oracle."""
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
from gpu_util import TOL, decode_dims, to_f64, upload  # noqa: E402
from test_contig_gpu import contiguous_cache  # noqa: E402

FLAG = pa.ASTR_DIMS_STABLE_INDICES


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def _paged(w, t, flags, num_splits=0, max_splits=32):
    dims = decode_dims(w, max_splits=max_splits, num_splits=num_splits)
    dims.flags = flags
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.full_like(t["q"], float("nan"))
    pa.astr_attn_paged_decode(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, out, dims,
                              w.sm_scale)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_configs_bit_identical_with_the_flag(cfg):
    w = workload.config(cfg)
    t = upload(w)
    ref = _paged(w, t, 0)
    for _ in range(2):  # back to back: the second call's planning overlaps the first's tail
        got = _paged(w, t, FLAG)
        assert np.array_equal(_bits(got), _bits(ref))
    assert np.abs(to_f64(got) - oracle.decode(w)).max() <= TOL


@pytest.mark.parametrize("n", [1, 5, 37])
def test_ragged_split_counts(n):
    rng = np.random.default_rng(1500 + n)
    w = make_from_lengths(rng, kind="decode", name="stable", seq_lens=[1, 33, 700, 0, 129, 64, 2000, 31], q_lens=None,
                          Hq=16, Hkv=4, d=64)
    t = upload(w)
    assert np.array_equal(_bits(_paged(w, t, FLAG, num_splits=n)), _bits(_paged(w, t, 0, num_splits=n)))


def test_split_then_combine_and_graph_replay():
    w = workload.config(2)
    t = upload(w)
    ref = _paged(w, t, 0)
    dims = decode_dims(w)
    dims.flags = FLAG
    o_part, ml_part = pa.alloc_decode_workspace(dims)
    out = torch.empty_like(t["q"])
    pa.astr_attn_decode_split(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, dims, w.sm_scale)
    pa.astr_attn_decode_combine(o_part, ml_part, t["seq"], t["kvi"], out, dims)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), _bits(ref))
    s = torch.cuda.Stream()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            pa.astr_attn_paged_decode(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, out,
                                      dims, w.sm_scale, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), _bits(ref))


def test_masked_contiguous_and_strided_forms():
    rng = np.random.default_rng(1510)
    w = make_from_lengths(rng, kind="decode", name="stable-forms", seq_lens=[40, 300, 1, 129, 900], q_lens=None,
                          Hq=32, Hkv=8, d=128)
    t = upload(w)
    m = pa.make_mask(torch.from_numpy(make_mask(w, 2, seed=1511, keep=0.6)).cuda())
    kc, vc, _ = contiguous_cache(w, "bhld")
    lay = pa.make_kv_layout(kc)

    def run(flags, form):
        dims = decode_dims(w, max_splits=32, num_splits=9)
        dims.flags = flags
        o_part, ml_part = pa.alloc_decode_workspace(dims)
        out = torch.full_like(t["q"], float("nan"))
        if form == "masked":
            pa.astr_attn_paged_decode_masked(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], m, o_part,
                                             ml_part, out, dims, w.sm_scale)
        elif form == "contig":
            pa.astr_attn_decode_contiguous(t["q"], kc, vc, lay, t["seq"], t["kvi"], o_part, ml_part, out, dims,
                                           w.sm_scale)
        else:
            pa.astr_attn_decode_strided(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], o_part, ml_part, out,
                                        dims, w.sm_scale, qo_layout=pa.make_qo_layout(t["q"], out, padded=False))
        torch.cuda.synchronize()
        return out

    for form in ("masked", "contig", "strided"):
        assert np.array_equal(_bits(run(FLAG, form)), _bits(run(0, form))), form
