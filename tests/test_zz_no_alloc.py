"""The allocation-free decode entry point, checked against the workspace entry point.

astr_attn_paged_decode_noalloc serves callers that cannot hand the library a workspace
(an operator inside a runtime whose memory planner owns all device memory, or a process
that must not grow device memory after start-up): its split partials live in a fixed
array compiled into the library.  This file runs last so that a failure here does not hide
the other GPU tests, and it passes both alone in a fresh process and after them.
"""
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
from gpu_util import TOL, decode_dims, run_decode, to_f64, upload  # noqa: E402


@pytest.mark.parametrize("cfg", [1, 2])
def test_noalloc_matches_workspace_entry_point_twice(cfg):
    w = workload.config(cfg)
    t = upload(w)
    max_splits = 8
    ref = to_f64(run_decode(w, t, max_splits=max_splits))  # the workspace entry point
    dims = decode_dims(w, max_splits=max_splits)
    for call in range(2):  # the second call reuses the array the first one left behind
        out = torch.full_like(t["q"], float("nan"))
        pa.astr_attn_paged_decode_noalloc(t["q"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], out, dims,
                                          w.sm_scale)
        torch.cuda.synchronize()
        got = to_f64(out)
        assert np.isfinite(got).all(), f"call {call}"
        assert np.abs(got - ref).max() <= TOL, f"call {call}: differs from the workspace entry point"
        assert np.abs(got - oracle.decode(w)).max() <= TOL, f"call {call}: differs from the oracle"


def test_partials_left_by_a_larger_call_are_never_read():
    """A large call fills much of the shared array; smaller calls with other split layouts
    (requests inside one chunk next to requests over several) must read only the partials
    they wrote themselves, whatever the array held before."""
    big = workload.config(2)
    tb = upload(big)
    out_b = torch.empty_like(tb["q"])
    pa.astr_attn_paged_decode_noalloc(tb["q"], tb["k"], tb["v"], tb["r2t"], tb["seq"], tb["kvi"], out_b,
                                      decode_dims(big, max_splits=16), big.sm_scale)
    rng = np.random.default_rng(4242)
    small = make_from_lengths(rng, kind="decode", name="after-big", seq_lens=[3, 200, 31, 33, 500, 1, 64, 0],
                              q_lens=None, Hq=8, Hkv=2, d=64)
    ts = upload(small)
    ref_small = oracle.decode(small)
    for n_chunks in (0, 5, 37, 3):
        dims = decode_dims(small, max_splits=8, num_splits=n_chunks)
        out = torch.full_like(ts["q"], float("nan"))
        pa.astr_attn_paged_decode_noalloc(ts["q"], ts["k"], ts["v"], ts["r2t"], ts["seq"], ts["kvi"], out, dims,
                                          small.sm_scale)
        torch.cuda.synchronize()
        got = to_f64(out)
        ref = to_f64(run_decode(small, ts, max_splits=8, num_splits=n_chunks))
        assert np.isfinite(got).all(), f"n_chunks={n_chunks}"
        assert np.abs(got - ref).max() <= TOL, f"n_chunks={n_chunks}: differs from the workspace entry point"
        assert np.abs(got - ref_small).max() <= TOL, f"n_chunks={n_chunks}: differs from the oracle"
    assert np.abs(to_f64(out_b) - oracle.decode(big)).max() <= TOL
