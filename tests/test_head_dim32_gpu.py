"""Head dim 32 (the size the pages' head-dim dispatch adds; 64-byte rows, 64-byte swizzle in
the prefill operand tiles) through decode, prefill, masks and contiguous caches, against the
fp64 oracle (max abs error <= 1e-2)."""
import numpy as np
import pytest

import oracle
from workload import make_from_lengths, make_mask

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import prefill_attention_gb300 as pa  # noqa: E402
from gpu_util import TOL, decode_dims, prefill_dims, run_decode, run_prefill, to_f64, upload  # noqa: E402
from test_contig_gpu import run_decode_contig, run_prefill_contig  # noqa: E402

SHAPES = [(8, 8), (16, 8), (32, 8), (64, 8), (128, 8), (8, 2)]   # (Hq, Hkv): G = 1, 2, 4, 8, 16, 4


def _err(got, ref):
    return float(np.abs(got - ref).max())


@pytest.mark.parametrize("Hq,Hkv", SHAPES)
def test_decode_head_dim_32_ragged(Hq, Hkv):
    rng = np.random.default_rng(3200 + Hq + Hkv)
    seq = [1, 7, 8, 9, 31, 33, 64, 65, 127, 128, 129, 200, 257, 0, 600, 2000]
    w = make_from_lengths(rng, kind="decode", name="d32", seq_lens=seq, q_lens=None, Hq=Hq, Hkv=Hkv, d=32)
    ref = oracle.decode(w)
    for n in (0, 1, 5, 37):
        assert _err(to_f64(run_decode(w, num_splits=n)), ref) <= TOL, f"n_chunks={n}"


def test_decode_head_dim_32_pages_shaped():
    """B=32, GQA 32/8, seq 200-2000 at d=32 (the decode microbench shape with the small head)."""
    rng = np.random.default_rng(3232)
    seq = rng.integers(200, 2001, 32)
    w = make_from_lengths(rng, kind="decode", name="d32-b32", seq_lens=seq, q_lens=None, Hq=32, Hkv=8, d=32)
    assert _err(to_f64(run_decode(w)), oracle.decode(w)) <= TOL


@pytest.mark.parametrize("Hq,Hkv", SHAPES)
def test_prefill_head_dim_32_ragged(Hq, Hkv):
    rng = np.random.default_rng(3300 + Hq + Hkv)
    ql = np.array([1, 5, 31, 32, 33, 64, 100, 129, 300])
    pre = np.array([0, 3, 0, 64, 17, 190, 1, 300, 700])
    w = make_from_lengths(rng, kind="prefill", name="d32-pf", seq_lens=pre + ql, q_lens=ql, Hq=Hq, Hkv=Hkv, d=32)
    assert _err(to_f64(run_prefill(w)), oracle.prefill(w)) <= TOL


def test_prefill_head_dim_32_empty_requests_and_padding_rows():
    """q_len 0 requests write nothing; rows of partial query tiles are never stored."""
    rng = np.random.default_rng(3311)
    ql = np.array([0, 3, 0, 40, 1])
    pre = np.array([5, 0, 9, 10, 0])
    w = make_from_lengths(rng, kind="prefill", name="d32-empty", seq_lens=pre + ql, q_lens=ql, Hq=16, Hkv=4, d=32)
    t = upload(w)
    pad = 64
    buf = torch.full((w.total_q * w.num_qo_heads * 32 + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[pad:pad + w.total_q * w.num_qo_heads * 32].view(w.total_q, w.num_qo_heads, 32)
    pa.astr_attn_prefill_ragged(t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"], out, prefill_dims(w),
                                w.sm_scale)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 7.0) and torch.all(buf[-pad:] == 7.0)
    assert _err(to_f64(out), oracle.prefill(w)) <= TOL


@pytest.mark.parametrize("dims", [2, 3])
def test_masked_head_dim_32(dims):
    rng = np.random.default_rng(3400 + dims)
    ql = np.array([1, 17, 64, 5])
    pre = np.array([30, 0, 100, 7])
    w = make_from_lengths(rng, kind="prefill", name="d32-mask", seq_lens=pre + ql, q_lens=ql, Hq=32, Hkv=8, d=32)
    m = make_mask(w, dims, seed=3401, keep=0.6)
    t = upload(w)
    dm = torch.from_numpy(m).cuda()
    for causal in (True, False):
        out = torch.empty_like(t["q"])
        pa.astr_attn_prefill_ragged_masked(t["q"], t["qo"], t["k"], t["v"], t["r2t"], t["seq"], t["kvi"],
                                           pa.make_mask(dm, causal), out, prefill_dims(w), w.sm_scale)
        torch.cuda.synchronize()
        assert _err(to_f64(out), oracle.masked(w, m, causal=causal)) <= TOL, f"causal={causal}"
    wd = make_from_lengths(rng, kind="decode", name="d32-mask-dec", seq_lens=[40, 300, 1, 129], q_lens=None, Hq=32,
                           Hkv=8, d=32)
    md = make_mask(wd, dims, seed=3402, keep=0.6)
    td = upload(wd)
    ddims = decode_dims(wd, max_splits=32, num_splits=9)
    o_part, ml_part = pa.alloc_decode_workspace(ddims)
    out = torch.empty_like(td["q"])
    pa.astr_attn_paged_decode_masked(td["q"], td["k"], td["v"], td["r2t"], td["seq"], td["kvi"],
                                     pa.make_mask(torch.from_numpy(md).cuda()), o_part, ml_part, out, ddims,
                                     wd.sm_scale)
    torch.cuda.synchronize()
    assert _err(to_f64(out), oracle.masked(wd, md)) <= TOL


@pytest.mark.parametrize("layout", ["blhd", "bhld"])
def test_contiguous_head_dim_32(layout):
    rng = np.random.default_rng(3500)
    wd = make_from_lengths(rng, kind="decode", name="d32-contig", seq_lens=[1, 33, 600, 0, 64], q_lens=None, Hq=16,
                           Hkv=4, d=32)
    assert _err(to_f64(run_decode_contig(wd, layout, num_splits=7)), oracle.decode(wd)) <= TOL
    ql = np.array([4, 64, 1])
    pre = np.array([0, 33, 200])
    wp = make_from_lengths(rng, kind="prefill", name="d32-contig-pf", seq_lens=pre + ql, q_lens=ql, Hq=16, Hkv=4,
                           d=32)
    assert _err(to_f64(run_prefill_contig(wp, layout)), oracle.prefill(wp)) <= TOL
