"""Host-side checks of the prefill work plan (astr_attn_prefill_plan): every work item of the
call exactly once, rows within the per-CTA limit, the header the kernel checks, the
longest-first balance bound, and the documented errors.  No GPU: the CTA count is given."""
import numpy as np
import pytest

import prefill_attention_gb300 as pa
from prefill_attention_gb300 import build as pbuild
import workload

HEADER, ROW, MAX_ITEMS = 8, 257, 128


@pytest.fixture(scope="module", autouse=True)
def lib():
    pbuild.build()
    return pa.load()


def _dims(qo, sl, Hq, Hkv, d=128, max_q_len=None):
    q_lens = np.diff(qo)
    return pa.make_dims(len(sl), Hq, Hkv, d, 1 << 20, max(int(sl.max()), 1), max(int(sl.max()), 1),
                        total_q=int(qo[-1]), max_q_len=int(q_lens.max()) if max_q_len is None else max_q_len)


def _items(qo, sl, G, H, causal=True):
    """(b, pair, kvh) -> the planner's cost estimate (about 10 ns units)."""
    bq2, bq, bn = 256 // G, 128 // G, 64
    out = {}
    for b in range(len(sl)):
        q_len, kvn = int(qo[b + 1] - qo[b]), int(sl[b])
        cb = kvn - q_len if causal else kvn - 1
        for pr in range((q_len + bq2 - 1) // bq2):
            first0 = pr * bq2
            nq = min(2, (q_len - first0 + bq - 1) // bq)
            last = min(q_len, first0 + nq * bq) - 1
            n_tiles = (min(cb + last + 1, kvn) + bn - 1) // bn
            units = sum((min(cb + min(q_len, first0 + (t + 1) * bq), kvn) + bn - 1) // bn for t in range(nq))
            cost = 53 * n_tiles + 13 * units + 260
            for h in range(H):
                out[(b, pr, h)] = cost
    return out


def _grid(dims, ctas):
    G = dims.num_qo_heads // dims.num_kv_heads
    bq = 256 // G
    tiles = min((dims.total_q + bq - 1) // bq + dims.batch, dims.batch * ((dims.max_q_len + bq - 1) // bq))
    return min(tiles * dims.num_kv_heads, ctas)


def _rows(plan, grid):
    rows = []
    for c in range(grid):
        r = plan[HEADER + c * ROW: HEADER + (c + 1) * ROW]
        n = int(r[0])
        assert 0 <= n <= MAX_ITEMS
        rows.append([(int(r[1 + 2 * k]), int(r[2 + 2 * k]) >> 16, int(r[2 + 2 * k]) & 0xFFFF) for k in range(n)])
        assert not r[1 + 2 * n:].any(), "unused row words are zero"
    return rows


def _mix(i, v):
    m = 0xFFFFFFFF
    h = (v * 0x9E3779B1 + i * 0x85EBCA77 + 0x165667B1) & m
    h ^= h >> 15
    h = (h * 0x2C1B3C6D) & m
    h ^= h >> 12
    h = (h * 0x297A2D39) & m
    h ^= h >> 15
    return h


def _checksum(qo, sl):
    h = sum(_mix(i, int(v) & 0xFFFFFFFF) for i, v in enumerate(qo))
    h += sum(_mix(0x40000000 + i, int(v) & 0xFFFFFFFF) for i, v in enumerate(sl))
    h &= 0xFFFFFFFF
    return h - (1 << 32) if h >= (1 << 31) else h


CASES = [
    ("extend", lambda: workload.config(5), 152),
    ("extend-100-ctas", lambda: workload.config(5), 100),
    ("few-items", lambda: workload.make_prefill(3, 8, 2, 64, (1, 40), (0, 30), seed=5, name="few"), 152),
    ("g1-long", lambda: workload.make_prefill(6, 8, 8, 128, (100, 900), (0, 3000), seed=6, name="g1"), 148),
    ("g16", lambda: workload.make_prefill(9, 32, 2, 64, (1, 300), (0, 900), seed=7, name="g16"), 152),
]


@pytest.mark.parametrize("name,make,ctas", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("causal", [True, False])
def test_plan_covers_every_item_once_and_balances(name, make, ctas, causal):
    w = make()
    qo, sl = w.qo_indptr.astype(np.int32), w.seq_lens.astype(np.int32)
    dims = _dims(qo, sl, w.num_qo_heads, w.num_kv_heads, w.head_dim)
    plan = pa.astr_attn_prefill_plan(qo, sl, dims, causal=causal, num_ctas=ctas)
    G = w.num_qo_heads // w.num_kv_heads
    grid = _grid(dims, ctas)
    assert plan.shape == (HEADER + grid * ROW,)
    assert list(plan[:6]) == [0x41535450, 1, w.batch, w.num_kv_heads, 256 // G, grid]
    assert plan[6] == _checksum(qo, sl) and plan[7] == int(causal)
    rows = _rows(plan, grid)
    items = _items(qo, sl, G, w.num_kv_heads, causal)
    dealt = [it for r in rows for it in r]
    assert len(dealt) == len(set(dealt)) == len(items) and set(dealt) == set(items)
    # longest first: the most-loaded CTA exceeds the least-loaded by at most one item's cost,
    # and every row lists its items in non-increasing cost order
    loads = [sum(items[it] for it in r) for r in rows]
    assert max(loads) - min(loads) <= max(items.values())
    for r in rows:
        costs = [items[it] for it in r]
        assert costs == sorted(costs, reverse=True)


def test_plan_is_deterministic_and_size_query_matches():
    w = workload.config(5)
    qo, sl = w.qo_indptr.astype(np.int32), w.seq_lens.astype(np.int32)
    dims = _dims(qo, sl, w.num_qo_heads, w.num_kv_heads)
    a = pa.astr_attn_prefill_plan(qo, sl, dims, num_ctas=152)
    b = pa.astr_attn_prefill_plan(qo, sl, dims, num_ctas=152)
    assert np.array_equal(a, b)
    import ctypes
    need = ctypes.c_size_t(0)
    st = pa.load().astr_attn_prefill_plan(qo.ctypes.data, sl.ctypes.data, ctypes.byref(dims), 1, 152, 0, None, 0,
                                          ctypes.byref(need))
    assert st == pa.ASTR_OK and need.value == a.size
    small = np.zeros(a.size - 1, np.int32)
    st = pa.load().astr_attn_prefill_plan(qo.ctypes.data, sl.ctypes.data, ctypes.byref(dims), 1, 152, 0,
                                          small.ctypes.data, small.size, ctypes.byref(need))
    assert st == pa.ASTR_ERR_INVALID_ARG


def test_plan_errors():
    w = workload.config(5)
    qo, sl = w.qo_indptr.astype(np.int32), w.seq_lens.astype(np.int32)
    dims = _dims(qo, sl, w.num_qo_heads, w.num_kv_heads)
    bad = sl.copy()
    bad[3] = int(qo[4] - qo[3]) - 1  # fewer keys than new queries: not a causal extend
    with pytest.raises(pa.AstrAttnError):
        pa.astr_attn_prefill_plan(qo, bad, dims, num_ctas=152)
    assert pa.astr_attn_prefill_plan(qo, bad, dims, causal=False, num_ctas=152) is not None
    # more requests than the kernel's shared tables hold: no plan applies
    B = 1100
    qo2 = np.arange(B + 1, dtype=np.int32)
    sl2 = np.full(B, 5, np.int32)
    assert pa.astr_attn_prefill_plan(qo2, sl2, _dims(qo2, sl2, 8, 2, 64), num_ctas=152) is None
    # more than 128 items on a CTA (natural order in the kernel): no plan
    B = 600
    qo3 = np.concatenate([[0], np.cumsum(np.full(B, 270))]).astype(np.int32)
    sl3 = np.full(B, 290, np.int32)
    assert pa.astr_attn_prefill_plan(qo3, sl3, _dims(qo3, sl3, 32, 32, 64), num_ctas=40) is None
    with pytest.raises(ValueError):
        pa.astr_attn_prefill_plan(qo[:-1], sl, dims, num_ctas=152)


def test_plan_edge_shapes():
    """Requests with no query rows contribute no items; one KV head; a grid larger than the
    items (one item per CTA at most); every row is listed longest first."""
    qo = np.array([0, 0, 5, 5, 300, 300], np.int32)      # requests 0, 2 and 4 have q_len 0
    sl = np.array([7, 40, 9, 1000, 300], np.int32)
    for Hq, Hkv in ((8, 1), (16, 16)):
        dims = _dims(qo, sl, Hq, Hkv)
        plan = pa.astr_attn_prefill_plan(qo, sl, dims, num_ctas=4096)
        G = Hq // Hkv
        items = _items(qo, sl, G, Hkv)
        grid = _grid(dims, 4096)
        assert int(plan[5]) == grid
        rows = _rows(plan, grid)
        dealt = [it for r in rows for it in r]
        assert sorted(dealt) == sorted(items)
        assert all(b in (1, 3) for b, _, _ in dealt), "only requests with query rows"
        assert max(len(r) for r in rows) <= 1 or grid < len(items)


def test_plan_without_causal_offset_allows_more_queries_than_keys():
    """With the causal rule off (explicit-mask calls), q_len may exceed seq_len; every key is
    visible to every row, so an item's KV tiles cover the whole key range."""
    qo = np.array([0, 100, 164], np.int32)
    sl = np.array([30, 64], np.int32)
    dims = _dims(qo, sl, 32, 8, max_q_len=100)
    with pytest.raises(pa.AstrAttnError):
        pa.astr_attn_prefill_plan(qo, sl, dims, causal=True, num_ctas=152)
    plan = pa.astr_attn_prefill_plan(qo, sl, dims, causal=False, num_ctas=152)
    items = _items(qo, sl, 4, 8, causal=False)
    rows = _rows(plan, _grid(dims, 152))
    assert sorted(it for r in rows for it in r) == sorted(items)


def test_plan_accepts_host_tensors_and_attach_checks_its_argument():
    torch = pytest.importorskip("torch")
    w = workload.config(5)
    qo, sl = w.qo_indptr.astype(np.int32), w.seq_lens.astype(np.int32)
    dims = _dims(qo, sl, w.num_qo_heads, w.num_kv_heads)
    a = pa.astr_attn_prefill_plan(qo, sl, dims, num_ctas=152)
    b = pa.astr_attn_prefill_plan(torch.from_numpy(qo), torch.from_numpy(sl).long(), dims, num_ctas=152)
    assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        pa.attach_prefill_plan(dims, torch.from_numpy(a))  # a host tensor is not a device plan
    assert pa.attach_prefill_plan(dims, None).prefill_plan is None
