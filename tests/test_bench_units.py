"""CPU checks of the benchmark's unit counts: the algorithmic FLOPs and bytes that the
roofline fractions divide by, recounted by brute force on small workloads."""
import numpy as np

import bench
import workload
from workload import make_from_lengths


def test_prefill_flops_counts_causal_visible_pairs():
    rng = np.random.default_rng(3)
    ql = np.array([1, 4, 7, 0, 3])
    pre = np.array([0, 5, 2, 4, 9])
    w = make_from_lengths(rng, kind="prefill", name="flops", seq_lens=pre + ql, q_lens=ql, Hq=8, Hkv=2, d=64)
    pairs = 0
    for b in range(w.batch):
        c = int(pre[b])
        for i in range(int(ql[b])):
            pairs += sum(1 for j in range(int(w.seq_lens[b])) if j <= c + i)
    # two matrix products (Q K^T and P V), 2 FLOP per multiply-add, d per dot product, Hq heads
    assert bench.prefill_flops(w) == 2 * 2 * w.head_dim * w.num_qo_heads * pairs


def test_decode_bytes_counts_each_attended_row_once():
    w = workload.make_decode(5, 8, 2, 64, (0, 40), seed=9)
    rows = int(w.seq_lens.sum()) * w.num_kv_heads          # (key, KV head) rows of K, and of V
    assert bench.decode_bytes(w)["kv"] == 2 * rows * w.head_dim * 2
    assert w.kv_bytes() == bench.decode_bytes(w)["kv"]


def test_source_digest_ignores_comments_and_whitespace(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    a.write_text("int f(int x) { return x + 1; }  // one\n/* block */\n")
    b.write_text("int f(int x)\n{\n  return x + 1;   // another comment\n}\n")
    assert bench.source_digest(str(a)) == bench.source_digest(str(b))
    b.write_text("int f(int x) { return x + 2; }\n")
    assert bench.source_digest(str(a)) != bench.source_digest(str(b))
