"""The test helper that turns the decode split schedule into key ranges, checked key by key
against the formula stated for astr_attn_decode_num_splits / astr_attn_paged_decode in
include/astr_attn.h (CPU only)."""
import numpy as np
import pytest

import split_schedule as ss

W = 32


def _header_chunk_len(seq_lens, max_seq_len, n_chunks, max_splits):
    """C = max(ceil(S / num_splits), F), F = max(1, ceil(ceil(max_seq_len / 32) / (max_splits - 1))),
    C = S when max_splits == 1 (S = the batch's 32-key slots)."""
    S = sum((int(n) + W - 1) // W for n in seq_lens if n > 0)
    if max_splits == 1:
        return max(S, 1)
    F = max(1, -(-((max_seq_len + W - 1) // W) // (max_splits - 1)))
    return max(-(-S // n_chunks), F)


CASES = [
    ([1, 31, 32, 33, 64, 65], 70, 5, 8),
    ([0, 0, 100, 0, 7], 100, 3, 2),
    ([2000] * 4 + [200] * 4, 2000, 76, 32),
    ([5], 5, 1, 1),
    ([40, 0, 1, 1, 1, 300, 299], 300, 200, 3),
]


@pytest.mark.parametrize("seq,max_len,n_chunks,max_splits", CASES)
def test_pieces_follow_the_header_formula_key_by_key(seq, max_len, n_chunks, max_splits):
    C = ss.chunk_slots(seq, max_len, n_chunks, max_splits)
    assert C == _header_chunk_len(seq, max_len, n_chunks, max_splits)
    ps = ss.pieces(seq, C)
    by_key = {}
    for (b, s, lo, hi) in ps:
        assert lo < hi, "a piece holds at least one key"
        for j in range(lo, hi):
            assert (b, j) not in by_key, "a key lies in two pieces"
            by_key[(b, j)] = s
    SP = 0
    for b, n in enumerate(seq):
        for j in range(n):
            slot = SP + j // W           # the batch slot that holds key j of request b
            chunk = slot // C            # the chunk that reads it
            assert by_key.pop((b, j)) == chunk - SP // C, f"request {b} key {j}"
        SP += (n + W - 1) // W
    assert not by_key, "pieces hold keys past a request's end"
    # the floor keeps every request within the partial capacity
    counts = ss.split_counts(seq, C)
    assert counts.max() <= max_splits


def test_random_batches():
    rng = np.random.default_rng(5)
    for _ in range(40):
        B = int(rng.integers(1, 40))
        seq = [int(x) for x in rng.integers(0, 500, size=B)]
        max_len = max(seq + [1])
        n_chunks = int(rng.integers(1, 300))
        max_splits = int(rng.integers(1, 40))
        test_pieces_follow_the_header_formula_key_by_key(seq, max_len, n_chunks, max_splits)
