"""The fp64 oracle against its pins (CPU only), plus planted-mistake checks of those pins."""
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=[f.__name__ for f in P.ALL_PINS])
def test_pin(pin):
    pin(None)


def test_sdpa_pages_shaped_decode():
    """The pages' decode microbench shape (B=32, GQA 32/8, d=128, seq 200..2000) against fp64 SDPA."""
    import workload
    P.pin_sdpa_decode(None, w=workload.config(2))


# Each mutant is one plausible slip in the oracle source; at least one pin must catch it.
MUTANTS = {
    "drop_sm_scale": ("return P->sm_scale * s;", "return s;"),
    "gqa_modulo": ("int kvh = h / G;", "int kvh = h % P->Hkv;"),
    "causal_off_by_one": ("c + i + 1, J->out", "c + i, J->out"),
    "top_left_causal": ("int64_t c = (int64_t)J->seq_lens[b] - q_len;", "int64_t c = 0 * q_len;"),
    "v_from_k_pool": ("const uint16_t *v = P->v_pool + ((int64_t)slots[j] * P->Hkv + kvh) * P->D;\n    for (int d = 0; d < D; ++d) out[d]",
                      "const uint16_t *v = P->k_pool + ((int64_t)slots[j] * P->Hkv + kvh) * P->D;\n    for (int d = 0; d < D; ++d) out[d]"),
    "normalise_by_count": ("for (int d = 0; d < D; ++d) out[d] /= l;", "for (int d = 0; d < D; ++d) out[d] /= (double)n;"),
    "combine_sign": ("exp(m - M);", "exp(M - m);"),
    "q_head_major": ("widen_row(J->q + ((int64_t)b * P->Hq + h) * D, D, qbuf);\n    attend",
                     "widen_row(J->q + ((int64_t)h * J->B + b) * D, D, qbuf);\n    attend"),
    "range_start_shifted": ("J->item_lo[it], J->item_hi[it],", "J->item_lo[it] + 1, J->item_hi[it],"),
    "split_floor_chunk": ("int64_t chunk = (n + J->S - 1) / J->S;", "int64_t chunk = n / J->S > 0 ? n / J->S : 1;"),
    "append_position_shift": ("r2t_stride + c + i];", "r2t_stride + c + i + 1];"),
    "append_k_into_v": ("memcpy(v_pool + (int64_t)slot * row, v_new", "memcpy(v_pool + (int64_t)slot * row, k_new"),
    "append_source_row_local": ("const int64_t src = (int64_t)qo_indptr[b] + i;", "const int64_t src = i;"),
    "mask_ignored": ("if (causal_ok && mrow[j] != 0)", "if (causal_ok)"),
    "mask_row_not_offset_by_query_row": ("((int64_t)b * J->q_pitch + i) * J->kv_pitch", "((int64_t)b * J->q_pitch) * J->kv_pitch"),
    "causal_flag_ignored": ("const int causal_ok = !J->causal || j <= c + i;", "const int causal_ok = j <= c + i;"),
    "mask_2d_row_pitch": ("J->mask + (int64_t)b * J->kv_pitch\n", "J->mask + (int64_t)b * J->q_pitch\n"),
    "key_index_transposed": ("k_pool + ((int64_t)slot * P->Hkv + kvh) * P->D", "k_pool + ((int64_t)kvh * P->Hkv + slot % P->Hkv) * P->D"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mut.c"
    so_path = tmp_path / "libmut.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", str(so_path), str(c_path), "-lm",
                    "-lpthread"], check=True)
    lib = oracle.load_variant(str(so_path))
    caught = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"
