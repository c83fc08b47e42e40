"""Host-side checks of the C ABI: the library loads, exports what the header declares, and
rejects bad arguments with the documented status codes before touching the GPU."""
import ctypes
import os
import re

import pytest

import prefill_attention_gb300 as pa
from prefill_attention_gb300 import build as pbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "astr_attn.h")


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return pa.load()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(astr_attn_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_and_library_exports_every_entry_point(lib):
    names = declared_functions()
    assert set(names) == set(pa.EXPORTED_SYMBOLS), names
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"


def test_dims_struct_layout_matches_header(tmp_path):
    """The ctypes mirror has the C struct's size and field offsets (compiled from the header)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    fields = [f for f, _ in pa.Dims._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "astr_attn.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(astr_attn_dims));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(astr_attn_dims, {f}));\n' for f in fields)
                   + "  return 0; }\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(pa.Dims)
    assert got[1:] == [getattr(pa.Dims, f).offset for f in fields]


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5, -6, 17):
        assert isinstance(pa.astr_attn_status_string(st), str)
    assert pa.astr_attn_version() >= 100


def _dims(**kw):
    base = dict(batch=4, num_qo_heads=32, num_kv_heads=8, head_dim=128, num_slots=1000, r2t_stride=2000,
                max_seq_len=2000, total_q=64, max_q_len=16, max_splits=8, num_splits=0)
    base.update(kw)
    return pa.make_dims(**base)


A = 1 << 20  # fake, 16-byte aligned device addresses: validation fails before any dereference


def _dec(d, **ptr):
    p = dict(q=A, k=A, v=A, r2t=A, seq=A, kvi=A, o=A, ml=A, out=A)
    p.update(ptr)
    return pa.astr_attn_paged_decode(p["q"], p["k"], p["v"], p["r2t"], p["seq"], p["kvi"], p["o"], p["ml"],
                                     p["out"], d, 0.1, stream=0, check=False)


def _pf(d, scale=0.1, **ptr):
    p = dict(q=A, qo=A, k=A, v=A, r2t=A, seq=A, kvi=A, out=A)
    p.update(ptr)
    return pa.astr_attn_prefill_ragged(p["q"], p["qo"], p["k"], p["v"], p["r2t"], p["seq"], p["kvi"], p["out"], d,
                                       scale, stream=0, check=False)


@pytest.mark.parametrize("name", ["q", "k", "v", "r2t", "seq", "kvi", "o", "ml", "out"])
def test_decode_null_pointer(lib, name):
    assert _dec(_dims(), **{name: 0}) == pa.ASTR_ERR_INVALID_ARG


@pytest.mark.parametrize("name,addr", [("q", A + 8), ("k", A + 2), ("out", A + 4), ("o", A + 4), ("ml", A + 8),
                                       ("r2t", A + 2), ("seq", A + 1)])
def test_decode_misaligned(lib, name, addr):
    assert _dec(_dims(), **{name: addr}) == pa.ASTR_ERR_MISALIGNED


def test_int_arrays_need_only_4_byte_alignment(lib):
    # 4-byte aligned int32 arrays pass the alignment check and fail later on the bad head_dim
    assert _dec(_dims(head_dim=96), r2t=A + 4, seq=A + 4, kvi=A + 12) == pa.ASTR_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), pa.ASTR_ERR_UNSUPPORTED),
    (dict(head_dim=256), pa.ASTR_ERR_UNSUPPORTED),
    (dict(num_qo_heads=30, num_kv_heads=8), pa.ASTR_ERR_UNSUPPORTED),
    (dict(num_qo_heads=128, num_kv_heads=4), pa.ASTR_ERR_UNSUPPORTED),   # group 32 not built
    (dict(batch=-1), pa.ASTR_ERR_INVALID_ARG),
    (dict(num_kv_heads=0), pa.ASTR_ERR_INVALID_ARG),
    (dict(r2t_stride=100), pa.ASTR_ERR_INVALID_ARG),                      # stride below max_seq_len
    (dict(max_splits=0), pa.ASTR_ERR_INVALID_ARG),
    (dict(num_splits=-1), pa.ASTR_ERR_INVALID_ARG),
    (dict(num_slots=0), pa.ASTR_ERR_INVALID_ARG),
    (dict(flags=2), pa.ASTR_ERR_INVALID_ARG),                             # an undefined flag bit
])
def test_decode_bad_dims(lib, kw, status):
    assert _dec(_dims(**kw)) == status


def test_combine_explicit_layout_needs_capacity(lib):
    # kv_indptr NULL: num_splits partials per row, which must fit in max_splits
    st = pa.astr_attn_decode_combine(A, A, None, None, A, _dims(num_splits=9), stream=0, check=False)
    assert st == pa.ASTR_ERR_WORKSPACE_TOO_SMALL
    st = pa.astr_attn_decode_combine(A, A, None, None, A, _dims(num_splits=0), stream=0, check=False)
    assert st == pa.ASTR_ERR_INVALID_ARG


def test_decode_non_finite_scale(lib):
    st = pa.astr_attn_paged_decode(A, A, A, A, A, A, A, A, A, _dims(), float("nan"), stream=0, check=False)
    assert st == pa.ASTR_ERR_INVALID_ARG


def test_decode_null_dims(lib):
    st = lib.astr_attn_paged_decode(A, A, A, A, A, A, A, A, A, None, ctypes.c_float(0.1), None)
    assert st == pa.ASTR_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["q", "qo", "k", "v", "r2t", "seq", "out"])
def test_prefill_null_pointer(lib, name):
    assert _pf(_dims(), **{name: 0}) == pa.ASTR_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=80), pa.ASTR_ERR_UNSUPPORTED),
    (dict(num_qo_heads=12, num_kv_heads=8), pa.ASTR_ERR_UNSUPPORTED),
    (dict(num_qo_heads=96, num_kv_heads=3), pa.ASTR_ERR_UNSUPPORTED),    # group 32 not built
    (dict(total_q=-1), pa.ASTR_ERR_INVALID_ARG),
    (dict(max_q_len=3000), pa.ASTR_ERR_INVALID_ARG),                    # q_len bound above max_seq_len
])
def test_prefill_bad_dims(lib, kw, status):
    assert _pf(_dims(**kw)) == status


def test_prefill_misaligned(lib):
    assert _pf(_dims(), q=A + 2) == pa.ASTR_ERR_MISALIGNED
    assert _pf(_dims(), qo=A + 2) == pa.ASTR_ERR_MISALIGNED
    assert _pf(_dims(), kvi=A + 1) == pa.ASTR_ERR_MISALIGNED


def test_prefill_kv_indptr_may_be_null_and_empty_batch_is_noop(lib):
    # batch 0 returns OK without launching (and without a GPU)
    assert _pf(_dims(batch=0), kvi=0) == pa.ASTR_OK


def test_workspace_bytes(lib):
    ob, mb = pa.astr_attn_decode_workspace_bytes(_dims(batch=32, max_splits=5))
    assert ob == 32 * 32 * 5 * 128 * 4 and mb == 32 * 32 * 5 * 2 * 4


def test_status_word_must_be_4_byte_aligned(lib):
    assert _dec(_dims(status=A + 2)) == pa.ASTR_ERR_MISALIGNED
    assert _pf(_dims(status=A + 1)) == pa.ASTR_ERR_MISALIGNED
    assert _app(_dims(status=A + 3)) == pa.ASTR_ERR_MISALIGNED
    # a 4-byte aligned word passes and the call fails later, on the bad head_dim
    assert _dec(_dims(status=A + 4, head_dim=96)) == pa.ASTR_ERR_UNSUPPORTED


def _noalloc(d, **ptr):
    p = dict(q=A, k=A, v=A, r2t=A, seq=A, kvi=A, out=A)
    p.update(ptr)
    return pa.astr_attn_paged_decode_noalloc(p["q"], p["k"], p["v"], p["r2t"], p["seq"], p["kvi"], p["out"], d, 0.1,
                                             stream=0, check=False)


@pytest.mark.parametrize("name,addr", [("q", 0), ("k", 0), ("v", 0), ("r2t", 0), ("seq", 0), ("kvi", 0), ("out", 0),
                                       ("q", A + 8), ("out", A + 2), ("r2t", A + 2), ("kvi", A + 1)])
@pytest.mark.parametrize("batch", [0, 4])
def test_noalloc_checks_arguments_like_the_workspace_entry_point(lib, name, addr, batch):
    """Same status as astr_attn_paged_decode for the same bad pointer, an empty batch included."""
    d = _dims(batch=batch)
    expect = pa.ASTR_ERR_INVALID_ARG if addr == 0 else pa.ASTR_ERR_MISALIGNED
    assert _dec(d, **{name: addr}) == expect
    assert _noalloc(d, **{name: addr}) == expect


def test_noalloc_rejects_oversize_and_null_dims_without_gpu(lib):
    # 256 x 32 heads x 64 splits x 130 floats = 272 MB > the fixed 16 MiB array
    st = pa.astr_attn_paged_decode_noalloc(A, A, A, A, A, A, A, _dims(batch=256, max_splits=64), 0.1, stream=0,
                                           check=False)
    assert st == pa.ASTR_ERR_WORKSPACE_TOO_SMALL
    st = lib.astr_attn_paged_decode_noalloc(A, A, A, A, A, A, A, None, ctypes.c_float(0.1), None)
    assert st == pa.ASTR_ERR_INVALID_ARG


def test_library_imports_no_device_allocator(lib):
    """No entry point can allocate: the library does not even import cudaMalloc/cudaFree."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    syms = subprocess.run([nm, "-D", "--undefined-only", pa.lib_path()], capture_output=True, text=True).stdout
    for bad in ("cudaMalloc", "cudaFree", "cudaMallocAsync", "cudaFreeAsync", "cudaMallocManaged"):
        assert f" {bad}" not in syms and f"U {bad}@" not in syms, bad


def _app(d, **ptr):
    p = dict(kn=A, vn=A, qo=A, r2t=A, seq=A, k=A, v=A)
    p.update(ptr)
    return pa.astr_attn_kv_append(p["kn"], p["vn"], p["qo"], p["r2t"], p["seq"], p["k"], p["v"], d, stream=0,
                                  check=False)


@pytest.mark.parametrize("name", ["kn", "vn", "qo", "r2t", "seq", "k", "v"])
def test_append_null_pointer(lib, name):
    assert _app(_dims(), **{name: 0}) == pa.ASTR_ERR_INVALID_ARG


def test_append_misaligned(lib):
    assert _app(_dims(), kn=A + 8) == pa.ASTR_ERR_MISALIGNED
    assert _app(_dims(), v=A + 2) == pa.ASTR_ERR_MISALIGNED
    assert _app(_dims(), r2t=A + 2) == pa.ASTR_ERR_MISALIGNED


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=80), pa.ASTR_ERR_UNSUPPORTED),
    (dict(total_q=-1), pa.ASTR_ERR_INVALID_ARG),
    (dict(num_slots=0), pa.ASTR_ERR_INVALID_ARG),
    (dict(r2t_stride=10), pa.ASTR_ERR_INVALID_ARG),   # below max_seq_len
])
def test_append_bad_dims(lib, kw, status):
    assert _app(_dims(**kw)) == status


def test_append_nothing_to_do_without_gpu(lib):
    assert _app(_dims(batch=0)) == pa.ASTR_OK
    assert _app(_dims(total_q=0)) == pa.ASTR_OK
    assert lib.astr_attn_kv_append(A, A, A, A, A, A, A, None, None) == pa.ASTR_ERR_INVALID_ARG


def _mask(ptr=A, dims=3, kv_pitch=2000, q_pitch=16, causal=1):
    return pa.Mask(ptr, dims, kv_pitch, q_pitch, causal)


def _pfm(d, m, **ptr):
    p = dict(q=A, qo=A, k=A, v=A, r2t=A, seq=A, kvi=A, out=A)
    p.update(ptr)
    return pa.astr_attn_prefill_ragged_masked(p["q"], p["qo"], p["k"], p["v"], p["r2t"], p["seq"], p["kvi"], m,
                                              p["out"], d, 0.1, stream=0, check=False)


def _decm(d, m):
    return pa.astr_attn_paged_decode_masked(A, A, A, A, A, A, m, A, A, A, d, 0.1, stream=0, check=False)


@pytest.mark.parametrize("kw,status", [
    (dict(dims=4), pa.ASTR_ERR_INVALID_ARG),
    (dict(kv_pitch=2008), pa.ASTR_ERR_INVALID_ARG),      # not a multiple of 16
    (dict(kv_pitch=1984), pa.ASTR_ERR_INVALID_ARG),      # below max_seq_len
    (dict(q_pitch=15), pa.ASTR_ERR_INVALID_ARG),         # below max_q_len
    (dict(causal=2), pa.ASTR_ERR_INVALID_ARG),
    (dict(ptr=A + 8), pa.ASTR_ERR_MISALIGNED),
])
def test_prefill_masked_bad_mask(lib, kw, status):
    assert _pfm(_dims(batch=0), _mask(**kw)) == status   # checked before the empty-batch early return


def test_prefill_masked_accepts_valid_masks_and_null_struct_is_rejected(lib):
    assert _pfm(_dims(batch=0), _mask()) == pa.ASTR_OK
    assert _pfm(_dims(batch=0), _mask(dims=2, q_pitch=0)) == pa.ASTR_OK
    assert _pfm(_dims(batch=0), _mask(ptr=None, dims=0, kv_pitch=0, q_pitch=0, causal=0)) == pa.ASTR_OK
    assert _pfm(_dims(batch=0), None) == pa.ASTR_ERR_INVALID_ARG
    assert _pfm(_dims(batch=0), _mask(), q=0) == pa.ASTR_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,status", [
    (dict(dims=1), pa.ASTR_ERR_INVALID_ARG),
    (dict(kv_pitch=0), pa.ASTR_ERR_INVALID_ARG),
    (dict(q_pitch=0), pa.ASTR_ERR_INVALID_ARG),          # 3-D needs at least one row per request
    (dict(ptr=A + 4), pa.ASTR_ERR_MISALIGNED),
])
def test_decode_masked_bad_mask(lib, kw, status):
    assert _decm(_dims(batch=0), _mask(**kw)) == status


def test_decode_masked_null_struct(lib):
    assert _decm(_dims(batch=0), None) == pa.ASTR_ERR_INVALID_ARG


def _lay(b=2000 * 8 * 128, t=8 * 128, h=128):
    return pa.KvLayout(b, t, h)


def _pfc(d, layout, **ptr):
    p = dict(q=A, qo=A, k=A, v=A, seq=A, kvi=A, out=A)
    p.update(ptr)
    return pa.astr_attn_prefill_contiguous(p["q"], p["qo"], p["k"], p["v"], layout, p["seq"], p["kvi"], p["out"], d,
                                           0.1, stream=0, check=False)


@pytest.mark.parametrize("kw,status", [
    (dict(t=-8), pa.ASTR_ERR_INVALID_ARG),
    (dict(h=100), pa.ASTR_ERR_MISALIGNED),     # not a multiple of 8 elements
    (dict(b=12), pa.ASTR_ERR_MISALIGNED),
])
def test_contiguous_bad_layout(lib, kw, status):
    assert _pfc(_dims(batch=0), _lay(**kw)) == status


def test_contiguous_null_layout_and_table_not_needed(lib):
    assert lib.astr_attn_prefill_contiguous(A, A, A, A, None, A, A, None, A, ctypes.byref(_dims(batch=0)),
                                            ctypes.c_float(0.1), None) == pa.ASTR_ERR_INVALID_ARG
    # no slot table: r2t_stride and num_slots are not read
    assert _pfc(_dims(batch=0, r2t_stride=0, num_slots=0), _lay()) == pa.ASTR_OK
    assert _pfc(_dims(batch=0), _lay(), k=A + 2) == pa.ASTR_ERR_MISALIGNED
    st = lib.astr_attn_decode_contiguous(A, A, A, None, A, A, None, A, A, A, ctypes.byref(_dims(batch=0)),
                                         ctypes.c_float(0.1), None)
    assert st == pa.ASTR_ERR_INVALID_ARG


def test_header_is_plain_c(tmp_path):
    """The ABI header compiles as C99 with warnings as errors (no C++ in the interface)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "use_header.c"
    src.write_text('#include "astr_attn.h"\n'
                   "int main(void) { astr_attn_dims d = {0}; astr_attn_mask m = {0}; astr_attn_kv_layout l = {0};\n"
                   "  int (*v)(void) = astr_attn_version; (void)d; (void)m; (void)l; (void)v; return 0; }\n")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.dirname(HEADER),
                        "-c", str(src), "-o", str(tmp_path / "use_header.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _qo(qb=0, qt=32 * 128, qh=128, ob=0, ot=32 * 128, oh=128):
    return pa.QoLayout(qb, qt, qh, ob, ot, oh)


@pytest.mark.parametrize("kw,status", [
    (dict(qh=-8), pa.ASTR_ERR_INVALID_ARG),
    (dict(ob=-128), pa.ASTR_ERR_INVALID_ARG),
    (dict(qt=100), pa.ASTR_ERR_MISALIGNED),       # not a multiple of 8 elements
    (dict(oh=4), pa.ASTR_ERR_MISALIGNED),
])
def test_strided_bad_qo_layout(lib, kw, status):
    d = _dims(batch=0)
    assert pa.astr_attn_prefill_strided(A, A, A, A, A, A, A, A, d, 0.1, qo_layout=_qo(**kw), stream=0,
                                        check=False) == status
    assert pa.astr_attn_decode_strided(A, A, A, A, A, A, A, A, A, d, 0.1, qo_layout=_qo(**kw), stream=0,
                                       check=False) == status


def test_strided_null_layouts_and_table_rules(lib):
    d = _dims(batch=0)
    # no layouts: the paged pool, packed rows -- the table is required then
    assert pa.astr_attn_prefill_strided(A, A, A, A, A, A, A, A, d, 0.1, stream=0, check=False) == pa.ASTR_OK
    assert pa.astr_attn_prefill_strided(A, A, A, A, 0, A, A, A, d, 0.1, stream=0,
                                        check=False) == pa.ASTR_ERR_INVALID_ARG
    # a contiguous cache: the table is not read (may be NULL)
    assert pa.astr_attn_prefill_strided(A, A, A, A, 0, A, A, A, _dims(batch=0, r2t_stride=0, num_slots=0), 0.1,
                                        kv_layout=_lay(), stream=0, check=False) == pa.ASTR_OK
    # (decode asks for the device's SM count after its argument checks: DEVICE where no GPU is present)
    st = pa.astr_attn_decode_strided(A, A, A, 0, A, A, A, A, A, d, 0.1, kv_layout=_lay(), qo_layout=_qo(), stream=0,
                                     check=False)
    assert st in (pa.ASTR_OK, pa.ASTR_ERR_DEVICE)
    assert pa.astr_attn_decode_strided(A, A, A, 0, A, A, A, A, A, d, 0.1, qo_layout=_qo(), stream=0,
                                       check=False) == pa.ASTR_ERR_INVALID_ARG   # paged pool needs the table
